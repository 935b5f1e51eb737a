// softmax_tc.cu - softmax branch on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA), bf16 inputs.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the softmax state is the set of keys and values
// of the chunks that chose softmax; inside a chunk both correlations are
// computed, so every query of chunk c attends to the retained chunks before
// c plus its own chunk causally (diagonal included).
//
// Tiling.  A query tile is 128 rows = the two chunks c0 = 2p and c1 = 2p + 1
// of one (b, h).  Its key/value blocks are 128 keys = two 64-token chunk
// slots: first the softmax chunks before c0 (sel_idx[0 .. nprev[c0]), in
// pairs), then the diagonal block (c0, c1).  Rows of c1 also see c0 when c0
// chose softmax; both diagonal slots are causal for their own rows.  Slots
// without a chunk are loaded with c0 (finite data) and masked.
//
// Persistent CTAs take tiles from a list ordered heaviest first (nprev grows
// with c) through a global counter, so CTAs that start late (the SMs may be
// shared with a concurrent kernel) or draw short tiles just take more; inside
// a CTA the K producer takes the tile and hands it to the other roles.
// Roles (256 threads):
//   warp 0     TMA producer of Q (one per tile) and of the K blocks (3-deep
//              ring); warp 2 the producer of the V blocks (2-deep ring)
//   warp 1     TMEM owner; lane 0 issues S_j = Q K_j^T into one of three
//              TMEM S buffers, up to three blocks ahead (a buffer is reused
//              once the P V product that read its P has completed)
//   warp 3     lane 0 issues O += P_j V_j, P_j read from TMEM (it overwrites
//              S_j in place).  Two issuing threads on two SM sub-partitions:
//              an MMA goes out only when its thread is scheduled, and each
//              shares its sub-partition with a busy softmax warp.
//   warps 4-7  softmax: thread r owns query row r (its TMEM lane); the row's
//              128 scores of a block are read from TMEM once, their max taken
//              in registers, and P_j packed to bf16 in TMEM, in the exp2
//              domain.  The running max used for the exponent is raised (and
//              O, l rescaled in place) only when a row max grows by more than
//              2^8, so P <= 256 and the rescale, which waits for the previous
//              P V product, is rare.
//              The tile epilogue writes the softmax half of the layer output
//              ("Kernmechanismen" item 4): w RMSNorm(O / l) in bf16, w the
//              query gate; the Gated DeltaNet side adds its half afterwards.
//              The rows go through a swizzled bf16 tile in shared memory and
//              leave with TMA stores.
//              It reads O before the warps release the next tile's first P,
//              so one O accumulator serves every tile.
// TMEM: S0, S1, S2 (128 columns each), O (D columns).
// Every wait is bounded (tc::kWaitLimitNs); on expiry the kernel records an
// error, drains what it issued and exits.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

enum { kFull = 0, kCausal = 1, kNone = 2 };
constexpr float kRescaleLog2 = 8.f;  // lazy-rescale threshold (log2 units)
constexpr int KS = 3;                // K ring depth
constexpr int VS = 2;                // V ring depth (the V producer runs far ahead of P V)
constexpr int NS = 3;                // S/P buffers in TMEM
constexpr int kTileTakers = 7;       // arrivals that free a tile-queue slot: 2 MMA issuers, V producer, 4 softmax warps

template <int D>
struct SoftmaxSmem {
  static constexpr int kHalf = 128 * 128;  // bytes of one 128-line x 64-col bf16 block
  static constexpr int kQ = 128 * D * 2;
  static constexpr int kKV = 128 * D * 2;
  static constexpr int offQ = 0;
  static constexpr int offK = offQ + kQ;
  static constexpr int offV = offK + KS * kKV;
  static constexpr int offOst = offV + VS * kKV;  // bf16 output tile of the epilogue (TMA store source)
  static constexpr int offBar = offOst + kQ;
  static constexpr int kNumBars = 2 + 2 * KS + 2 * VS + 3 * NS + 1 + 4 + 2 + 2;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int offNw = offTmem + 16;  // RMSNorm weights of the softmax branch, D floats
  static constexpr int offTq = offNw + D * 4;  // two-slot tile queue (ints)
  static constexpr int kBytes = offTq + 16 + 1024;  // + alignment slack
};

// barrier slots
enum {
  B_QF = 0, B_QE = 1, B_KF = 2, B_KE = B_KF + KS, B_VF = B_KE + KS, B_VE = B_VF + VS,
  B_SF = B_VE + VS, B_PF = B_SF + NS, B_PV = B_PF + NS, B_OF = B_PV + NS, B_TF = B_OF + 1, B_TE = B_TF + 2,
  B_OSF = B_TE + 2, B_OSE = B_OSF + 1, B_SDR = B_OSE + 1, B_PDR = B_SDR + 1
};

// Masked keys of a 32-column chunk become -inf.  key0 = index of v[0] within
// its 64-token chunk slot; rr = this row's index within its own chunk.
__device__ __forceinline__ void mask_chunk(float (&v)[32], int mode, int key0, int rr) {
  if (mode == kNone) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = -INFINITY;
  } else if (mode == kCausal) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = (key0 + x <= rr) ? v[x] : -INFINITY;
  }
}

struct TileInfo {
  int p, c0, n0, nbp, nb;
  long long bh;
  bool has_c1, c0_soft;
};

__device__ __forceinline__ TileInfo tile_info(int i, long long BH, int T, int N, const int32_t* nprev,
                                              const uint8_t* sel) {
  TileInfo t;
  t.p = T - 1 - (int)(i / BH);
  t.bh = i % BH;
  t.c0 = 2 * t.p;
  t.has_c1 = t.c0 + 1 < N;
  t.n0 = nprev[t.bh * N + t.c0];
  t.nbp = (t.n0 + 1) >> 1;
  t.nb = t.nbp + 1;
  t.c0_soft = sel[t.bh * N + t.c0] == 0;
  return t;
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    softmax_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const int32_t* __restrict__ nprev,
                      const int32_t* __restrict__ sel_idx, const uint8_t* __restrict__ sel, int L, int N,
                      int T, long long BH, float sl2, const float* __restrict__ gate,
                      const float* __restrict__ nw_s, float eps, __nv_bfloat16* __restrict__ out,
                      float* __restrict__ o_s, float* __restrict__ lse_out, int* __restrict__ err,
                      int* __restrict__ tile_ctr) {
  using S = SoftmaxSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* Qs = smem + S::offQ;
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int n_tiles = (int)(BH * T);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* nw_sm = (float*)(smem + S::offNw);
  for (int c = threadIdx.x; c < D; c += blockDim.x) nw_sm[c] = nw_s ? nw_s[c] : 1.f;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[B_QF], 1);
    tc::mbar_init(&bars[B_QE], 1);
    for (int s = 0; s < KS; ++s) {
      tc::mbar_init(&bars[B_KF + s], 1);
      tc::mbar_init(&bars[B_KE + s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      tc::mbar_init(&bars[B_VF + s], 1);
      tc::mbar_init(&bars[B_VE + s], 1);
    }
    tc::mbar_init(&bars[B_OSF], 128);  // output tile written by the 128 softmax threads
    tc::mbar_init(&bars[B_OSE], 1);    // previous tile's TMA store has read the tile
    tc::mbar_init(&bars[B_SDR], 1);    // drains of the two MMA-issuing threads
    tc::mbar_init(&bars[B_PDR], 1);
    for (int b = 0; b < NS; ++b) {
      tc::mbar_init(&bars[B_SF + b], 1);
      tc::mbar_init(&bars[B_PF + b], 128);
      tc::mbar_init(&bars[B_PV + b], 1);
    }
    tc::mbar_init(&bars[B_OF], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[B_TF + s], 1);
      tc::mbar_init(&bars[B_TE + s], kTileTakers);
    }
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- dynamic tile schedule.  Tiles are numbered heaviest first; the K
  // producer takes the next one from a global counter and publishes it in a
  // two-slot queue in shared memory; every other role reads each entry once.
  // -1 ends the list, -2 means a wait expired.
  volatile int* tileq = (volatile int*)(smem + S::offTq);
  auto publish = [&](int n) -> int {  // K producer: tile of sequence number n
    const int s = n & 1;
    if (!tc::mbar_wait(&bars[B_TE + s], ((n >> 1) & 1) ^ 1, err)) return -2;
    const int a = atomicAdd(tile_ctr, 1);
    const int t = a < n_tiles ? a : -1;
    tileq[s] = t;
    tc::mbar_arrive(&bars[B_TF + s]);  // release: the entry is visible to whoever sees the phase
    return t;
  };
  auto take = [&](int n, bool release) -> int {  // every other role
    const int s = n & 1;
    if (!tc::mbar_wait(&bars[B_TF + s], (n >> 1) & 1, err)) return -2;
    const int t = tileq[s];
    if (release) tc::mbar_arrive(&bars[B_TE + s]);
    return t;
  };

  if (warp == 0 || warp == 2) {
    // ----------------------------------------------------------- producers
    // warp 0 loads Q and K, warp 2 loads V: separate streams, so that a K
    // block is never queued behind a V block whose ring slot is still held
    // by an earlier P V product
    if (lane == 0) {
      const bool kq = (warp == 0);
      if (kq) tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(kq ? &tm_k : &tm_v);
      const CUtensorMap* tm = kq ? &tm_k : &tm_v;
      uint8_t* ring = smem + (kq ? S::offK : S::offV);
      uint64_t* full = &bars[kq ? B_KF : B_VF];
      uint64_t* empty = &bars[kq ? B_KE : B_VE];
      const int RD = kq ? KS : VS;  // ring depth
      int gj = 0, tn = 0;
      bool ok = true;
      auto next = [&](int n) { return kq ? publish(n) : take(n, true); };
      int cur = next(0);
      int nxt = cur >= 0 ? next(1) : -1;
      // each tile's descriptor is read one tile ahead (global latency)
      TileInfo tnx = tile_info(cur >= 0 ? cur : 0, BH, T, N, nprev, sel);
      for (; cur >= 0 && ok; ++tn) {
        const TileInfo ti = tnx;
        if (nxt >= 0) tnx = tile_info(nxt, BH, T, N, nprev, sel);
        const long long row0 = ti.bh * (long long)L;
        if (kq) {
          if (!(ok = tc::mbar_wait(&bars[B_QE], (tn & 1) ^ 1, err))) break;
          tc::mbar_arrive_expect_tx(&bars[B_QF], S::kQ);
          for (int h = 0; h < D / 64; ++h)
            for (int rc = 0; rc < 2; ++rc)
              tc::tma_load_2d(Qs + h * S::kHalf + rc * (S::kHalf / 2), &tm_q, 64 * h,
                              (int)(row0 + 128LL * ti.p + 64 * rc), &bars[B_QF]);
        }
        // chunk pair of block j (the softmax chunks before c0, in pairs, then
        // the diagonal pair), read one block ahead to hide the global latency
        auto pair = [&](int j, int& c0, int& c1) {
          if (j < ti.nbp) {
            c0 = sel_idx[ti.bh * N + 2 * j];
            c1 = (2 * j + 1 < ti.n0) ? sel_idx[ti.bh * N + 2 * j + 1] : ti.c0;
          } else {
            c0 = ti.c0;
            c1 = ti.has_c1 ? ti.c0 + 1 : ti.c0;
          }
        };
        int ch0, ch1;
        pair(0, ch0, ch1);
        for (int j = 0; j < ti.nb; ++j, ++gj) {
          int nx0 = 0, nx1 = 0;
          if (j + 1 < ti.nb) pair(j + 1, nx0, nx1);
          const int ks = gj % RD, par = ((gj / RD) & 1) ^ 1;
          uint8_t* buf = ring + ks * S::kKV;
          if (!(ok = tc::mbar_wait(&empty[ks], par, err))) break;
          tc::mbar_arrive_expect_tx(&full[ks], S::kKV);
          for (int slot = 0; slot < 2; ++slot)
            for (int h = 0; h < D / 64; ++h)
              tc::tma_load_2d(buf + h * S::kHalf + slot * (S::kHalf / 2), tm, 64 * h,
                              (int)(row0 + 64LL * (slot ? ch1 : ch0)), &full[ks]);
          ch0 = nx0;
          ch1 = nx1;
        }
        if (!ok) break;
        cur = nxt;
        nxt = cur >= 0 ? next(tn + 2) : -1;
      }
      if (cur == -2 || nxt == -2) ok = false;
      // make sure every load completed and every release commit landed
      for (int s = 0; s < RD; ++s) {
        const int uses = gj > s ? (gj - 1 - s) / RD + 1 : 0;
        if (uses > 0) {
          tc::mbar_wait(&full[s], (uses - 1) & 1, nullptr);
          if (ok) tc::mbar_wait(&empty[s], (uses - 1) & 1, err);
        }
      }
      if (kq && tn > 0) {
        tc::mbar_wait(&bars[B_QF], (tn - 1) & 1, nullptr);
        if (ok) tc::mbar_wait(&bars[B_QE], (tn - 1) & 1, err);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ----------------------------------------------------------------- MMA
    // Two issuing threads on different SM sub-partitions: warp 1 issues
    // S_j = Q K_j^T, warp 3 issues O += P_j V_j.  An MMA goes out only when
    // its thread is scheduled, and each of these threads shares its
    // sub-partition with a softmax warp that keeps the issue port busy;
    // split, each has half the MMAs to issue.  S_j reuses the TMEM buffer of
    // P_{j-3}, so warp 1 waits for that product first (B_PV); every P V comes
    // from warp 3, so O accumulates them in order.
    if (lane == 0) {
      const bool s_role = (warp == 1);
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, D, false, true);
      // descriptors are built once; each MMA only offsets the address field
      const uint64_t qd0 = tc::smem_desc_sw128(tc::smem_u32(Qs), 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(tc::smem_u32(smem + S::offK), 16, 1024);
      const uint64_t vd0 = tc::smem_desc_sw128(tc::smem_u32(smem + S::offV), S::kHalf, 1024);
      const uint32_t tO = tmem + NS * 128;
      int gj = 0, tn = 0;
      bool ok = true;
      int cur = take(0, true);
      int nxt = cur >= 0 ? take(1, true) : -1;
      // each tile's descriptor is read one tile ahead (global latency)
      TileInfo tnx = tile_info(cur >= 0 ? cur : 0, BH, T, N, nprev, sel);
      for (; cur >= 0 && ok; ++tn) {
        const TileInfo ti = tnx;
        if (nxt >= 0) tnx = tile_info(nxt, BH, T, N, nprev, sel);
        if (s_role) {
          if (!(ok = tc::mbar_wait(&bars[B_QF], tn & 1, err))) break;
          for (int j = 0; j < ti.nb; ++j) {
            const int g = gj + j, b = g % NS, ks = g % KS;
            // the buffer's previous P has been read by its P V product
            if (g >= NS && !(ok = tc::mbar_wait(&bars[B_PV + b], ((g - NS) / NS) & 1, err))) break;
            if (!(ok = tc::mbar_wait(&bars[B_KF + ks], (g / KS) & 1, err))) break;
            tc::fence_after();
            const uint64_t kd = tc::desc_add(kd0, ks * S::kKV);
            const uint32_t tS = tmem + b * 128;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * S::kHalf + (kk & 3) * 32;
              tc::mma_bf16(tS, tc::desc_add(qd0, off), tc::desc_add(kd, off), idesc_qk, kk > 0);
            }
            tc::mma_commit(&bars[B_SF + b]);
            tc::mma_commit(&bars[B_KE + ks]);
            if (j + 1 == ti.nb) tc::mma_commit(&bars[B_QE]);  // Q may be replaced once these S are done
          }
        } else {
          // The previous tile's O was read out by the softmax warps before
          // they released this tile's first P, so its P V may overwrite O.
          for (int j = 0; j < ti.nb; ++j) {
            const int g = gj + j, b = g % NS, vs = g % VS;
            if (!(ok = tc::mbar_wait(&bars[B_PF + b], (g / NS) & 1, err))) break;
            if (!(ok = tc::mbar_wait(&bars[B_VF + vs], (g / VS) & 1, err))) break;
            tc::fence_after();
            const uint64_t vd = tc::desc_add(vd0, vs * S::kKV);
            const uint32_t tP = tmem + b * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc::mma_bf16_ts(tO, tP + kk * 8, tc::desc_add(vd, kk * 2048), idesc_pv, (j > 0) || (kk > 0));
            tc::mma_commit(&bars[B_PV + b]);
            tc::mma_commit(&bars[B_VE + vs]);
          }
          if (ok) tc::mma_commit(&bars[B_OF]);
        }
        if (!ok) break;
        gj += ti.nb;
        cur = nxt;
        nxt = cur >= 0 ? take(tn + 2, true) : -1;
      }
      // drain: every MMA this thread issued completes before the commit lands
      uint64_t* dr = &bars[s_role ? B_SDR : B_PDR];
      tc::mma_commit(dr);
      tc::mbar_wait(dr, 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x - 128;
    const int half = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    int gj = 0, tn = 0;
    bool ok = true;
    // tile descriptor and the rows' query gate are read one tile ahead
    auto gate_of = [&](const TileInfo& t) -> float {
      return (half == 0 || t.has_c1) ? gate[t.bh * (long long)L + 128LL * t.p + r] : 0.f;
    };
    auto take_w = [&](int n) -> int {  // one read per warp of a tile-queue entry
      const int t = __shfl_sync(0xffffffffu, take(n, false), 0);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_TE + (n & 1)]);
      return t;
    };
    int cur = take_w(0);
    int nxt = cur >= 0 ? take_w(1) : -1;
    TileInfo tnx = tile_info(cur >= 0 ? cur : 0, BH, T, N, nprev, sel);
    float wnx = cur >= 0 ? gate_of(tnx) : 0.f;
    for (; cur >= 0 && ok; ++tn) {
      const TileInfo ti = tnx;
      const float w = wnx;
      if (nxt >= 0) {
        tnx = tile_info(nxt, BH, T, N, nprev, sel);
        wnx = gate_of(tnx);
      }
      const uint32_t o_addr = tmem + NS * 128 + lane_off;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < ti.nb; ++j, ++gj) {
        const int b = gj % NS;
        if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_SF + b], (gj / NS) & 1, err)))) break;
        tc::fence_after();
        int mode0, mode1;
        if (j < ti.nbp) {
          mode0 = kFull;
          mode1 = (2 * j + 1 < ti.n0) ? kFull : kNone;
        } else if (half == 0) {
          mode0 = kCausal;
          mode1 = kNone;
        } else {
          mode0 = ti.has_c1 ? (ti.c0_soft ? kFull : kNone) : kFull;
          mode1 = ti.has_c1 ? kCausal : kNone;
        }
        const uint32_t s_addr = tmem + b * 128 + lane_off;
        // The whole 128-column block of the row is read from TMEM once (one
        // wait), masked in registers, reduced to its max with eight partial
        // maxima (short dependency chains), then exponentiated in place.
        const bool masked = (mode0 != kFull) || (mode1 != kFull);
        float v[128];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(s_addr + ch * 32, *reinterpret_cast<float(*)[32]>(&v[32 * ch]));
        tc::tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            mask_chunk(*reinterpret_cast<float(*)[32]>(&v[32 * ch]), ch < 2 ? mode0 : mode1, (ch & 1) * 32, rr);
        }
        float mxa[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mxa[x] = v[x];
#pragma unroll
        for (int x = 8; x < 128; x += 2) mxa[(x >> 1) & 7] = tc::max3(mxa[(x >> 1) & 7], v[x], v[x + 1]);
        const float mx = fmaxf(tc::max3(mxa[0], mxa[1], mxa[2]), fmaxf(tc::max3(mxa[3], mxa[4], mxa[5]),
                                                                          fmaxf(mxa[6], mxa[7])));
        const float m_cand = mx * sl2;  // every row sees >= 1 key of every block
        const bool need = (j > 0) && (m_cand > m_used + kRescaleLog2);
        const float alpha = need ? tc::fast_exp2(m_used - m_cand) : 1.f;
        if (j == 0 || need) m_used = m_cand;
        // P = exp2(S scale - m) (masked keys -> exp2(-inf) = 0), packed to
        // bf16 over S in place (P column c holds keys 2c, 2c+1); the scaling
        // and the row sum run on fp32 pairs
        const uint64_t sc2 = tc::f2_pack(sl2, sl2), nm2 = tc::f2_pack(-m_used, -m_used);
        uint64_t sa2[4] = {0, 0, 0, 0};  // four pairs of partial sums (+0.0f bits)
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            float t0, t1;
            tc::f2_unpack(tc::f2_fma(tc::f2_pack(v[32 * ch + 2 * x], v[32 * ch + 2 * x + 1]), sc2, nm2), t0, t1);
            const float e0 = tc::fast_exp2(t0), e1 = tc::fast_exp2(t1);
            sa2[x & 3] = tc::f2_add(sa2[x & 3], tc::f2_pack(e0, e1));
            pk[x] = tc::pack_bf16x2(e0, e1);
          }
          tc::tmem_st16u(s_addr + ch * 16, pk);
        }
        float sa[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) tc::f2_unpack(sa2[x], sa[2 * x], sa[2 * x + 1]);
        const float sum = ((sa[0] + sa[1]) + (sa[2] + sa[3])) + ((sa[4] + sa[5]) + (sa[6] + sa[7]));
        tc::tmem_st_wait();
        if (__any_sync(0xffffffffu, need)) {
          // O must hold every product so far before it is rescaled in place
          const int gp = gj - 1;
          if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_PV + gp % NS], (gp / NS) & 1, err)))) break;
          tc::fence_after();
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float o[32];
            tc::tmem_ld32(o_addr + ch * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            tc::tmem_st32(o_addr + ch * 32, o);
          }
          tc::tmem_st_wait();
        }
        l = l * alpha + sum;
        tc::fence_before();
        tc::mbar_arrive(&bars[B_PF + b]);
      }
      if (!ok) break;
      // epilogue: out = w RMSNorm(O / l)   (validity is warp-uniform: a warp's rows share a half)
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OF], tn & 1, err)))) break;
      tc::fence_after();
      // the rows go through a swizzled bf16 tile in shared memory and leave
      // with TMA stores (coalesced lines, not one 256-byte row per thread);
      // the previous tile's stores must have read the tile first
      if (tn > 0) {
        if (warp == 4 && lane == 0) {
          tc::bulk_wait_read_all();
          tc::mbar_arrive(&bars[B_OSE]);
        }
        if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OSE], (tn - 1) & 1, err)))) break;
      }
      if (half == 0 || ti.has_c1) {
        // one TMEM pass: the row of O in registers, its mean square, then
        // the scaled row packed to bf16
        const float inv = 1.f / l;
        const size_t row = (size_t)(ti.bh * (long long)L + 128LL * ti.p + r);
        // the row's log-sum-exp of its scaled scores, base 2 (saved for the backward pass)
        if (lse_out) lse_out[row] = m_used + __log2f(l);
        float o[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tc::tmem_ld32(o_addr + ch * 32, *reinterpret_cast<float(*)[32]>(&o[32 * ch]));
        tc::tmem_ld_wait();
        float ssa[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) ssa[x] = 0.f;
#pragma unroll
        for (int x = 0; x < D; ++x) ssa[x & 7] = fmaf(o[x], o[x], ssa[x & 7]);
        const float ss = ((ssa[0] + ssa[1]) + (ssa[2] + ssa[3])) + ((ssa[4] + ssa[5]) + (ssa[6] + ssa[7]));
        const float ms = ss * inv * inv * (1.f / D);
        const float cs = w * inv * rsqrtf(ms + eps);
        if (o_s) {
#pragma unroll
          for (int x = 0; x < D / 4; ++x)
            ((float4*)(o_s + row * D))[x] =
                make_float4(o[4 * x] * inv, o[4 * x + 1] * inv, o[4 * x + 2] * inv, o[4 * x + 3] * inv);
        }
        uint8_t* ost = smem + S::offOst + r * 128;
#pragma unroll
        for (int g8 = 0; g8 < D / 8; ++g8) {
          uint4 pk;
          uint32_t* p32 = (uint32_t*)&pk;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int cc = g8 * 8 + 2 * x;
            p32[x] = tc::pack_bf16x2(cs * nw_sm[cc] * o[cc], cs * nw_sm[cc + 1] * o[cc + 1]);
          }
          // 16-byte granule (g8 & 7) of row r in half (g8 >> 3), 128-byte swizzle
          *(uint4*)(ost + (g8 >> 3) * S::kHalf + (((g8 & 7) ^ (r & 7)) << 4)) = pk;
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars[B_OSF]);
      if (warp == 4 && lane == 0 && (ok = tc::mbar_wait(&bars[B_OSF], tn & 1, err))) {
        const int orow0 = (int)(ti.bh * (long long)L + 128LL * ti.p);
        for (int hh = 0; hh < D / 64; ++hh)
          for (int rc = 0; rc < (ti.has_c1 ? 2 : 1); ++rc)
            tc::tma_store_2d(&tm_o, smem + S::offOst + hh * S::kHalf + rc * (S::kHalf / 2), 64 * hh, orow0 + 64 * rc);
        tc::bulk_commit();
      }
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      cur = nxt;
      nxt = cur >= 0 ? take_w(tn + 2) : -1;
    }
    if (warp == 4 && lane == 0) tc::bulk_wait_all();  // the output tiles are written before exit
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  });
  return fn;
}

}  // namespace

// [rows, D] bf16 row-major matrix viewed as 64 x 64 boxes, 128-byte swizzle.
bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_tc_t(const Problem& p, const void* q, const void* k, const void* v,
                               const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel,
                               const float* gate, const float* nw_s, void* out, float* o_s, float* lse_out,
                               int* err, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  const long long rows = p.BH * p.L;
  if (!make_tile_map(&mq, q, rows, D) || !make_tile_map(&mk, k, rows, D) || !make_tile_map(&mv, v, rows, D) ||
      !make_tile_map(&mo, out, rows, D))
    return cudaErrorInvalidValue;
  auto kern = softmax_tc_kernel<D>;
  const int smem = SoftmaxSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int T = (p.N + 1) / 2;
  const long long tiles = p.BH * T;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  kern<<<grid, 256, smem, st>>>(mq, mk, mv, mo, nprev, sel_idx, sel, p.L, p.N, T, p.BH,
                                p.scale * 1.4426950408889634f, gate, nw_s, p.eps, (__nv_bfloat16*)out, o_s,
                                lse_out, err, err + 1);
  return cudaGetLastError();
}

cudaError_t launch_softmax_tc(const Problem& p, const void* q, const void* k, const void* v,
                              const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel,
                              const float* gate, const float* nw_s, void* out, float* o_s, float* lse_out,
                              int* err, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? launch_tc_t<64>(p, q, k, v, nprev, sel_idx, sel, gate, nw_s, out, o_s, lse_out, err, st)
                   : launch_tc_t<128>(p, q, k, v, nprev, sel_idx, sel, gate, nw_s, out, o_s, lse_out, err, st);
}

}  // namespace nats
