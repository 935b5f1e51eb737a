// gdn_scan_tc.cu - Gated DeltaNet phase 2 on the 5th-generation tensor cores:
// the chunk-by-chunk state scan with pseudo-update and rollback (bf16 path).
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the linear state is pseudo-updated for every
// chunk; for a chunk that chose softmax it is rolled back to the chunk start.
// With the phase-1 factors of a chunk (S0 = state at its start, dv x dk;
// G = in-chunk cumulative log-decay, gamma = e^G; Q~ = diag(scale gamma) Q;
// K~ = diag(gamma_C / gamma) K, both formed here in shared memory from the
// chunk's Q and K tiles):
//   Delta^T = U^T - S0 W^T                    (dv x 64)
//   O^T     = S0 Q~^T + Delta^T P^T           (dv x 64)
//   S_C     = gamma_C S0 + Delta^T K~         (linear chunks only)
// Everything is computed transposed, so the state row dv is the TMEM lane:
// the per-chunk elementwise work spreads over all 128 lanes (all four SM
// sub-partitions), and S0 and Delta^T stay in TMEM as MMA A operands.
//
// One CTA per (b, h) walks the N chunks in order; the fp32 state S stays in
// TMEM for the whole sequence, next to its bf16 copy S0.  Per chunk c:
//   MMA1  X = S0 W^T, then O = S0 Q~^T, into TMEM buffer c % 2 (M = 128
//         lanes >= dv, N = 64 each, K = dk; X first, so Delta starts early)
//   all   Delta^T = U^T - X -> TMEM (bf16)
//   MMA3  S += Delta^T K~                (linear chunks only), then
//   MMA2  O += Delta^T P^T
//   all   O^T of chunk c - 1 -> o_l while MMA3 runs, then S -> bf16 S0 and
//         S *= gamma_C of the next chunk when it is linear
// Roles (448 threads): warps 0-7 elementwise, warp w owning TMEM lanes
// 32 (w % 4) .. +31 and half (w / 4) of the columns; warp 8 TMA producer
// (W, Q, K, U^T, P and G of coming chunks, three stages); warp 9 TMEM owner
// and MMA issuer; warps 10-13 scale the staged Q and K rows in place into Q~
// and K~ (two chunks ahead of the products that read them).  Every wait is
// bounded (tc::kWaitLimitNs).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {

bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D);

namespace {

template <int D>
struct ScanSmem {
  static constexpr int kWQ = 128 * D * 2;  // [W; Q] tile: 128 lines (t), D/64 halves of 16 KiB
  static constexpr int kK = 64 * D * 2;    // K chunk: 64 lines (t), D/64 halves of 8 KiB
  static constexpr int kU = D * 64 * 2;    // U^T chunk: D lines (dv) x 64 cols (t), 8 KiB per 64 lines
  static constexpr int kP = 64 * 64 * 2;   // P chunk: 64 lines (t) x 64 cols (i)
  static constexpr int kStage = kWQ + kK + kU + kP;
  static constexpr int kStages = 3;  // chunks in flight: the loads run two chunks ahead
  static constexpr int offStage = 0;
  static constexpr int offG = kStages * kStage;  // fp32 [kStages][64]: G of the staged chunks
  static constexpr int offBar = offG + kStages * 64 * 4;
  static constexpr int kNumBars = 16;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
};

// SB_OFREE + b: O^T of the chunks using O buffer b has been read (one barrier
// per buffer, so a waiter is never two phases behind)
// SB_SCALED + s: Q~ and K~ of stage s are in place
enum {
  SB_FULL = 0, SB_EMPTY = 3, SB_S0 = 6, SB_Z = 7, SB_DELTA = 8, SB_OFREE = 9, SB_SDONE = 11, SB_DONE = 12,
  SB_SCALED = 13
};

// TMEM columns
constexpr uint32_t kColXO = 0;     // two buffers of 128 columns: [S0 W^T | O^T] of chunks c % 2
constexpr uint32_t kColS = 256;    // state, D columns (fp32)
constexpr uint32_t kColS0 = 384;   // state bf16, D / 2 columns (two dk per column)
constexpr uint32_t kColDT = 448;   // Delta^T bf16, 32 columns (64 t)

// byte offset of element (line, col) in a 128-byte-swizzled tile whose
// 64-column halves are `half_bytes` apart
__device__ __forceinline__ uint32_t sw_off(int line, int col, int half_bytes) {
  return (uint32_t)((col >> 6) * half_bytes + line * 128 + ((((col & 63) >> 3) ^ (line & 7)) << 4) + (col & 7) * 2);
}

template <int D>
__global__ void __launch_bounds__(448, 1)
    gdn_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_u,
                       const __grid_constant__ CUtensorMap tm_p, const uint8_t* __restrict__ sel,
                       const float* __restrict__ G, int L, int N, float scale, float* __restrict__ o_l,
                       __nv_bfloat16* __restrict__ o_l16,
                       float* __restrict__ state_out, float* __restrict__ s0_out, int* __restrict__ err) {
  using S = ScanSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);

  const long long bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      tc::mbar_init(&bars[SB_FULL + s], 1);
      tc::mbar_init(&bars[SB_EMPTY + s], 1);
    }
    tc::mbar_init(&bars[SB_S0], 256);
    tc::mbar_init(&bars[SB_Z], 1);
    tc::mbar_init(&bars[SB_DELTA], 256);
    for (int b = 0; b < 2; ++b) tc::mbar_init(&bars[SB_OFREE + b], 256);
    tc::mbar_init(&bars[SB_SDONE], 1);
    tc::mbar_init(&bars[SB_DONE], 1);
    for (int s = 0; s < S::kStages; ++s) tc::mbar_init(&bars[SB_SCALED + s], 4);
    tc::fence_barrier_init();
  }
  if (warp == 9) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_w);
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_u);
      tc::prefetch_tensormap(&tm_p);
      int issued[S::kStages] = {};
      bool ok = true;
      for (int c = 0; c < N; ++c) {
        const int s = c % S::kStages;
        if (!(ok = tc::mbar_wait(&bars[SB_EMPTY + s], ((c / S::kStages) & 1) ^ 1, err))) break;
        uint8_t* WQ = smem + S::offStage + s * S::kStage;
        uint8_t* Kb = WQ + S::kWQ;
        uint8_t* Ub = Kb + S::kK;
        uint8_t* Pb = Ub + S::kU;
        const int yc = (int)((bh * N + c) * 64);   // row of this chunk in W / P / Q~ / K / ...
        const int yt = (int)(bh * L + 64LL * c);   // row of this chunk in Q~ / K
        const int yu = (int)((bh * N + c) * D);    // first line of this chunk in U^T
        tc::mbar_arrive_expect_tx(&bars[SB_FULL + s], S::kStage + 64 * 4);
        tc::bulk_load_1d(smem + S::offG + s * 256, G + yt, 256, &bars[SB_FULL + s]);
        for (int h = 0; h < D / 64; ++h) {
          tc::tma_load_2d(WQ + h * 16384, &tm_w, 64 * h, yc, &bars[SB_FULL + s]);
          tc::tma_load_2d(WQ + h * 16384 + 8192, &tm_q, 64 * h, yt, &bars[SB_FULL + s]);
          tc::tma_load_2d(Kb + h * 8192, &tm_k, 64 * h, yt, &bars[SB_FULL + s]);
          tc::tma_load_2d(Ub + h * 8192, &tm_u, 0, yu + 64 * h, &bars[SB_FULL + s]);
        }
        tc::tma_load_2d(Pb, &tm_p, 0, yc, &bars[SB_FULL + s]);
        issued[s]++;
      }
      for (int s = 0; s < S::kStages; ++s) {
        if (issued[s] == 0) continue;
        tc::mbar_wait(&bars[SB_FULL + s], (issued[s] - 1) & 1, nullptr);
        if (ok) tc::mbar_wait(&bars[SB_EMPTY + s], (issued[s] - 1) & 1, err);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id2 = tc::idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id3 = tc::idesc_bf16_f32(128, D, false, true);
      // descriptors are built once per stage; each MMA only offsets them
      const uint32_t w0 = tc::smem_u32(smem + S::offStage);
      const uint64_t wd0 = tc::smem_desc_sw128(w0, 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(w0 + S::kWQ, 8192, 1024);
      const uint64_t pd0 = tc::smem_desc_sw128(w0 + S::kWQ + S::kK + S::kU, 16, 1024);
      bool ok = true;
      uint8_t sel_c = sel[bh * N];  // selections are read one chunk ahead (global latency)
      for (int c = 0; c < N && ok; ++c) {
        const int s = c % S::kStages;
        const uint8_t sel_n = (c + 1 < N) ? sel[bh * N + c + 1] : 0;
        const uint32_t tX = tmem + kColXO + (c & 1) * 128, tO = tX + 64;
        const uint32_t sb = s * S::kStage;
        const uint64_t wd = tc::desc_add(wd0, sb), kd = tc::desc_add(kd0, sb), pd = tc::desc_add(pd0, sb);
        if (!(ok = tc::mbar_wait(&bars[SB_FULL + s], (c / S::kStages) & 1, err))) break;
        if (!(ok = tc::mbar_wait(&bars[SB_SCALED + s], (c / S::kStages) & 1, err))) break;
        if (!(ok = tc::mbar_wait(&bars[SB_S0], c & 1, err))) break;
        tc::fence_after();
        // X = S0 W^T first (the W lines of the stacked [W; Q~] tile), so that
        // Delta can start; then the first term of O, S0 Q~^T (the Q~ lines),
        // once O buffer c % 2 has been read out
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offb = (kk >> 2) * 16384 + (kk & 3) * 32;
          tc::mma_bf16_ts(tX, tmem + kColS0 + kk * 8, tc::desc_add(wd, offb), id2, kk > 0);
        }
        tc::mma_commit(&bars[SB_Z]);
        if (c >= 2 && !(ok = tc::mbar_wait(&bars[SB_OFREE + (c & 1)], ((c - 2) / 2) & 1, err))) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offb = (kk >> 2) * 16384 + (kk & 3) * 32 + 8192;
          tc::mma_bf16_ts(tO, tmem + kColS0 + kk * 8, tc::desc_add(wd, offb), id2, kk > 0);
        }
        if (!(ok = tc::mbar_wait(&bars[SB_DELTA], c & 1, err))) break;
        tc::fence_after();
        // the state update first (the next chunk waits for it), then O
        if (sel_c != 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(tmem + kColS, tmem + kColDT + kk * 8, tc::desc_add(kd, kk * 2048), id3, 1);
        }
        tc::mma_commit(&bars[SB_SDONE]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16_ts(tO, tmem + kColDT + kk * 8, tc::desc_add(pd, kk * 32), id2, 1);
        tc::mma_commit(&bars[SB_EMPTY + s]);
        sel_c = sel_n;
      }
      tc::mma_commit(&bars[SB_DONE]);
      tc::mbar_wait(&bars[SB_DONE], 0, err);
    }
  } else if (warp >= 10) {
    // ----------------------------------------- Q~ and K~ in place (warps 10-13)
    // Q~_t = scale e^{G_t} q_t and K~_t = e^{G_C - G_t} k_t, rounded to bf16;
    // a thread takes 16-byte granules (8 features of one token) of both tiles
    constexpr int VPR = D / 8;
    const int el = threadIdx.x - 320;
    bool ok = true;
    for (int c = 0; c < N && ok; ++c) {
      const int s = c % S::kStages;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_FULL + s], (c / S::kStages) & 1, err)))) break;
      uint8_t* Qb = smem + S::offStage + s * S::kStage + 8192;  // Q lines follow the W lines in each half
      uint8_t* Kb = smem + S::offStage + s * S::kStage + S::kWQ;
      const float* Gs = (const float*)(smem + S::offG + s * 256);
      const float GC = Gs[63];
#pragma unroll 2
      for (int e = el; e < 64 * VPR; e += 128) {
        const int t = e / VPR, x = e % VPR;
        const uint32_t off = (uint32_t)(t * 128 + ((((x & 7) ^ (t & 7))) << 4));
        const float Gt = Gs[t];
        const float fq = scale * __expf(Gt), fk = __expf(GC - Gt);
        uint4* pq = (uint4*)(Qb + (x >> 3) * 16384 + off);
        uint4* pk = (uint4*)(Kb + (x >> 3) * 8192 + off);
        const uint4 iq = *pq, ik = *pk;
        const __nv_bfloat162* hq = (const __nv_bfloat162*)&iq;
        const __nv_bfloat162* hk = (const __nv_bfloat162*)&ik;
        uint4 oq, ok4;
        uint32_t* q32 = (uint32_t*)&oq;
        uint32_t* k32 = (uint32_t*)&ok4;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 a = __bfloat1622float2(hq[u]), b = __bfloat1622float2(hk[u]);
          q32[u] = tc::pack_bf16x2(a.x * fq, a.y * fq);
          k32[u] = tc::pack_bf16x2(b.x * fk, b.y * fk);
        }
        *pq = oq;
        *pk = ok4;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[SB_SCALED + s]);
    }
  } else {
    // ------------------------------------------------- elementwise (warps 0-7)
    const int q4 = warp & 3;        // TMEM lane quarter
    const int r = 32 * q4 + lane;   // TMEM lane = state row (dv)
    const int hf = warp >> 2;       // column half
    const bool has_row = r < D;     // warp-uniform (lanes come in 32s, D is 64 or 128)
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    constexpr int SC = D / 2;       // state columns per thread
    // S = 0 in TMEM, fp32 and bf16
    {
      float z[32];
      uint32_t zu[16];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) zu[i] = 0u;
#pragma unroll
      for (int ch = 0; ch < SC / 32; ++ch) tc::tmem_st32(tmem + kColS + lane_off + hf * SC + ch * 32, z);
#pragma unroll
      for (int ch = 0; ch < SC / 32; ++ch) tc::tmem_st16u(tmem + kColS0 + lane_off + hf * (SC / 2) + ch * 16, zu);
      tc::tmem_st_wait();
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_S0]);
    }
    // O work of chunk cc: o_l[t][dv] for t = 32 hf .. +31; a warp's 32 lanes
    // write 128 contiguous bytes per t
    auto o_phase = [&](int cc) {
      float o[32];  // warp-collective load (lanes >= D hold no state row)
      tc::tmem_ld32(tmem + kColXO + (cc & 1) * 128 + 64 + lane_off + 32 * hf, o);
      tc::tmem_ld_wait();
      if (has_row) {
        const size_t off = (bh * (long long)L + 64LL * cc + 32 * hf) * D + r;
        if (o_l16) {  // bf16 copy for the merge (the caller did not ask for o_l)
#pragma unroll
          for (int i = 0; i < 32; ++i) o_l16[off + (size_t)i * D] = __float2bfloat16_rn(o[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o_l[off + (size_t)i * D] = o[i];
        }
      }
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_OFREE + (cc & 1)]);
    };
    bool ok = true;
    // per-chunk selections and end-of-chunk log-decays, read two chunks ahead
    // (a global load on the critical path costs more than a chunk's MMAs)
    const uint8_t* selh = sel + bh * N;
    const float* Gh = G + bh * (long long)L;
    bool lin_c = selh[0] != 0;
    bool lin_n = N > 1 && selh[1] != 0;
    float gC_n = N > 1 ? Gh[64 + 63] : 0.f;
    // U^T of a chunk is read into registers one chunk ahead, while the
    // previous chunk waits for its state update
    uint4 uvn[4];
    auto load_u = [&](int cc) -> bool {
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_FULL + cc % S::kStages], (cc / S::kStages) & 1, err)))
        return false;
      if (has_row) {
        const uint8_t* Ub = smem + S::offStage + (cc % S::kStages) * S::kStage + S::kWQ + S::kK;
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          uvn[g8] = *(const uint4*)(Ub + sw_off(r & 63, 32 * hf + 8 * g8, 0) + (r >> 6) * 8192);
      }
      return true;
    };
    if (N > 0) ok = load_u(0);
    for (int c = 0; c < N && ok; ++c) {
      const bool has_nn = c + 2 < N;
      const uint8_t sel_nn = has_nn ? selh[c + 2] : 0;
      const float gC_nn = has_nn ? Gh[64LL * (c + 2) + 63] : 0.f;
      const bool lin = lin_c, lin_next = lin_n;
      const float gnext = lin_next ? __expf(gC_n) : 1.f;
      const uint32_t tX = tmem + kColXO + (c & 1) * 128 + lane_off;
      // ---- Delta^T (columns t = 32 hf .. 32 hf + 31 of this row)
      {
        float x[32];
        uint32_t pd[16];
        uint4 uv[4];
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) uv[g8] = uvn[g8];
        if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_Z], c & 1, err)))) break;
        tc::fence_after();
        tc::tmem_ld32(tX + 32 * hf, x);
        tc::tmem_ld_wait();
        if (has_row) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const __nv_bfloat162* u2 = (const __nv_bfloat162*)&uv[g8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 uf = __bfloat1622float2(u2[i]);
              pd[4 * g8 + i] = tc::pack_bf16x2(uf.x - x[8 * g8 + 2 * i], uf.y - x[8 * g8 + 2 * i + 1]);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) pd[i] = 0u;
        }
        tc::tmem_st16u(tmem + kColDT + lane_off + 16 * hf, pd);
        tc::tmem_st_wait();
        tc::fence_before();
        tc::mbar_arrive(&bars[SB_DELTA]);
      }
      if (c + 1 < N && !(ok = load_u(c + 1))) break;
      // O of the previous chunk (complete: its last product was issued
      // before this chunk's S0 W^T, which Delta waited for), while this
      // chunk's state update runs
      if (c > 0) o_phase(c - 1);
      // ---- state: bf16 copy after this chunk's update, and the decay of the
      // next linear chunk applied ahead of its MMA3
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_SDONE], c & 1, err)))) break;
      tc::fence_after();
      // 32 state columns at a time (registers): the bf16 copy first, it is
      // on the critical path
      if (lin && has_row) {
#pragma unroll 1
        for (int ch = 0; ch < SC / 32; ++ch) {
          float v[32];
          tc::tmem_ld32(tmem + kColS + lane_off + hf * SC + ch * 32, v);
          tc::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = tc::pack_bf16x2(v[2 * i], v[2 * i + 1]);
          tc::tmem_st16u(tmem + kColS0 + lane_off + (hf * SC + ch * 32) / 2, pk);
        }
        tc::tmem_st_wait();
      }
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_S0]);
      // the state at the start of chunk c + 1 (after this chunk's update or
      // rollback), fp32, when the caller keeps them (backward recompute),
      // stored transposed ([dk][dv]): for each column the warp's 32 rows are
      // 128 contiguous bytes; no product writes S before this thread's next
      // Delta
      if (s0_out && c + 1 < N && has_row) {
#pragma unroll 1
        for (int ch = 0; ch < SC / 32; ++ch) {
          float v[32];
          tc::tmem_ld32(tmem + kColS + lane_off + hf * SC + ch * 32, v);
          tc::tmem_ld_wait();
          float* dst = s0_out + ((bh * N + c + 1) * D + hf * SC + ch * 32) * (long long)D + r;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[(size_t)i * D] = v[i];
        }
      }
      // the next chunk's MMA3 accumulates onto gamma_C S: scale now, off the
      // critical path (that MMA3 also waits for this thread's next Delta)
      if (lin_next && has_row) {
#pragma unroll 1
        for (int ch = 0; ch < SC / 32; ++ch) {
          float v[32];
          tc::tmem_ld32(tmem + kColS + lane_off + hf * SC + ch * 32, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gnext;
          tc::tmem_st32(tmem + kColS + lane_off + hf * SC + ch * 32, v);
        }
        tc::tmem_st_wait();
      }
      // the loads for chunk c + 2 issued at the top are consumed only here
      lin_c = lin_n;
      lin_n = sel_nn != 0;
      gC_n = gC_nn;
    }
    // the last chunk's O work, once every MMA has completed
    if (ok && N > 0 && (ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_DONE], 0, err)))) {
      tc::fence_after();
      o_phase(N - 1);
    }
    if (ok && state_out && has_row) {
      tc::fence_after();
#pragma unroll 1
      for (int ch = 0; ch < SC / 32; ++ch) {
        float v[32];
        tc::tmem_ld32(tmem + kColS + lane_off + hf * SC + ch * 32, v);
        tc::tmem_ld_wait();
        float* dst = state_out + (bh * D + r) * (long long)D + hf * SC + ch * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) ((float4*)dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
static cudaError_t launch_scan_tc_t(const Problem& p, const void* q, const void* k, const uint8_t* sel,
                                    const float* G, const void* W16, const void* UT16, const void* P16,
                                    float* o_l, __nv_bfloat16* o_l16, float* state_out, float* s0_out, int* err,
                                    cudaStream_t st) {
  CUtensorMap mw, mq, mk, mu, mp;
  const long long rows = p.BH * p.L;  // = BH * N * 64
  if (!make_tile_map(&mw, W16, rows, D) || !make_tile_map(&mq, q, rows, D) || !make_tile_map(&mk, k, rows, D) ||
      !make_tile_map(&mu, UT16, p.BH * (long long)p.N * D, 64) || !make_tile_map(&mp, P16, rows, 64))
    return cudaErrorInvalidValue;
  auto kern = gdn_scan_tc_kernel<D>;
  const int smem = ScanSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (s0_out) {  // chunk 0 starts from the zero state
    e = cudaMemset2DAsync(s0_out, (size_t)p.N * D * D * sizeof(float), 0, (size_t)D * D * sizeof(float),
                          (size_t)p.BH, st);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)p.BH, 448, smem, st>>>(mw, mq, mk, mu, mp, sel, G, p.L, p.N, p.scale, o_l, o_l16, state_out,
                                          s0_out, err);
  return cudaGetLastError();
}

cudaError_t launch_gdn_scan_tc(const Problem& p, const void* q, const void* k, const uint8_t* sel, const float* G,
                               const void* W16, const void* UT16, const void* P16, float* o_l, void* o_l16,
                               float* state_out, int* err, cudaStream_t st, float* s0_out) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  __nv_bfloat16* ol16 = (__nv_bfloat16*)o_l16;
  return p.d == 64 ? launch_scan_tc_t<64>(p, q, k, sel, G, W16, UT16, P16, o_l, ol16, state_out, s0_out, err, st)
                   : launch_scan_tc_t<128>(p, q, k, sel, G, W16, UT16, P16, o_l, ol16, state_out, s0_out, err, st);
}

}  // namespace nats
