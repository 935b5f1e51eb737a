// softmax_bwd_tc.cu - the softmax branch of the backward pass on the
// 5th-generation tensor cores (bf16 layers): tcgen05.mma with accumulators in
// TMEM, operands staged by TMA.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" items 3 and 5: every query of chunk c attends to the
// retained chunks (the softmax chunks before c) plus its own chunk causally;
// the layer is trained end to end.  With z = scale q . k, P = softmax(z) over
// the visible keys, dO the gradient of the branch output and
// delta_i = dO_i . O_i:
//   dP = dO V^T,  dS = P (dP - delta),  dq = scale dS K,  dk = scale dS^T Q,
//   dv = P^T dO.
//
// Two kernels, one CTA per 128-row tile (two 64-token chunks of one head),
// heaviest tiles first.  Roles: warp 0 TMA producer, warp 1 TMEM owner and
// MMA issuer (one thread), warps 4-7 elementwise (thread r owns TMEM lane r).
//   softmax_bwd_dq_tc_kernel  query tile: key blocks = the retained chunks
//     before it, in pairs, then the diagonal pair (the forward's order).
//     Pass 1 recomputes S = Q K^T for the row log-sum-exp (written out for the
//     second kernel); pass 2 recomputes S and forms dP = dO V^T, dS in place
//     of S (bf16), dQ += dS K.  TMEM: two S buffers, dP, dQ.
//   softmax_bwd_dkv_tc_kernel  key tiles, in two launches: the chunk pairs
//     against their own query pair (each chunk's causal block), then pairs
//     of the head's softmax chunks (the compacted list, no key row that
//     later queries cannot see) against every later query pair; taken one
//     64-query chunk at a time: S^T = K Q^T, dP^T = V dO^T (N = 64, issued
//     one chunk ahead into the other TMEM half); P^T and dS^T in place
//     (bf16); dV += P^T dO, dK += dS^T Q.  TMEM: S^T x 2, dP^T x 2 (64
//     columns each), dV, dK.
// Every wait is bounded (tc::kWaitLimitNs); on expiry a kernel records an
// error, drains what it issued and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {

bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D);

namespace {

enum { kFull = 0, kCausal = 1, kNone = 2 };
constexpr int kHalf = 128 * 128;  // bytes of one 128-line x 64-column bf16 block

// ------------------------------------------------------------------- dq
template <int D>
struct DqSm {
  static constexpr int kT = 128 * D * 2;  // a 128-line tile
  static constexpr int offQ = 0;
  static constexpr int offO = offQ + kT;
  static constexpr int offK = offO + kT;   // K ring, 2 deep
  static constexpr int offV = offK + 2 * kT;  // V ring, 2 deep
  static constexpr int offBar = offV + 2 * kT;
  static constexpr int kNumBars = 16;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
};
enum { DQ_QF = 0, DQ_KF = 1, DQ_KE = 3, DQ_VF = 5, DQ_VE = 7, DQ_SF = 9, DQ_SR = 11, DQ_PF = 13, DQ_DONE = 14,
       DQ_DR = 15 };

struct QTile {
  int p, c0, n0, nbp, nb;
  long long bh;
  bool has_c1, c0_soft;
};

__device__ __forceinline__ QTile q_tile(int i, long long BH, int T, int N, const int32_t* nprev,
                                        const uint8_t* sel) {
  QTile t;
  t.p = T - 1 - (int)(i / BH);  // heaviest first (the retained set grows with the position)
  t.bh = i % BH;
  t.c0 = 2 * t.p;
  t.has_c1 = t.c0 + 1 < N;
  t.n0 = nprev[t.bh * N + t.c0];
  t.nbp = (t.n0 + 1) >> 1;
  t.nb = t.nbp + 1;
  t.c0_soft = sel[t.bh * N + t.c0] == 0;
  return t;
}

// masked entries of 32 consecutive columns become -inf (row view: key0 is
// the key index of v[0] within its chunk, rr the query's index in its chunk)
__device__ __forceinline__ void mask_keys(float (&v)[32], int mode, int key0, int rr) {
  if (mode == kNone) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = -INFINITY;
  } else if (mode == kCausal) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = (key0 + x <= rr) ? v[x] : -INFINITY;
  }
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    softmax_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                             const int32_t* __restrict__ nprev, const int32_t* __restrict__ sel_idx,
                             const uint8_t* __restrict__ sel, int L, int N, int T, long long BH, float scale,
                             const float* __restrict__ delta, float* __restrict__ lse,
                             const float* __restrict__ lse_in, float* __restrict__ dq, int* __restrict__ err) {
  using S = DqSm<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const QTile ti = q_tile(blockIdx.x, BH, T, N, nprev, sel);
  const long long row0 = ti.bh * (long long)L;
  const int nb = ti.nb;
  const int gp = lse_in ? 0 : nb;  // blocks of pass 1 (none when the forward's row statistic is given)
  const float sl2 = scale * 1.4426950408889634f;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[DQ_QF], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[DQ_KF + s], 1);
      tc::mbar_init(&bars[DQ_KE + s], 1);
      tc::mbar_init(&bars[DQ_VF + s], 1);
      tc::mbar_init(&bars[DQ_VE + s], 1);
      tc::mbar_init(&bars[DQ_SF + s], 1);
      tc::mbar_init(&bars[DQ_SR + s], 128);
    }
    tc::mbar_init(&bars[DQ_PF], 1);
    tc::mbar_init(&bars[DQ_DONE], 1);
    tc::mbar_init(&bars[DQ_DR], 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;  // S0 | S1 | dP | dQ, 128 columns each

  // key chunk pair of block j
  auto pair = [&](int j, int& a, int& b) {
    if (j < ti.nbp) {
      a = sel_idx[ti.bh * N + 2 * j];
      b = (2 * j + 1 < ti.n0) ? sel_idx[ti.bh * N + 2 * j + 1] : ti.c0;
    } else {
      a = ti.c0;
      b = ti.has_c1 ? ti.c0 + 1 : ti.c0;
    }
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_v);
      tc::prefetch_tensormap(&tm_do);
      tc::mbar_arrive_expect_tx(&bars[DQ_QF], 2 * S::kT);
      for (int h = 0; h < D / 64; ++h)
        for (int rc = 0; rc < 2; ++rc) {
          const int y = (int)(row0 + 128LL * ti.p + 64 * rc);
          tc::tma_load_2d(smem + S::offQ + h * kHalf + rc * (kHalf / 2), &tm_q, 64 * h, y, &bars[DQ_QF]);
          tc::tma_load_2d(smem + S::offO + h * kHalf + rc * (kHalf / 2), &tm_do, 64 * h, y, &bars[DQ_QF]);
        }
      bool ok = true;
      auto load_block = [&](const CUtensorMap* tm, uint8_t* buf, uint64_t* full, int j) {
        int a, b;
        pair(j, a, b);
        tc::mbar_arrive_expect_tx(full, S::kT);
        for (int slot = 0; slot < 2; ++slot)
          for (int h = 0; h < D / 64; ++h)
            tc::tma_load_2d(buf + h * kHalf + slot * (kHalf / 2), tm, 64 * h, (int)(row0 + 64LL * (slot ? b : a)),
                            full);
      };
      // K blocks of both passes through the K ring; the V block of a pass-2
      // block right after its K block
      int nv = 0, nk = 0;
      for (int g = 0; g < gp + nb && ok; ++g) {
        const int ks = g & 1;
        if (!(ok = tc::mbar_wait(&bars[DQ_KE + ks], ((g >> 1) & 1) ^ 1, err))) break;
        load_block(&tm_k, smem + S::offK + ks * S::kT, &bars[DQ_KF + ks], g < gp ? g : g - gp);
        ++nk;
        if (g >= gp) {
          const int j = g - gp, vs = j & 1;
          if (!(ok = tc::mbar_wait(&bars[DQ_VE + vs], ((j >> 1) & 1) ^ 1, err))) break;
          load_block(&tm_v, smem + S::offV + vs * S::kT, &bars[DQ_VF + vs], j);
          ++nv;
        }
      }
      // every copy issued has landed before the CTA may exit
      tc::mbar_wait(&bars[DQ_QF], 0, nullptr);
      for (int s = 0; s < 2; ++s) {
        const int nks = nk > s ? (nk - 1 - s) / 2 + 1 : 0;
        if (nks > 0) tc::mbar_wait(&bars[DQ_KF + s], (nks - 1) & 1, nullptr);
        const int nvs = nv > s ? (nv - 1 - s) / 2 + 1 : 0;
        if (nvs > 0) tc::mbar_wait(&bars[DQ_VF + s], (nvs - 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_qk = tc::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, D, false, true);
      const uint64_t qd = tc::smem_desc_sw128(tc::smem_u32(smem + S::offQ), 16, 1024);
      const uint64_t od = tc::smem_desc_sw128(tc::smem_u32(smem + S::offO), 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(tc::smem_u32(smem + S::offK), 16, 1024);
      const uint64_t kn0 = tc::smem_desc_sw128(tc::smem_u32(smem + S::offK), kHalf, 1024);
      const uint64_t vd0 = tc::smem_desc_sw128(tc::smem_u32(smem + S::offV), 16, 1024);
      const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
      bool ok = tc::mbar_wait(&bars[DQ_QF], 0, err);
      // S_g = Q K_g^T into buffer g & 1, once the elementwise warps are done
      // with the buffer's previous block
      auto issue_s = [&](int g) -> bool {
        const int b = g & 1;
        if (!tc::mbar_wait(&bars[DQ_KF + b], (g >> 1) & 1, err)) return false;
        if (g >= 2 && !tc::mbar_wait(&bars[DQ_SR + b], ((g - 2) >> 1) & 1, err)) return false;
        tc::fence_after();
        const uint64_t kd = tc::desc_add(kd0, b * S::kT);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + 128 * b, tc::desc_add(qd, off), tc::desc_add(kd, off), id_qk, kk > 0);
        }
        tc::mma_commit(&bars[DQ_SF + b]);
        return true;
      };
      // pass 1: S only, for the row statistics
      for (int g = 0; g < gp && ok; ++g) {
        if (!(ok = issue_s(g))) break;
        tc::mma_commit(&bars[DQ_KE + (g & 1)]);
      }
      // pass 2: S (one block ahead), dP = dO V^T, then dQ += dS K
      if (ok) ok = issue_s(gp);
      for (int j = 0; j < nb && ok; ++j) {
        const int g = gp + j, b = g & 1, vs = j & 1;
        if (!(ok = tc::mbar_wait(&bars[DQ_VF + vs], (j >> 1) & 1, err))) break;
        // the dP buffer: the elementwise warps are done with the previous block
        if (j > 0 && !(ok = tc::mbar_wait(&bars[DQ_SR + ((g - 1) & 1)], ((g - 1) >> 1) & 1, err))) break;
        tc::fence_after();
        const uint64_t vd = tc::desc_add(vd0, vs * S::kT);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tdP, tc::desc_add(od, off), tc::desc_add(vd, off), id_qk, kk > 0);
        }
        tc::mma_commit(&bars[DQ_PF]);
        tc::mma_commit(&bars[DQ_VE + vs]);
        if (j + 1 < nb && !(ok = issue_s(g + 1))) break;
        // dS of block g is in place of its S
        if (!(ok = tc::mbar_wait(&bars[DQ_SR + b], (g >> 1) & 1, err))) break;
        tc::fence_after();
        const uint64_t kn = tc::desc_add(kn0, b * S::kT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16_ts(tdQ, tmem + 128 * b + kk * 8, tc::desc_add(kn, kk * 2048), id_pv, (j > 0) || (kk > 0));
        tc::mma_commit(&bars[DQ_KE + b]);
      }
      if (ok) tc::mma_commit(&bars[DQ_DONE]);
      tc::mma_commit(&bars[DQ_DR]);
      tc::mbar_wait(&bars[DQ_DR], 0, nullptr);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------- elementwise
    const int r = threadIdx.x - 128;
    const int half = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const bool valid = half == 0 || ti.has_c1;
    const size_t row = (size_t)(row0 + 128LL * ti.p + r);
    const float dl = valid ? delta[row] : 0.f;
    auto modes = [&](int j, int& m0, int& m1) {
      if (j < ti.nbp) {
        m0 = kFull;
        m1 = (2 * j + 1 < ti.n0) ? kFull : kNone;
      } else if (half == 0) {
        m0 = kCausal;
        m1 = kNone;
      } else {
        m0 = ti.has_c1 ? (ti.c0_soft ? kFull : kNone) : kFull;
        m1 = ti.has_c1 ? kCausal : kNone;
      }
    };
    bool ok = true;
    // pass 1: running max and sum in the exp2 domain
    float m = -INFINITY, l = 0.f;
    for (int g = 0; g < gp && ok; ++g) {
      const int b = g & 1;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[DQ_SF + b], (g >> 1) & 1, err)))) break;
      tc::fence_after();
      int md0, md1;
      modes(g, md0, md1);
      float v[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        tc::tmem_ld32(tmem + 128 * b + lane_off + 32 * ch, *reinterpret_cast<float(*)[32]>(&v[32 * ch]));
      tc::tmem_ld_wait();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        mask_keys(*reinterpret_cast<float(*)[32]>(&v[32 * ch]), ch < 2 ? md0 : md1, (ch & 1) * 32, rr);
      float mx = -INFINITY;
#pragma unroll
      for (int x = 0; x < 128; ++x) mx = fmaxf(mx, v[x]);
      const float mn = fmaxf(m, mx * sl2);  // finite: every row sees a key of every block
      float sum = 0.f;
#pragma unroll
      for (int x = 0; x < 128; ++x) sum += tc::fast_exp2(v[x] * sl2 - mn);
      l = l * tc::fast_exp2(m - mn) + sum;
      m = mn;
      tc::fence_before();
      tc::mbar_arrive(&bars[DQ_SR + b]);
    }
    const float lse2 = lse_in ? (valid ? lse_in[row] : 0.f) : m + __log2f(l);
    if (ok && valid && !lse_in) lse[row] = lse2;
    // pass 2: dS = P (dP - delta) in place of S
    for (int j = 0; j < nb && ok; ++j) {
      const int g = gp + j, b = g & 1;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[DQ_SF + b], (g >> 1) & 1, err)))) break;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[DQ_PF], j & 1, err)))) break;
      tc::fence_after();
      int md0, md1;
      modes(j, md0, md1);
      const uint32_t ts = tmem + 128 * b + lane_off, tp = tmem + 256 + lane_off;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float sv[32], pv[32];
        tc::tmem_ld32(ts + 32 * ch, sv);
        tc::tmem_ld32(tp + 32 * ch, pv);
        tc::tmem_ld_wait();
        mask_keys(sv, ch < 2 ? md0 : md1, (ch & 1) * 32, rr);
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float p0 = tc::fast_exp2(sv[2 * x] * sl2 - lse2), p1 = tc::fast_exp2(sv[2 * x + 1] * sl2 - lse2);
          pk[x] = tc::pack_bf16x2(p0 * (pv[2 * x] - dl), p1 * (pv[2 * x + 1] - dl));
        }
        tc::tmem_st16u(ts + 16 * ch, pk);  // columns already read
      }
      tc::tmem_st_wait();
      tc::fence_before();
      tc::mbar_arrive(&bars[DQ_SR + b]);
    }
    // epilogue: dq += scale dQ
    if (ok && (ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[DQ_DONE], 0, err)))) {
      tc::fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        tc::tmem_ld32(tmem + 384 + lane_off + 32 * ch, o);
        tc::tmem_ld_wait();
        if (valid) {
          float4* dst = (float4*)(dq + row * D + 32 * ch);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            float4 a = dst[x];
            a.x += scale * o[4 * x];
            a.y += scale * o[4 * x + 1];
            a.z += scale * o[4 * x + 2];
            a.w += scale * o[4 * x + 3];
            dst[x] = a;
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dkv
template <int D>
struct DkvSm {
  static constexpr int kT = 128 * D * 2;
  static constexpr int offK = 0;
  static constexpr int offV = offK + kT;
  static constexpr int offQ = offV + kT;          // 2 stages of [Q | dO]
  static constexpr int offVec = offQ + 4 * kT;    // 2 stages of [lse (128) | delta (128)] fp32
  static constexpr int offBar = offVec + 2 * 1024;
  static constexpr int kNumBars = 14;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
};
enum { KV_F = 0, KV_QF = 1, KV_QE = 3, KV_SF = 5, KV_PF = 7, KV_SR = 9, KV_DONE = 11, KV_DR = 12 };

template <int D>
__global__ void __launch_bounds__(256, 1)
    softmax_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                              const uint8_t* __restrict__ sel, const int32_t* __restrict__ nprev,
                              const int32_t* __restrict__ sel_idx, int L, int N, int T, long long BH,
                              float scale, int retained, const float* __restrict__ lse,
                              const float* __restrict__ delta, float* __restrict__ dk, float* __restrict__ dv,
                              int* __restrict__ err) {
  using S = DkvSm<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The key tile: two chunk slots.  Local tiles (retained = 0) are the
  // chunk pairs (2p, 2p + 1) against their own query pair only: each
  // chunk's causal block and, when 2p chose softmax, 2p + 1's queries on its
  // keys; they write dk, dv.  Retained tiles (retained = 1) are pairs of the
  // head's softmax chunks (its compacted list) against every later query
  // chunk, and add into dk, dv.  Heaviest tiles first in both.
  const int jt = (int)(blockIdx.x / BH);
  const long long bh = blockIdx.x % BH;
  const long long row0 = bh * (long long)L;
  int kc0, kc1, r0, nq;
  bool has_k1, soft0, soft1;
  if (!retained) {
    kc0 = 2 * jt;
    has_k1 = kc0 + 1 < N;
    kc1 = has_k1 ? kc0 + 1 : kc0;
    soft0 = sel[bh * N + kc0] == 0;
    soft1 = has_k1 && sel[bh * N + kc1] == 0;
    r0 = jt;
    nq = 1;
  } else {
    const int nsoft = nprev[bh * N + N - 1] + (sel[bh * N + N - 1] == 0 ? 1 : 0);
    if (2 * jt >= nsoft) return;  // (uniform over the CTA, before any barrier)
    kc0 = sel_idx[bh * N + 2 * jt];
    has_k1 = 2 * jt + 1 < nsoft;
    kc1 = has_k1 ? sel_idx[bh * N + 2 * jt + 1] : kc0;
    soft0 = true;
    soft1 = has_k1;
    r0 = kc0 / 2 + 1;  // the first query pair after kc0's own (which the local tile covers)
    nq = T - r0;
    if (nq <= 0) return;
  }
  const float sl2 = scale * 1.4426950408889634f;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[KV_F], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[KV_QF + s], 1);
      tc::mbar_init(&bars[KV_QE + s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      tc::mbar_init(&bars[KV_SF + h], 1);
      tc::mbar_init(&bars[KV_PF + h], 1);
      tc::mbar_init(&bars[KV_SR + h], 128);
    }
    tc::mbar_init(&bars[KV_DONE], 1);
    tc::mbar_init(&bars[KV_DR], 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // S^T of query chunks h = 0, 1 (64 columns each) | dP^T likewise | dV | dK
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_v);
      tc::prefetch_tensormap(&tm_do);
      tc::mbar_arrive_expect_tx(&bars[KV_F], 2 * S::kT);
      for (int slot = 0; slot < 2; ++slot) {
        const int y = (int)(row0 + 64LL * (slot ? kc1 : kc0));
        for (int h = 0; h < D / 64; ++h) {
          tc::tma_load_2d(smem + S::offK + h * kHalf + slot * (kHalf / 2), &tm_k, 64 * h, y, &bars[KV_F]);
          tc::tma_load_2d(smem + S::offV + h * kHalf + slot * (kHalf / 2), &tm_v, 64 * h, y, &bars[KV_F]);
        }
      }
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nq && ok; ++i) {
        const int s = i & 1, r = r0 + i;
        const bool has_q1 = 2 * r + 1 < N;
        const uint32_t vb = has_q1 ? 512 : 256;  // the rows' lse and delta that exist
        if (!(ok = tc::mbar_wait(&bars[KV_QE + s], ((i >> 1) & 1) ^ 1, err))) break;
        uint8_t* st = smem + S::offQ + s * 2 * S::kT;
        float* vec = (float*)(smem + S::offVec + s * 1024);
        tc::mbar_arrive_expect_tx(&bars[KV_QF + s], 2 * S::kT + 2 * vb);
        for (int rc = 0; rc < 2; ++rc) {
          const int y = (int)(row0 + 128LL * r + 64 * rc);
          for (int h = 0; h < D / 64; ++h) {
            tc::tma_load_2d(st + h * kHalf + rc * (kHalf / 2), &tm_q, 64 * h, y, &bars[KV_QF + s]);
            tc::tma_load_2d(st + S::kT + h * kHalf + rc * (kHalf / 2), &tm_do, 64 * h, y, &bars[KV_QF + s]);
          }
        }
        tc::bulk_load_1d(vec, lse + row0 + 128LL * r, vb, &bars[KV_QF + s]);
        tc::bulk_load_1d(vec + 128, delta + row0 + 128LL * r, vb, &bars[KV_QF + s]);
        ++issued;
      }
      tc::mbar_wait(&bars[KV_F], 0, nullptr);
      for (int s = 0; s < 2; ++s) {
        const int n = issued > s ? (issued - 1 - s) / 2 + 1 : 0;
        if (n > 0) tc::mbar_wait(&bars[KV_QF + s], (n - 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    // One step per query chunk u (chunk 2r + h of query pair r = p + u / 2):
    // its S^T and dP^T (N = 64) go to TMEM half h, and are issued one chunk
    // ahead, so the tensor pipe works on chunk u + 1 while the elementwise
    // warps turn chunk u into P^T and dS^T; then dV += P^T dO and
    // dK += dS^T Q over the chunk's 64 queries.
    if (lane == 0) {
      constexpr uint32_t id_qk = tc::idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, D, false, true);
      const uint64_t kd = tc::smem_desc_sw128(tc::smem_u32(smem + S::offK), 16, 1024);
      const uint64_t vd = tc::smem_desc_sw128(tc::smem_u32(smem + S::offV), 16, 1024);
      const uint32_t qb = tc::smem_u32(smem + S::offQ);
      const uint32_t tdV = tmem + 256, tdK = tmem + 384;
      const int nu = 2 * nq;
      bool ok = tc::mbar_wait(&bars[KV_F], 0, err);
      auto issue_sp = [&](int u) -> bool {
        const int i = u >> 1, h = u & 1, s = i & 1;
        if (h == 0 && !tc::mbar_wait(&bars[KV_QF + s], (i >> 1) & 1, err)) return false;
        tc::fence_after();
        const uint32_t cb = qb + s * 2 * S::kT + h * (kHalf / 2);  // query chunk h of the stage
        const uint64_t qk = tc::smem_desc_sw128(cb, 16, 1024), ok_ = tc::smem_desc_sw128(cb + S::kT, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + 64 * h, tc::desc_add(kd, off), tc::desc_add(qk, off), id_qk, kk > 0);
        }
        tc::mma_commit(&bars[KV_SF + h]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + 128 + 64 * h, tc::desc_add(vd, off), tc::desc_add(ok_, off), id_qk, kk > 0);
        }
        tc::mma_commit(&bars[KV_PF + h]);
        return true;
      };
      if (ok) ok = issue_sp(0);
      for (int u = 0; u < nu && ok; ++u) {
        const int i = u >> 1, h = u & 1, s = i & 1;
        // the next chunk's buffers were last read by chunk u - 1's products,
        // issued before (in order) once its P^T / dS^T were in place
        if (u + 1 < nu && !(ok = issue_sp(u + 1))) break;
        if (!(ok = tc::mbar_wait(&bars[KV_SR + h], (u >> 1) & 1, err))) break;
        tc::fence_after();
        const uint32_t sb = qb + s * 2 * S::kT;
        const uint64_t qn = tc::smem_desc_sw128(sb, kHalf, 1024), on = tc::smem_desc_sw128(sb + S::kT, kHalf, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16_ts(tdV, tmem + 64 * h + kk * 8, tc::desc_add(on, h * (kHalf / 2) + kk * 2048), id_pv,
                          (u > 0) || (kk > 0));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16_ts(tdK, tmem + 128 + 64 * h + kk * 8, tc::desc_add(qn, h * (kHalf / 2) + kk * 2048), id_pv,
                          (u > 0) || (kk > 0));
        if (h == 1) tc::mma_commit(&bars[KV_QE + s]);
      }
      if (ok) tc::mma_commit(&bars[KV_DONE]);
      tc::mma_commit(&bars[KV_DR]);
      tc::mbar_wait(&bars[KV_DR], 0, nullptr);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------- elementwise
    const int kr = threadIdx.x - 128;
    const int ks = kr >> 6, ki = kr & 63;
    const int kc = ks ? kc1 : kc0;
    const bool valid = ks == 0 || has_k1;
    const bool soft_k = ks == 0 ? soft0 : soft1;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    bool ok = true;
    for (int u = 0; u < 2 * nq && ok; ++u) {
      const int i = u >> 1, h = u & 1, s = i & 1;
      const int qc = 2 * (r0 + i) + h;  // the query chunk of this step
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[KV_SF + h], (u >> 1) & 1, err)))) break;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[KV_PF + h], (u >> 1) & 1, err)))) break;
      tc::fence_after();
      const float* ls = (const float*)(smem + S::offVec + s * 1024) + 64 * h;
      const float* dls = ls + 128;
      int mode = kNone;  // whether this key row sees the chunk's queries (its own chunk: local tiles only)
      if (valid && qc < N) {
        if (!retained) mode = qc == kc ? kCausal : ((soft_k && qc > kc) ? kFull : kNone);
        else mode = (qc >> 1) > (kc >> 1) ? kFull : kNone;  // query pairs after the key chunk's own
      }
      const uint32_t ts = tmem + 64 * h + lane_off, tp = tmem + 128 + 64 * h + lane_off;
      if (mode == kNone) {  // (warp-uniform: a warp's rows share a key chunk) nothing to read
        uint32_t z[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) z[x] = 0u;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          tc::tmem_st16u(ts + 16 * ch, z);
          tc::tmem_st16u(tp + 16 * ch, z);
        }
      } else {
        const float4* ls4 = (const float4*)ls;
        const float4* dl4 = (const float4*)dls;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          float sv[32], pv[32];
          tc::tmem_ld32(ts + 32 * ch, sv);
          tc::tmem_ld32(tp + 32 * ch, pv);
          tc::tmem_ld_wait();
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int y = 0; y < 8; ++y) {
            const float4 l = ls4[8 * ch + y], dd = dl4[8 * ch + y];
            const float lv[4] = {l.x, l.y, l.z, l.w}, dv4[4] = {dd.x, dd.y, dd.z, dd.w};
            float e[4], g4[4];
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const int c = 32 * ch + 4 * y + w4;  // query index within the chunk
              const bool vis = mode == kFull || c >= ki;
              // (queries that do not exist read stale lse / delta: selected away)
              e[w4] = vis ? tc::fast_exp2(sv[4 * y + w4] * sl2 - lv[w4]) : 0.f;
              g4[w4] = vis ? e[w4] * (pv[4 * y + w4] - dv4[w4]) : 0.f;
            }
            pp[2 * y] = tc::pack_bf16x2(e[0], e[1]);
            pp[2 * y + 1] = tc::pack_bf16x2(e[2], e[3]);
            pd[2 * y] = tc::pack_bf16x2(g4[0], g4[1]);
            pd[2 * y + 1] = tc::pack_bf16x2(g4[2], g4[3]);
          }
          tc::tmem_st16u(ts + 16 * ch, pp);  // columns already read
          tc::tmem_st16u(tp + 16 * ch, pd);
        }
      }
      tc::tmem_st_wait();
      tc::fence_before();
      tc::mbar_arrive(&bars[KV_SR + h]);
    }
    // epilogue: dv = dV, dk = scale dK (every key row belongs to one tile)
    if (ok && (ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[KV_DONE], 0, err)))) {
      tc::fence_after();
      const size_t row = (size_t)(row0 + 64LL * kc + ki);
#pragma unroll 1
      for (int w2 = 0; w2 < 2; ++w2) {
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float o[32];
          tc::tmem_ld32(tmem + 256 + 128 * w2 + lane_off + 32 * ch, o);
          tc::tmem_ld_wait();
          if (valid) {
            const float f = w2 ? scale : 1.f;
            float4* dst = (float4*)((w2 ? dk : dv) + row * D + 32 * ch);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              float4 a = make_float4(f * o[4 * x], f * o[4 * x + 1], f * o[4 * x + 2], f * o[4 * x + 3]);
              if (retained) {  // add to the local tile's
                const float4 b = dst[x];
                a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
              }
              dst[x] = a;
            }
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t run(const Problem& p, const void* q, const void* k, const void* v, const void* dos,
                const float* delta, const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel, float* lse,
                const float* lse_in, float* dq, float* dk, float* dv, int* err, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  const long long rows = p.BH * p.L;
  if (!make_tile_map(&mq, q, rows, D) || !make_tile_map(&mk, k, rows, D) || !make_tile_map(&mv, v, rows, D) ||
      !make_tile_map(&mo, dos, rows, D))
    return cudaErrorInvalidValue;
  static const cudaError_t attr = [] {
    cudaError_t e = cudaFuncSetAttribute(softmax_bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqSm<D>::kBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(softmax_bwd_dkv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DkvSm<D>::kBytes);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  const int T = (p.N + 1) / 2;
  const unsigned grid = (unsigned)(p.BH * T);
  softmax_bwd_dq_tc_kernel<D><<<grid, 256, DqSm<D>::kBytes, st>>>(mq, mk, mv, mo, nprev, sel_idx, sel, p.L, p.N, T,
                                                                  p.BH, p.scale, delta, lse, lse_in, dq, err);
  for (int retained = 0; retained < 2; ++retained)
    softmax_bwd_dkv_tc_kernel<D><<<grid, 256, DkvSm<D>::kBytes, st>>>(mq, mk, mv, mo, sel, nprev, sel_idx, p.L, p.N,
                                                                      T, p.BH, p.scale, retained,
                                                                      lse_in ? lse_in : lse, delta, dk, dv, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_bwd_tc(const Problem& p, const void* q, const void* k, const void* v, const void* dos,
                                  const float* delta, const int32_t* nprev, const int32_t* sel_idx,
                                  const uint8_t* sel, float* lse, const float* lse_in, float* dq, float* dk,
                                  float* dv, int* err, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run<64>(p, q, k, v, dos, delta, nprev, sel_idx, sel, lse, lse_in, dq, dk, dv, err, st)
                   : run<128>(p, q, k, v, dos, delta, nprev, sel_idx, sel, lse, lse_in, dq, dk, dv, err, st);
}

}  // namespace nats
