// gdn_scan_tc.cu - Gated DeltaNet phase 2 on the 5th-generation tensor cores:
// the chunk-by-chunk state scan with pseudo-update and rollback (bf16 path).
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the linear state is pseudo-updated for every
// chunk; for a chunk that chose softmax it is rolled back to the chunk start.
// With the phase-1 factors W, U, P of a chunk (S0 = state at its start,
// G = in-chunk cumulative log-decay, gamma = e^G):
//   Delta = U - W S0^T
//   O     = gamma * (scale Q S0^T) + P Delta
//   S_C   = gamma_C S0 + Delta^T diag(gamma_C / gamma) K     (linear chunks only)
//
// One CTA per (b, h) walks the N chunks in order; the fp32 state S (dv x dk)
// stays in TMEM for the whole sequence and a bf16 copy in shared memory feeds
// the next chunk's MMA.  Per chunk:
//   MMA1  X = [W; Q] S0^T          (M=128 = 64 W rows + 64 Q rows, N=dv, K=dk)
//   thr   Delta, Delta~ = diag(gamma_C/gamma) Delta -> smem (bf16); S *= gamma_C
//   MMA2  Y = [. ; P] Delta        (rows 64..127 = P Delta, aligned with Q S0^T)
//   MMA3  S += Delta~^T K          (linear chunks only; M = dv, N = dk, K = 64)
//   thr   O = gamma scale (Q S0^T) + P Delta -> o_l;  S -> bf16 copy
// Roles: warps 0-3 elementwise (thread r <-> TMEM lane r), warp 4 TMA
// producer (W, Q, K, U, P of the next chunk, double-buffered), warp 5 TMEM
// owner and MMA issuer.  Every wait is bounded (tc::kWaitLimitNs).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {

bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D);

namespace {

template <int D>
struct ScanSmem {
  static constexpr int kWQ = 128 * D * 2;  // [W; Q] tile, D/64 halves of 128 lines
  static constexpr int kK = 64 * D * 2;    // K chunk, D/64 halves of 64 lines
  static constexpr int kU = 64 * D * 2;    // U chunk
  static constexpr int kP = 128 * 128;     // 128 lines x 64 cols (P in lines 64..127)
  static constexpr int kStage = kWQ + kK + kU + kP;
  static constexpr int offStage = 0;
  static constexpr int offS0 = 2 * kStage;         // bf16 S0, K-major (lines dv, cols dk)
  static constexpr int kS0 = D * D * 2;
  static constexpr int offDelta = offS0 + kS0;     // Delta  [t][dv], MN-major B operand
  static constexpr int offDeltaT = offDelta + 64 * D * 2;  // Delta~ [t][dv], MN-major A (2 halves)
  static constexpr int offBar = offDeltaT + 64 * 128 * 2;
  static constexpr int kNumBars = 10;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
};

enum { SB_FULL = 0, SB_EMPTY = 2, SB_S0 = 4, SB_X = 5, SB_DELTA = 6, SB_Y = 7, SB_SDONE = 8, SB_DONE = 9 };

// byte offset of element (line, col) in a 128-byte-swizzled tile whose
// 64-column halves are `half_bytes` apart
__device__ __forceinline__ uint32_t sw_off(int line, int col, int half_bytes) {
  return (uint32_t)((col >> 6) * half_bytes + line * 128 + ((((col & 63) >> 3) ^ (line & 7)) << 4) + (col & 7) * 2);
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    gdn_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_u,
                       const __grid_constant__ CUtensorMap tm_p, const uint8_t* __restrict__ sel,
                       const float* __restrict__ G, int L, int N, float scale, float* __restrict__ o_l,
                       float* __restrict__ state_out, int* __restrict__ err) {
  using S = ScanSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  uint8_t* S0s = smem + S::offS0;
  uint8_t* Ds = smem + S::offDelta;
  uint8_t* Dts = smem + S::offDeltaT;

  const long long bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[SB_FULL + s], 1);
      tc::mbar_init(&bars[SB_EMPTY + s], 1);
    }
    tc::mbar_init(&bars[SB_S0], 128);
    tc::mbar_init(&bars[SB_X], 1);
    tc::mbar_init(&bars[SB_DELTA], 128);
    tc::mbar_init(&bars[SB_Y], 1);
    tc::mbar_init(&bars[SB_SDONE], 1);
    tc::mbar_init(&bars[SB_DONE], 1);
    tc::fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tX = tmem, tY = tmem + 128, tS = tmem + 256;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_w);
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_u);
      tc::prefetch_tensormap(&tm_p);
      int issued[2] = {0, 0};
      bool ok = true;
      for (int c = 0; c < N; ++c) {
        const int s = c & 1;
        if (!(ok = tc::mbar_wait(&bars[SB_EMPTY + s], ((c >> 1) & 1) ^ 1, err))) break;
        uint8_t* st = smem + S::offStage + s * S::kStage;
        uint8_t* WQ = st;
        uint8_t* Kb = WQ + S::kWQ;
        uint8_t* Ub = Kb + S::kK;
        uint8_t* Pb = Ub + S::kU;
        const int yc = (int)((bh * N + c) * 64);   // row of this chunk in W / U / P
        const int yt = (int)(bh * L + 64LL * c);   // row of this chunk in Q / K
        tc::mbar_arrive_expect_tx(&bars[SB_FULL + s], 4 * 64 * D * 2 + 64 * 64 * 2);
        for (int h = 0; h < D / 64; ++h) {
          tc::tma_load_2d(WQ + h * 16384, &tm_w, 64 * h, yc, &bars[SB_FULL + s]);
          tc::tma_load_2d(WQ + h * 16384 + 8192, &tm_q, 64 * h, yt, &bars[SB_FULL + s]);
          tc::tma_load_2d(Kb + h * 8192, &tm_k, 64 * h, yt, &bars[SB_FULL + s]);
          tc::tma_load_2d(Ub + h * 8192, &tm_u, 64 * h, yc, &bars[SB_FULL + s]);
        }
        tc::tma_load_2d(Pb + 8192, &tm_p, 0, yc, &bars[SB_FULL + s]);
        issued[s]++;
      }
      if (ok) {
        for (int s = 0; s < 2; ++s)
          if (issued[s] > 0) tc::mbar_wait(&bars[SB_EMPTY + s], (issued[s] - 1) & 1, err);
      } else {
        for (int s = 0; s < 2; ++s)
          if (issued[s] > 0) tc::mbar_wait(&bars[SB_FULL + s], (issued[s] - 1) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id1 = tc::idesc_bf16_f32(128, D, false, false);
      constexpr uint32_t id2 = tc::idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t id3 = tc::idesc_bf16_f32(128, D, true, true);
      const uint32_t s0 = tc::smem_u32(S0s), dsa = tc::smem_u32(Ds), dta = tc::smem_u32(Dts);
      bool ok = true;
      for (int c = 0; c < N && ok; ++c) {
        const int s = c & 1;
        const uint32_t st = tc::smem_u32(smem + S::offStage + s * S::kStage);
        const uint32_t wq = st, kb = st + S::kWQ, pb = st + S::kWQ + S::kK + S::kU;
        if (!(ok = tc::mbar_wait(&bars[SB_FULL + s], (c >> 1) & 1, err))) break;
        if (!(ok = tc::mbar_wait(&bars[SB_S0], c & 1, err))) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * (D * 128) + (kk & 3) * 32;
          tc::mma_bf16(tX, tc::smem_desc_sw128(wq + off, 16, 1024), tc::smem_desc_sw128(s0 + offb, 16, 1024), id1,
                       kk > 0);
        }
        tc::mma_commit(&bars[SB_X]);
        if (!(ok = tc::mbar_wait(&bars[SB_DELTA], c & 1, err))) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tY, tc::smem_desc_sw128(pb + kk * 32, 16, 1024),
                       tc::smem_desc_sw128(dsa + kk * 2048, 8192, 1024), id2, kk > 0);
        tc::mma_commit(&bars[SB_Y]);
        if (sel[bh * N + c] != 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(tS, tc::smem_desc_sw128(dta + kk * 2048, 8192, 1024),
                         tc::smem_desc_sw128(kb + kk * 2048, 8192, 1024), id3, 1);
        }
        tc::mma_commit(&bars[SB_SDONE]);
        tc::mma_commit(&bars[SB_EMPTY + s]);
      }
      tc::mma_commit(&bars[SB_DONE]);
      tc::mbar_wait(&bars[SB_DONE], 0, err);
    }
  } else {
    // ------------------------------------------------- elementwise (warps 0-3)
    const int r = threadIdx.x;  // TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    // S = 0 in TMEM and in the bf16 copy
    {
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) tc::tmem_st32(tS + lane_off + ch * 32, z);
      tc::tmem_st_wait();
      for (int e = r; e < D * D / 8; e += 128) ((uint4*)S0s)[e] = make_uint4(0, 0, 0, 0);
      tc::fence_proxy_async_smem();
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_S0]);
    }
    bool ok = true;
    for (int c = 0; c < N; ++c) {
      const int s = c & 1;
      const uint8_t* Ub = smem + S::offStage + s * S::kStage + S::kWQ + S::kK;
      const bool lin = sel[bh * N + c] != 0;
      const float* Gc = G + bh * (long long)L + 64LL * c;
      const float GC = Gc[63];
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_X], c & 1, err)))) break;
      tc::fence_after();
      if (r < 64) {
        // Delta[t] = U[t] - (W S0^T)[t];  Delta~[t] = Delta[t] * e^{G_C - G_t}
        const int t = r;
        const float dec = __expf(GC - Gc[t]);
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float x[32];
          tc::tmem_ld32(tX + lane_off + ch * 32, x);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int col = ch * 32 + g8 * 8;
            const uint32_t off = sw_off(t, col, 8192);
            const uint4 uv = *(const uint4*)(Ub + off);
            const __nv_bfloat162* u2 = (const __nv_bfloat162*)&uv;
            float d[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 uf = __bfloat1622float2(u2[i]);
              d[2 * i] = uf.x - x[g8 * 8 + 2 * i];
              d[2 * i + 1] = uf.y - x[g8 * 8 + 2 * i + 1];
            }
            uint4 pk, pt;
            pk.x = tc::pack_bf16x2(d[0], d[1]);
            pk.y = tc::pack_bf16x2(d[2], d[3]);
            pk.z = tc::pack_bf16x2(d[4], d[5]);
            pk.w = tc::pack_bf16x2(d[6], d[7]);
            pt.x = tc::pack_bf16x2(d[0] * dec, d[1] * dec);
            pt.y = tc::pack_bf16x2(d[2] * dec, d[3] * dec);
            pt.z = tc::pack_bf16x2(d[4] * dec, d[5] * dec);
            pt.w = tc::pack_bf16x2(d[6] * dec, d[7] * dec);
            *(uint4*)(Ds + off) = pk;
            *(uint4*)(Dts + off) = pt;
          }
        }
      }
      if (lin) {
        // S *= gamma_C before the rank-64 update is accumulated onto it
        const float gC = __expf(GC);
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float v[32];
          tc::tmem_ld32(tS + lane_off + ch * 32, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gC;
          tc::tmem_st32(tS + lane_off + ch * 32, v);
        }
        tc::tmem_st_wait();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_DELTA]);
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_Y], c & 1, err)))) break;
      tc::fence_after();
      if (r >= 64) {
        // O[t] = e^{G_t} scale (Q S0^T)[t] + (P Delta)[t]
        const int t = r - 64;
        const float gq = __expf(Gc[t]) * scale;
        float* dst = o_l + (bh * (long long)L + 64LL * c + t) * D;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float x[32], y[32];
          tc::tmem_ld32(tX + lane_off + ch * 32, x);
          tc::tmem_ld32(tY + lane_off + ch * 32, y);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            ((float4*)(dst + ch * 32))[i] = make_float4(fmaf(gq, x[4 * i], y[4 * i]), fmaf(gq, x[4 * i + 1], y[4 * i + 1]),
                                                        fmaf(gq, x[4 * i + 2], y[4 * i + 2]),
                                                        fmaf(gq, x[4 * i + 3], y[4 * i + 3]));
        }
      }
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[SB_SDONE], c & 1, err)))) break;
      tc::fence_after();
      if (lin && r < D) {
        // bf16 copy of the new state for the next chunk's MMA1 (lines dv, cols dk)
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float v[32];
          tc::tmem_ld32(tS + lane_off + ch * 32, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            uint4 pk;
            pk.x = tc::pack_bf16x2(v[g8 * 8 + 0], v[g8 * 8 + 1]);
            pk.y = tc::pack_bf16x2(v[g8 * 8 + 2], v[g8 * 8 + 3]);
            pk.z = tc::pack_bf16x2(v[g8 * 8 + 4], v[g8 * 8 + 5]);
            pk.w = tc::pack_bf16x2(v[g8 * 8 + 6], v[g8 * 8 + 7]);
            *(uint4*)(S0s + sw_off(r, ch * 32 + g8 * 8, D * 128)) = pk;
          }
        }
      } else if (lin) {
        float v[32];  // lanes >= D hold no state, but the load is warp-collective
        tc::tmem_ld32(tS + lane_off, v);
        tc::tmem_ld_wait();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before();
      tc::mbar_arrive(&bars[SB_S0]);
    }
    if (ok && state_out) {
      tc::fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float v[32];
        tc::tmem_ld32(tS + lane_off + ch * 32, v);
        tc::tmem_ld_wait();
        if (r < D) {
          float* dst = state_out + (bh * D + r) * (long long)D + ch * 32;
#pragma unroll
          for (int i = 0; i < 8; ++i) ((float4*)dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
static cudaError_t launch_scan_tc_t(const Problem& p, const void* q, const void* k, const uint8_t* sel,
                                    const float* G, const void* W16, const void* U16, const void* P16,
                                    float* o_l, float* state_out, int* err, cudaStream_t st) {
  CUtensorMap mw, mq, mk, mu, mp;
  const long long rows = p.BH * p.L;  // = BH * N * 64
  if (!make_tile_map(&mw, W16, rows, D) || !make_tile_map(&mq, q, rows, D) || !make_tile_map(&mk, k, rows, D) ||
      !make_tile_map(&mu, U16, rows, D) || !make_tile_map(&mp, P16, rows, 64))
    return cudaErrorInvalidValue;
  auto kern = gdn_scan_tc_kernel<D>;
  const int smem = ScanSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)p.BH, 192, smem, st>>>(mw, mq, mk, mu, mp, sel, G, p.L, p.N, p.scale, o_l, state_out, err);
  return cudaGetLastError();
}

cudaError_t launch_gdn_scan_tc(const Problem& p, const void* q, const void* k, const uint8_t* sel, const float* G,
                               const void* W16, const void* U16, const void* P16, float* o_l, float* state_out,
                               int* err, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? launch_scan_tc_t<64>(p, q, k, sel, G, W16, U16, P16, o_l, state_out, err, st)
                   : launch_scan_tc_t<128>(p, q, k, sel, G, W16, U16, P16, o_l, state_out, err, st);
}

}  // namespace nats
