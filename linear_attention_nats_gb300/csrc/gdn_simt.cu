// gdn_simt.cu - chunkwise Gated DeltaNet branch with pseudo-update and
// rollback, plain fp32 FMA (the fp32-input path).
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the linear state is pseudo-updated for every
// chunk and rolled back to the chunk start when the chunk chose softmax.
// Gated DeltaNet: S_t = a_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = S_t (scale q_t), a_t = exp(g_t).
//
// Chunkwise form (exact rewrite of the recurrence; S0 = state at the chunk
// start, G = in-chunk cumulative sum of g, gamma = e^G):
//   A     = strict_lower(beta_t e^{G_t - G_i} k_t . k_i),   T = (I + A)^{-1}
//   U     = T diag(beta) V,        W = T diag(beta gamma) K
//   Delta = U - W S0^T
//   O     = gamma * (scale Q S0^T) + P Delta,   P = lower_incl(e^{G_t - G_i} scale q_t . k_i)
//   S_C   = gamma_C S0 + Delta^T diag(gamma_C / gamma) K      (committed only if linear)
// Phase 1 (prep) is parallel over all chunks; phase 2 (scan) walks the
// chunks of one (b, h) in order, split over 32-row slices of the value dim.
#include "common.cuh"
#include "kernels.h"

namespace nats {

// Phase 1: one CTA per (b, h, chunk).
template <class T, int D>
__global__ void __launch_bounds__(256) gdn_prep_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ g, const float* __restrict__ beta, int L, int N, float scale,
    float* __restrict__ Gout, float* __restrict__ Wout, float* __restrict__ Uout,
    float* __restrict__ Pout) {
  constexpr int C = kChunk, KP = D + 1, CP = C + 1;
  extern __shared__ float smem[];
  float* Ks = smem;           // [C][D+1]
  float* Qs = Ks + C * KP;    // [C][D+1]
  float* Vs = Qs + C * KP;    // [C][D]
  float* As = Vs + C * D;     // [C][C+1]
  float* Ts = As + C * CP;    // [C][C+1]
  float* Gs = Ts + C * CP;    // [C]
  float* Bs = Gs + C;         // [C] beta
  float* Bg = Bs + C;         // [C] beta e^{G}
  const long long blk = blockIdx.x;
  const int c = (int)(blk % N);
  const long long bh = blk / N;
  const int tid = threadIdx.x;
  const size_t tok0 = (size_t)bh * L + (size_t)c * C;
  for (int e = tid; e < C * D; e += 256) {
    const int t = e / D, f = e % D;
    Ks[t * KP + f] = to_f32(k[tok0 * D + e]);
    Qs[t * KP + f] = to_f32(q[tok0 * D + e]);
    Vs[e] = to_f32(v[tok0 * D + e]);
  }
  if (tid < 32) {  // inclusive cumulative sum of g over the chunk
    const float g0 = g[tok0 + 2 * tid], g1 = g[tok0 + 2 * tid + 1];
    float x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
    }
    const float excl = x - (g0 + g1);
    Gs[2 * tid] = excl + g0;
    Gs[2 * tid + 1] = excl + g0 + g1;
    Gout[tok0 + 2 * tid] = excl + g0;
    Gout[tok0 + 2 * tid + 1] = excl + g0 + g1;
  } else if (tid < 96) {
    Bs[tid - 32] = beta[tok0 + tid - 32];
  }
  __syncthreads();
  if (tid < C) Bg[tid] = Bs[tid] * expf(Gs[tid]);
  float* P = Pout + (size_t)blk * C * C;
  for (int e = tid; e < C * C; e += 256) {
    const int t = e / C, i = e % C;
    float a = 0.f, pv = 0.f;
    if (i <= t) {
      const float* kt = Ks + t * KP;
      const float* ki = Ks + i * KP;
      const float* qt = Qs + t * KP;
      float kk = 0.f, qk = 0.f;
#pragma unroll 8
      for (int f = 0; f < D; ++f) {
        kk = fmaf(kt[f], ki[f], kk);
        qk = fmaf(qt[f], ki[f], qk);
      }
      const float dec = expf(Gs[t] - Gs[i]);
      if (i < t) a = Bs[t] * dec * kk;
      pv = scale * dec * qk;
    }
    As[t * CP + i] = a;
    P[e] = pv;
  }
  __syncthreads();
  // T = (I + A)^{-1}, unit lower triangular, by forward substitution:
  // T[t][j] = -sum_{j <= i < t} A[t][i] T[i][j].
  for (int t = 0; t < C; ++t) {
    if (tid < C) {
      const int j = tid;
      float x = (j == t) ? 1.f : 0.f;
      if (j < t) {
        for (int i = j; i < t; ++i) x = fmaf(-As[t * CP + i], Ts[i * CP + j], x);
      }
      Ts[t * CP + j] = x;
    }
    __syncthreads();
  }
  float* W = Wout + (size_t)blk * C * D;
  float* U = Uout + (size_t)blk * C * D;
  for (int e = tid; e < C * D; e += 256) {
    const int t = e / D, f = e % D;
    float w = 0.f, u = 0.f;
    for (int i = 0; i <= t; ++i) {
      const float ti = Ts[t * CP + i];
      u = fmaf(ti * Bs[i], Vs[i * D + f], u);
      w = fmaf(ti * Bg[i], Ks[i * KP + f], w);
    }
    W[e] = w;
    U[e] = u;
  }
}

// Phase 2: one CTA per (32-row value slice, b*h); the state slice S[32][D]
// stays in shared memory for the whole sequence.
template <class T, int D>
__global__ void __launch_bounds__(256) gdn_scan_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const uint8_t* __restrict__ sel,
    const float* __restrict__ Gin, const float* __restrict__ Win, const float* __restrict__ Uin,
    const float* __restrict__ Pin, int L, int N, float scale, float* __restrict__ o_l,
    float* __restrict__ state_out) {
  constexpr int C = kChunk, KP = D + 1, CP = C + 1, R = 32, RP = R + 1;
  extern __shared__ float smem[];
  float* S = smem;            // [R][D+1]
  float* Ws = S + R * KP;     // [C][D+1]
  float* Qs = Ws + C * KP;    // [C][D+1]
  float* Ks = Qs + C * KP;    // [C][D+1]
  float* Us = Ks + C * KP;    // [C][R+1]
  float* Ps = Us + C * RP;    // [C][C+1]
  float* Ds = Ps + C * CP;    // [C][R+1]  Delta
  float* Eg = Ds + C * RP;    // [C] e^{G_t}
  float* Er = Eg + C;         // [C] e^{G_C - G_t}
  const int slice = blockIdx.x;
  const long long bh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < R * KP; e += 256) S[e] = 0.f;
  for (int c = 0; c < N; ++c) {
    const long long blk = bh * N + c;
    const size_t tok0 = (size_t)bh * L + (size_t)c * C;
    __syncthreads();
    for (int e = tid; e < C * D; e += 256) {
      const int t = e / D, f = e % D;
      Ws[t * KP + f] = Win[(size_t)blk * C * D + e];
      Qs[t * KP + f] = to_f32(q[tok0 * D + e]);
      Ks[t * KP + f] = to_f32(k[tok0 * D + e]);
    }
    for (int e = tid; e < C * R; e += 256) {
      const int t = e / R, r = e % R;
      Us[t * RP + r] = Uin[(size_t)blk * C * D + t * D + slice * R + r];
    }
    for (int e = tid; e < C * C; e += 256) Ps[(e / C) * CP + e % C] = Pin[(size_t)blk * C * C + e];
    if (tid < C) {
      const float Gt = Gin[tok0 + tid];
      const float GC = Gin[tok0 + C - 1];
      Eg[tid] = expf(Gt);
      Er[tid] = expf(GC - Gt);
    }
    __syncthreads();
    // Delta[t][r] = U[t][r] - sum_i W[t][i] S[r][i]      (lane = r)
    for (int t = warp; t < C; t += 8) {
      float x = 0.f;
      const float* wt = Ws + t * KP;
      const float* sr = S + lane * KP;
#pragma unroll 8
      for (int i = 0; i < D; ++i) x = fmaf(wt[i], sr[i], x);
      Ds[t * RP + lane] = Us[t * RP + lane] - x;
    }
    __syncthreads();
    // O[t][r] = e^{G_t} scale (Q S^T)[t][r] + sum_{j<=t} P[t][j] Delta[j][r]
    for (int t = warp; t < C; t += 8) {
      float x = 0.f, y = 0.f;
      const float* qt = Qs + t * KP;
      const float* sr = S + lane * KP;
#pragma unroll 8
      for (int i = 0; i < D; ++i) x = fmaf(qt[i], sr[i], x);
      for (int j = 0; j <= t; ++j) y = fmaf(Ps[t * CP + j], Ds[j * RP + lane], y);
      o_l[(tok0 + t) * D + slice * R + lane] = Eg[t] * scale * x + y;
    }
    if (sel[blk] != 0) {  // linear chunk: commit the pseudo-update
      __syncthreads();
      const float eC = Eg[C - 1];
      for (int e = tid; e < R * D; e += 256) {
        const int r = e / D, i = e % D;
        float x = 0.f;
        for (int t = 0; t < C; ++t) x = fmaf(Ds[t * RP + r] * Er[t], Ks[t * KP + i], x);
        S[r * KP + i] = eC * S[r * KP + i] + x;
      }
    }  // else: rollback, S keeps its chunk-start value
  }
  if (state_out) {
    __syncthreads();
    for (int e = tid; e < R * D; e += 256) {
      const int r = e / D, i = e % D;
      state_out[((size_t)bh * D + slice * R + r) * D + i] = S[r * KP + i];
    }
  }
}

template <class T, int D>
static cudaError_t launch_prep_t(const Problem& p, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const Workspace& ws,
                                 cudaStream_t st) {
  constexpr int C = kChunk;
  const size_t sm = sizeof(float) * (size_t)(2 * C * (D + 1) + C * D + 2 * C * (C + 1) + 3 * C);
  auto kern = gdn_prep_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(p.BH * p.N), 256, sm, st>>>((const T*)q, (const T*)k, (const T*)v, g, beta, p.L,
                                                p.N, p.scale, ws.G, ws.W, ws.U, ws.P);
  return cudaGetLastError();
}

template <class T, int D>
static cudaError_t launch_scan_t(const Problem& p, const void* q, const void* k, const uint8_t* sel,
                                 const Workspace& ws, float* o_l, float* state_out,
                                 cudaStream_t st) {
  constexpr int C = kChunk;
  const size_t sm =
      sizeof(float) * (size_t)(32 * (D + 1) + 3 * C * (D + 1) + 2 * C * 33 + C * (C + 1) + 2 * C);
  auto kern = gdn_scan_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid(D / 32, (unsigned)p.BH);
  kern<<<grid, 256, sm, st>>>((const T*)q, (const T*)k, sel, ws.G, ws.W, ws.U, ws.P, p.L, p.N,
                              p.scale, o_l, state_out);
  return cudaGetLastError();
}

cudaError_t launch_gdn_prep_simt(const Problem& p, int dtype, const void* q, const void* k,
                                 const void* v, const float* g, const float* beta,
                                 const Workspace& ws, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  if (dtype == 0)
    return p.d == 64 ? launch_prep_t<__nv_bfloat16, 64>(p, q, k, v, g, beta, ws, st)
                     : launch_prep_t<__nv_bfloat16, 128>(p, q, k, v, g, beta, ws, st);
  return p.d == 64 ? launch_prep_t<float, 64>(p, q, k, v, g, beta, ws, st)
                   : launch_prep_t<float, 128>(p, q, k, v, g, beta, ws, st);
}

cudaError_t launch_gdn_scan_simt(const Problem& p, int dtype, const void* q, const void* k,
                                 const uint8_t* sel, const Workspace& ws, float* o_l,
                                 float* state_out, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  if (dtype == 0)
    return p.d == 64 ? launch_scan_t<__nv_bfloat16, 64>(p, q, k, sel, ws, o_l, state_out, st)
                     : launch_scan_t<__nv_bfloat16, 128>(p, q, k, sel, ws, o_l, state_out, st);
  return p.d == 64 ? launch_scan_t<float, 64>(p, q, k, sel, ws, o_l, state_out, st)
                   : launch_scan_t<float, 128>(p, q, k, sel, ws, o_l, state_out, st);
}

}  // namespace nats
