// score_bwd.cu - the score layer's gradient under a straight-through
// surrogate ("Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 5: the score layer learns end to end; the pages
// name no estimator, so this is an opt-in reading, BWD-2).
//
// Per chunk c of head h: p_c = the chunk mean of [q_t ; k_t] (unscaled q),
// s_c = W_s[h] p_c + b_s[h], pi_c = softmax(s_c) over the two operations and
// sel_c the forward's argmax.  Every output row of the chunk is read as
// scaled by pi_c[sel_c] / (the same probability held constant), which leaves
// the value alone and gives
//   ds_c = G_c (e_sel - pi_c),   G_c = sum_{t in c} <dout_t, out_t>,
//   dW_s[h] += ds_c p_c^T,   db_s[h] += ds_c,
//   dq_t, dk_t += (W_s[h]^T ds_c) / 64   for every token t of the chunk
// (the first d columns of W_s act on q, the last d on k).
//
// One CTA of 256 threads walks kGroup chunks of one (b, h); thread f owns
// feature f of [q ; k] (pooling, the score dot products, the dq / dk rows),
// and the W_s / b_s sums of the group go out with one atomic each.
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int kGroup = 8;  // chunks per CTA

template <typename T, int D>
__global__ void __launch_bounds__(256) score_bwd_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                        const float* __restrict__ w_s,
                                                        const float* __restrict__ b_s,
                                                        const uint8_t* __restrict__ sel, const T* __restrict__ out,
                                                        const T* __restrict__ dout, int H, int N, int L,
                                                        float* __restrict__ dq, float* __restrict__ dk,
                                                        float* __restrict__ dw_s, float* __restrict__ db_s) {
  constexpr int F = 2 * D;           // features of the pooled vector
  constexpr int RS = 256 / D;        // row groups of the <dout, out> sum
  const int groups = (N + kGroup - 1) / kGroup;
  const long long bh = blockIdx.x / groups;
  const int c0 = (int)(blockIdx.x % groups) * kGroup;
  const int h = (int)(bh % H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool feat = tid < F;
  const float* W = w_s + (size_t)h * 2 * F;
  const float w0 = feat ? W[tid] : 0.f, w1 = feat ? W[F + tid] : 0.f;
  const float bs0 = b_s ? b_s[2 * h] : 0.f, bs1 = b_s ? b_s[2 * h + 1] : 0.f;
  __shared__ float red[3][8];
  __shared__ float ds_sh[2];
  float gw0 = 0.f, gw1 = 0.f, gb0 = 0.f, gb1 = 0.f;
  for (int c = c0; c < min(c0 + kGroup, N); ++c) {
    const size_t base = ((size_t)bh * L + (size_t)c * kChunk) * D;
    // pooled feature, the two score partials, the <dout, out> partial
    float p = 0.f;
    if (feat) {
      const T* src = tid < D ? q + base + tid : k + base + (tid - D);
#pragma unroll 8
      for (int t = 0; t < kChunk; ++t) p += to_f32(src[(size_t)t * D]);
      p *= 1.0f / kChunk;
    }
    float gp = 0.f;
    {
      const int col = tid % D, r0 = tid / D;
#pragma unroll 4
      for (int t = r0; t < kChunk; t += RS) gp += to_f32(dout[base + (size_t)t * D + col]) *
                                                   to_f32(out[base + (size_t)t * D + col]);
    }
    float s0 = warp_sum(w0 * p), s1 = warp_sum(w1 * p);
    gp = warp_sum(gp);
    if (lane == 0) {
      red[0][warp] = s0;
      red[1][warp] = s1;
      red[2][warp] = gp;
    }
    __syncthreads();
    if (tid == 0) {
      float a = bs0, b = bs1, G = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) a += red[0][w], b += red[1][w], G += red[2][w];
      // pi = softmax(a, b); ds = G (e_sel - pi)
      const float m = fmaxf(a, b);
      const float ea = expf(a - m), eb = expf(b - m);
      const float pa = ea / (ea + eb), pb = eb / (ea + eb);
      const int s = sel[bh * N + c];
      ds_sh[0] = G * ((s == 0 ? 1.f : 0.f) - pa);
      ds_sh[1] = G * ((s == 1 ? 1.f : 0.f) - pb);
    }
    __syncthreads();
    const float ds0 = ds_sh[0], ds1 = ds_sh[1];
    gb0 += ds0;
    gb1 += ds1;
    if (feat) {
      gw0 += ds0 * p;
      gw1 += ds1 * p;
      const float r = (w0 * ds0 + w1 * ds1) * (1.0f / kChunk);
      float* dst = tid < D ? dq + base + tid : dk + base + (tid - D);
#pragma unroll 8
      for (int t = 0; t < kChunk; ++t) dst[(size_t)t * D] += r;
    }
    __syncthreads();  // red / ds_sh are rewritten by the next chunk
  }
  if (feat) {
    atomicAdd(dw_s + (size_t)h * 2 * F + tid, gw0);
    atomicAdd(dw_s + (size_t)h * 2 * F + F + tid, gw1);
  }
  if (tid == 0) {
    atomicAdd(db_s + 2 * h, gb0);
    atomicAdd(db_s + 2 * h + 1, gb1);
  }
}

}  // namespace

cudaError_t launch_score_bwd(const Problem& p, int dtype, const void* q, const void* k, const float* w_s,
                             const float* b_s, const uint8_t* sel, const void* out, const void* dout, float* dq,
                             float* dk, float* dw_s, float* db_s, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dw_s, 0, (size_t)p.H * 2 * 2 * p.d * sizeof(float), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(db_s, 0, (size_t)p.H * 2 * sizeof(float), st);
  if (e != cudaSuccess || p.BH == 0 || p.N == 0) return e;
  const unsigned grid = (unsigned)(p.BH * ((p.N + kGroup - 1) / kGroup));
  using bf = __nv_bfloat16;
  if (dtype == 0) {
    if (p.d == 64)
      score_bwd_kernel<bf, 64><<<grid, 256, 0, st>>>((const bf*)q, (const bf*)k, w_s, b_s, sel, (const bf*)out,
                                                     (const bf*)dout, p.H, p.N, p.L, dq, dk, dw_s, db_s);
    else
      score_bwd_kernel<bf, 128><<<grid, 256, 0, st>>>((const bf*)q, (const bf*)k, w_s, b_s, sel, (const bf*)out,
                                                      (const bf*)dout, p.H, p.N, p.L, dq, dk, dw_s, db_s);
  } else {
    if (p.d == 64)
      score_bwd_kernel<float, 64><<<grid, 256, 0, st>>>((const float*)q, (const float*)k, w_s, b_s, sel,
                                                        (const float*)out, (const float*)dout, p.H, p.N, p.L, dq,
                                                        dk, dw_s, db_s);
    else
      score_bwd_kernel<float, 128><<<grid, 256, 0, st>>>((const float*)q, (const float*)k, w_s, b_s, sel,
                                                         (const float*)out, (const float*)dout, p.H, p.N, p.L,
                                                         dq, dk, dw_s, db_s);
  }
  return cudaGetLastError();
}

}  // namespace nats
