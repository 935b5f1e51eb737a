// merge.cu - per-branch RMSNorm and query-gated weighted sum.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 4: both branch outputs are RMS-normalised on their
// own and combined by a weighted sum whose weight is generated from the
// query: out = w N_soft + (1 - w) N_lin, w = sigmoid(q . W_g[h] + b_g[h]),
// N_x = x / sqrt(mean(x^2) + eps) * norm_w.
#include "common.cuh"
#include "kernels.h"

namespace nats {

// One warp per token row; a lane owns D/32 strided columns (coalesced).
template <class T, int D>
__global__ void __launch_bounds__(256) norm_merge_kernel(
    const float* __restrict__ o_s, const float* __restrict__ o_l, const T* __restrict__ q,
    const float* __restrict__ w_g, const float* __restrict__ b_g, const float* __restrict__ nw_s,
    const float* __restrict__ nw_l, int H, int L, long long rows, float eps, T* __restrict__ out) {
  constexpr int NC = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int h = (int)((row / L) % H);
  const size_t base = (size_t)row * D;
  float xs[NC], xl[NC];
  float ss = 0.f, sl = 0.f, z = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int col = lane + 32 * i;
    xs[i] = o_s[base + col];
    xl[i] = o_l[base + col];
    ss = fmaf(xs[i], xs[i], ss);
    sl = fmaf(xl[i], xl[i], sl);
    z = fmaf(to_f32(q[base + col]), w_g[(size_t)h * D + col], z);
  }
  ss = warp_sum(ss);
  sl = warp_sum(sl);
  z = warp_sum(z) + (b_g ? b_g[h] : 0.f);
  const float rs = rsqrtf(ss * (1.f / D) + eps);
  const float rl = rsqrtf(sl * (1.f / D) + eps);
  const float w = 1.f / (1.f + expf(-z));
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int col = lane + 32 * i;
    const float ns = xs[i] * rs * (nw_s ? nw_s[col] : 1.f);
    const float nl = xl[i] * rl * (nw_l ? nw_l[col] : 1.f);
    out[base + col] = from_f32<T>(w * ns + (1.f - w) * nl);
  }
}

// bf16 path, second half of the merge: out already holds w RMSNorm(o_s)
// (written by the softmax kernel's epilogue); add (1 - w) RMSNorm(o_l).  One
// warp per token row, coalesced; HBM-bound.  o_l is fp32, or the bf16 copy the
// scan writes when the caller does not ask for o_l (half the bytes to read).
template <int D, class TL>
__global__ void __launch_bounds__(256) merge_lin_kernel(const TL* __restrict__ o_l,
                                                        const float* __restrict__ gate,
                                                        const float* __restrict__ nw_l, long long rows,
                                                        float eps, __nv_bfloat16* __restrict__ out) {
  constexpr int E = D / 32;  // contiguous elements per lane (vector loads / stores)
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const size_t base = (size_t)row * D + E * lane;
  float xl[E], sl = 0.f;
  if constexpr (sizeof(TL) == 2) {
    // bf16: E = 4 -> one 8-byte load, E = 2 -> one 4-byte load
    if constexpr (E == 4) {
      const uint2 u = *(const uint2*)(o_l + base);
      const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)&u.x);
      const float2 b = __bfloat1622float2(*(const __nv_bfloat162*)&u.y);
      xl[0] = a.x; xl[1] = a.y; xl[2] = b.x; xl[3] = b.y;
    } else {
      const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)(o_l + base));
      xl[0] = a.x; xl[1] = a.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) xl[i] = to_f32(o_l[base + i]);
  }
#pragma unroll
  for (int i = 0; i < E; ++i) sl = fmaf(xl[i], xl[i], sl);
  sl = warp_sum(sl);
  const float f = (1.f - gate[row]) * rsqrtf(sl * (1.f / D) + eps);
  __nv_bfloat162* o2 = (__nv_bfloat162*)(out + base);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 prev = __bfloat1622float2(o2[i]);
    const int col = E * lane + 2 * i;
    const float w0 = nw_l ? nw_l[col] : 1.f, w1 = nw_l ? nw_l[col + 1] : 1.f;
    o2[i] = __floats2bfloat162_rn(prev.x + f * xl[2 * i] * w0, prev.y + f * xl[2 * i + 1] * w1);
  }
}

template <class T, int D>
static cudaError_t launch_t(const Problem& p, const float* o_s, const float* o_l, const void* q,
                            const float* w_g, const float* b_g, const float* nw_s,
                            const float* nw_l, void* out, cudaStream_t st) {
  const long long rows = p.BH * p.L;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  norm_merge_kernel<T, D><<<blocks, 256, 0, st>>>(o_s, o_l, (const T*)q, w_g, b_g, nw_s, nw_l, p.H,
                                                  p.L, rows, p.eps, (T*)out);
  return cudaGetLastError();
}

cudaError_t launch_norm_merge(const Problem& p, int dtype, const float* o_s, const float* o_l,
                              const void* q, const float* w_g, const float* b_g, const float* nw_s,
                              const float* nw_l, void* out, cudaStream_t st) {
  if (p.BH == 0 || p.L == 0) return cudaSuccess;
  if (dtype == 0)
    return p.d == 64 ? launch_t<__nv_bfloat16, 64>(p, o_s, o_l, q, w_g, b_g, nw_s, nw_l, out, st)
                     : launch_t<__nv_bfloat16, 128>(p, o_s, o_l, q, w_g, b_g, nw_s, nw_l, out, st);
  return p.d == 64 ? launch_t<float, 64>(p, o_s, o_l, q, w_g, b_g, nw_s, nw_l, out, st)
                   : launch_t<float, 128>(p, o_s, o_l, q, w_g, b_g, nw_s, nw_l, out, st);
}

cudaError_t launch_merge_lin(const Problem& p, const float* o_l, const void* o_l16, const float* gate,
                             const float* nw_l, void* out, cudaStream_t st) {
  const long long rows = p.BH * p.L;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  __nv_bfloat16* o = (__nv_bfloat16*)out;
  const __nv_bfloat16* l16 = (const __nv_bfloat16*)o_l16;
  if (l16)
    p.d == 64 ? merge_lin_kernel<64><<<blocks, 256, 0, st>>>(l16, gate, nw_l, rows, p.eps, o)
              : merge_lin_kernel<128><<<blocks, 256, 0, st>>>(l16, gate, nw_l, rows, p.eps, o);
  else
    p.d == 64 ? merge_lin_kernel<64><<<blocks, 256, 0, st>>>(o_l, gate, nw_l, rows, p.eps, o)
              : merge_lin_kernel<128><<<blocks, 256, 0, st>>>(o_l, gate, nw_l, rows, p.eps, o);
  return cudaGetLastError();
}

}  // namespace nats
