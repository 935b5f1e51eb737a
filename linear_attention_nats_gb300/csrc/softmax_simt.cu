// softmax_simt.cu - softmax branch over the retained KV set, plain fp32 FMA
// (no tensor cores).  This is the fp32-input path: fp32 operands need fp32
// arithmetic to meet a 1e-4 relative bound, which the bf16 tensor-core
// kernel cannot give.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the softmax state is the set of keys and values
// of the chunks that chose softmax; inside a chunk both correlations are
// computed, so every query of chunk c attends to the retained chunks before
// c plus its own chunk causally (diagonal included).
#include "common.cuh"
#include "kernels.h"

namespace nats {

// One CTA (8 warps) per (query chunk c, b*h).  Warp w owns query rows
// 8w .. 8w+7; a lane keeps D/32 output columns of each row and computes the
// logits of keys lane and lane+32.  Online softmax in the exp2 domain.
template <class T, int D>
__global__ void __launch_bounds__(256) softmax_simt_kernel(const T* __restrict__ q,
                                                           const T* __restrict__ k,
                                                           const T* __restrict__ v,
                                                           const int32_t* __restrict__ nprev,
                                                           const int32_t* __restrict__ sel_idx,
                                                           int L, int N, float qscale,
                                                           float* __restrict__ o_s) {
  constexpr int C = kChunk, KP = D + 1, NC = D / 32;
  extern __shared__ float smem[];
  float* Qs = smem;            // [C][D]   q * scale * log2(e)
  float* Ks = Qs + C * D;      // [C][D+1]
  float* Vs = Ks + C * KP;     // [C][D]
  const int c = blockIdx.x;
  const long long bh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t head = (size_t)bh * L * D;
  for (int e = tid; e < C * D; e += 256) Qs[e] = to_f32(q[head + (size_t)c * C * D + e]) * qscale;
  float m[8], l[8], o[8][NC];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int i = 0; i < NC; ++i) o[r][i] = 0.f;
  }
  const int n_prev = nprev[bh * N + c];
  for (int item = 0; item <= n_prev; ++item) {
    const bool diag = (item == n_prev);
    const int kc = diag ? c : sel_idx[bh * N + item];
    __syncthreads();
    const size_t kb = head + (size_t)kc * C * D;
    for (int e = tid; e < C * D; e += 256) {
      const int t = e / D, f = e % D;
      Ks[t * KP + f] = to_f32(k[kb + e]);
      Vs[e] = to_f32(v[kb + e]);
    }
    __syncthreads();
#pragma unroll 1
    for (int r = 0; r < 8; ++r) {
      const int row = warp * 8 + r;
      const float* qr = Qs + row * D;
      const float* k0 = Ks + lane * KP;
      const float* k1 = Ks + (lane + 32) * KP;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int f = 0; f < D; ++f) {
        const float qf = qr[f];
        s0 = fmaf(qf, k0[f], s0);
        s1 = fmaf(qf, k1[f], s1);
      }
      if (diag) {
        if (lane > row) s0 = -INFINITY;
        if (lane + 32 > row) s1 = -INFINITY;
      }
      const float m_new = fmaxf(m[r], warp_max(fmaxf(s0, s1)));
      const float alpha = exp2f(m[r] - m_new);
      const float p0 = exp2f(s0 - m_new), p1 = exp2f(s1 - m_new);
      l[r] = l[r] * alpha + warp_sum(p0 + p1);
      m[r] = m_new;
#pragma unroll
      for (int i = 0; i < NC; ++i) o[r][i] *= alpha;
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const float pa = __shfl_sync(0xffffffffu, p0, j);
        const float pb = __shfl_sync(0xffffffffu, p1, j);
#pragma unroll
        for (int i = 0; i < NC; ++i)
          o[r][i] = fmaf(pa, Vs[j * D + lane + 32 * i], fmaf(pb, Vs[(j + 32) * D + lane + 32 * i], o[r][i]));
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = warp * 8 + r;
    const float inv = 1.f / l[r];
    float* dst = o_s + head + (size_t)(c * C + row) * D;
#pragma unroll
    for (int i = 0; i < NC; ++i) dst[lane + 32 * i] = o[r][i] * inv;
  }
}

template <class T, int D>
static cudaError_t launch_t(const Problem& p, const void* q, const void* k, const void* v,
                            const int32_t* nprev, const int32_t* sel_idx, float* o_s,
                            cudaStream_t st) {
  constexpr int C = kChunk;
  const size_t smem = sizeof(float) * (size_t)(C * D + C * (D + 1) + C * D);
  auto kern = softmax_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.N, (unsigned)p.BH);
  kern<<<grid, 256, smem, st>>>((const T*)q, (const T*)k, (const T*)v, nprev, sel_idx, p.L, p.N,
                                p.scale * 1.4426950408889634f, o_s);
  return cudaGetLastError();
}

cudaError_t launch_softmax_simt(const Problem& p, int dtype, const void* q, const void* k,
                                const void* v, const int32_t* nprev, const int32_t* sel_idx,
                                float* o_s, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  if (dtype == 0) {
    return p.d == 64 ? launch_t<__nv_bfloat16, 64>(p, q, k, v, nprev, sel_idx, o_s, st)
                     : launch_t<__nv_bfloat16, 128>(p, q, k, v, nprev, sel_idx, o_s, st);
  }
  return p.d == 64 ? launch_t<float, 64>(p, q, k, v, nprev, sel_idx, o_s, st)
                   : launch_t<float, 128>(p, q, k, v, nprev, sel_idx, o_s, st);
}

}  // namespace nats
