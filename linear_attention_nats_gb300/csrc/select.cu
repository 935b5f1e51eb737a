// select.cu - chunk scorer (mean pool + linear score + argmax) and the
// compaction of softmax-selected chunks.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 1 (Attention Score Layer: mean pooling followed by
// a linear layer, one score per operation, highest score wins) and item 3
// (only the selected operation keeps a chunk's keys and values: the softmax
// branch of chunk c sees exactly the softmax-selected chunks before c).
#include "common.cuh"
#include "kernels.h"

namespace nats {

// One CTA of 128 threads per (b, h, chunk).  Thread j owns pooled features
// j and j + 128 of [q ; k] (2d <= 256); every load of a token row is
// coalesced across the CTA.  HBM-bound: each chunk's Q and K are read once.
template <class T>
__global__ void __launch_bounds__(128) score_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                    const float* __restrict__ w_s,
                                                    const float* __restrict__ b_s, int H, int L,
                                                    int d, int N, uint8_t* __restrict__ sel,
                                                    float* __restrict__ scores) {
  const long long blk = blockIdx.x;  // (bh, c)
  const int c = (int)(blk % N);
  const long long bh = blk / N;
  const int h = (int)(bh % H);
  const int tid = threadIdx.x;
  const int F = 2 * d;
  const size_t base = ((size_t)bh * L + (size_t)c * kChunk) * d;
  float acc[2] = {0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int f = tid + 128 * u;
    if (f < F) {
      const T* src = (f < d) ? (q + base + f) : (k + base + (f - d));
      float s = 0.f;
#pragma unroll 8
      for (int t = 0; t < kChunk; ++t) s += to_f32(src[(size_t)t * d]);
      acc[u] = s * (1.0f / kChunk);
    }
  }
  const float* W = w_s + (size_t)h * 2 * F;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int f = tid + 128 * u;
    if (f < F) {
      s0 += W[f] * acc[u];
      s1 += W[F + f] * acc[u];
    }
  }
  __shared__ float red[2][4];
  s0 = warp_sum(s0);
  s1 = warp_sum(s1);
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = s0;
    red[1][tid >> 5] = s1;
  }
  __syncthreads();
  if (tid == 0) {
    float a = red[0][0] + red[0][1] + red[0][2] + red[0][3];
    float b = red[1][0] + red[1][1] + red[1][2] + red[1][3];
    if (b_s) {
      a += b_s[2 * h];
      b += b_s[2 * h + 1];
    }
    sel[blk] = (a >= b) ? 0 : 1;  // ties go to softmax
    if (scores) {
      scores[2 * blk] = a;
      scores[2 * blk + 1] = b;
    }
  }
}

// One CTA per (b, h): exclusive prefix count of softmax chunks and the
// compacted, ordered list of their indices.  Optionally mirrors the
// selection into a second buffer (sel_copy).
__global__ void __launch_bounds__(256) compact_kernel(const uint8_t* __restrict__ sel, int N,
                                                      int32_t* __restrict__ nprev,
                                                      int32_t* __restrict__ sel_idx,
                                                      uint8_t* __restrict__ sel_copy) {
  const long long bh = blockIdx.x;
  const uint8_t* s = sel + bh * N;
  int32_t* np = nprev + bh * N;
  int32_t* si = sel_idx + bh * N;
  __shared__ int warp_tot[8];
  __shared__ int running;
  if (threadIdx.x == 0) running = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int c0 = 0; c0 < N; c0 += 256) {
    const int c = c0 + threadIdx.x;
    const uint8_t code = (c < N) ? s[c] : 1;
    if (c < N && sel_copy) sel_copy[bh * N + c] = code;
    const int flag = (c < N && code == 0) ? 1 : 0;
    int x = flag;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    int before = running;
    for (int w = 0; w < wid; ++w) before += warp_tot[w];
    const int excl = before + x - flag;
    if (c < N) {
      np[c] = excl;
      if (flag) si[excl] = c;
    }
    __syncthreads();
    if (threadIdx.x == 255) running = excl + flag;
    __syncthreads();
  }
}

cudaError_t launch_score(const Problem& p, int dtype, const void* q, const void* k, const float* w_s,
                         const float* b_s, uint8_t* sel, float* scores, cudaStream_t st) {
  const long long blocks = p.BH * p.N;
  if (blocks == 0) return cudaSuccess;
  if (dtype == 0)
    score_kernel<__nv_bfloat16><<<(unsigned)blocks, 128, 0, st>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, w_s, b_s, p.H, p.L, p.d, p.N, sel, scores);
  else
    score_kernel<float><<<(unsigned)blocks, 128, 0, st>>>((const float*)q, (const float*)k, w_s, b_s,
                                                          p.H, p.L, p.d, p.N, sel, scores);
  return cudaGetLastError();
}

cudaError_t launch_compact(const Problem& p, const uint8_t* sel, int32_t* nprev, int32_t* sel_idx,
                           uint8_t* sel_copy, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  compact_kernel<<<(unsigned)p.BH, 256, 0, st>>>(sel, p.N, nprev, sel_idx, sel_copy);
  return cudaGetLastError();
}

}  // namespace nats
