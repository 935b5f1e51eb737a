// common.cuh - shared device helpers and the problem / workspace description
// of libnats (NAtS-L hybrid attention layer forward).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nats {

constexpr int kChunk = 64;  // tokens per chunk (selection and chunkwise form)

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <class T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Sizes of one call.  BH = B * H; N = L / kChunk; d = dk = dv.
struct Problem {
  int B, H, L, d, N;
  long long BH;
  float scale;  // resolved (never 0)
  float eps;
};

// Device workspace carved from the caller's buffer (all 256-byte aligned).
struct Workspace {
  uint8_t* sel;      // [BH, N]   0 softmax / 1 Gated DeltaNet
  int32_t* nprev;    // [BH, N]   softmax chunks before chunk c
  int32_t* sel_idx;  // [BH, N]   compacted list of softmax chunks, in order
  float* G;          // [BH, L]   in-chunk cumulative log-decay
  float* W;          // [BH, N, C, dk]  T diag(beta e^G) K  (bf16 path: bf16)
  float* U;          // [BH, N, C, dv]  T diag(beta) V      (bf16 path: bf16, transposed [dv][C])
  float* P;          // [BH, N, C, C]   lower(e^{G_t - G_i} scale q_t . k_i)
  float* o_s;        // [BH, L, dv] softmax branch output (before norm)
  float* o_l;        // [BH, L, dv] Gated DeltaNet branch output (before norm)
  float* gate;       // [BH, L] merge weight w = sigmoid(q . W_g + b_g) (bf16 path)
  int* err;          // [0] set by a kernel whose bounded wait expired; [1] softmax tile counter
                     // (both zeroed at the start of each call)
};

}  // namespace nats
