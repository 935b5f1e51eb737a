// proj.cu - the projections around the layer: x -> Q, K, V, g, beta (two
// GEMMs and one split kernel), the layer forward, and the output projection.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 4 (the merge weights come from projections of the
// query); the projections themselves follow the plain Gated DeltaNet form,
// as the reading stated in include/nats.h:
//   [q | k' | v] = bf16(x W_qkv), k = bf16(k' / |k'|) per head,
//   [a | b] = x W_ab, g = -a_scale softplus(a + b_a), beta = sigmoid(b + b_b),
//   y = bf16(o_flat W_o), o_flat[t] = [o_t,0 | o_t,1 | ...] (heads side by side).
// The GEMMs are cuBLAS (plain dense products, fp32 accumulate); the rest is
// two memory-bound kernels of this file.
#include <cublas_v2.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/nats.h"
#include "common.cuh"

namespace nats {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct XWorkspace {
  __nv_bfloat16* qkv;  // [B L, 3 H d] GEMM output; reused as o_flat [B L, H d]
  float* ab;           // [B L, 2 H]
  __nv_bfloat16 *q, *k, *v;  // [B, H, L, d]
  float *g, *beta;           // [B, H, L]
  __nv_bfloat16* o;          // [B, H, L, d] layer output
  void* layer;               // nats_hybrid_fwd workspace
  size_t layer_bytes;
};

size_t x_layout(const nats_dims* d, int hidden, char* base, XWorkspace* w) {
  (void)hidden;
  const size_t BL = (size_t)d->B * d->L, H = (size_t)d->H, D = (size_t)d->dk;
  const size_t BHL = (size_t)d->B * d->H * d->L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  XWorkspace x;
  x.qkv = (__nv_bfloat16*)take(BL * 3 * H * D * 2);
  x.ab = (float*)take(BL * 2 * H * 4);
  x.q = (__nv_bfloat16*)take(BHL * D * 2);
  x.k = (__nv_bfloat16*)take(BHL * D * 2);
  x.v = (__nv_bfloat16*)take(BHL * D * 2);
  x.g = (float*)take(BHL * 4);
  x.beta = (float*)take(BHL * 4);
  x.o = (__nv_bfloat16*)take(BHL * D * 2);
  x.layer_bytes = nats_workspace_size(d);
  x.layer = take(x.layer_bytes);
  if (w) *w = x;
  return off;
}

// One warp per (token, head): splits the projected row into q, k, v in the
// layer's [B, H, L, d] layout, normalises k, and forms g and beta.
template <int D>
__global__ void __launch_bounds__(256) proj_split_kernel(const __nv_bfloat16* __restrict__ qkv,
                                                         const float* __restrict__ ab, int B, int H, int L,
                                                         const float* __restrict__ b_a,
                                                         const float* __restrict__ a_scale,
                                                         const float* __restrict__ b_b,
                                                         __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                                                         __nv_bfloat16* __restrict__ v, float* __restrict__ g,
                                                         float* __restrict__ beta) {
  constexpr int E = D / 32;  // elements per lane
  const long long item = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (row, h), h fastest
  const long long rows = (long long)B * L;
  if (item >= rows * H) return;
  const int lane = threadIdx.x & 31;
  const int h = (int)(item % H);
  const long long row = item / H;  // b L + l
  const long long b = row / L, l = row - b * L;
  const size_t src = (size_t)row * 3 * H * D + (size_t)h * D + E * lane;
  const size_t dst = (((size_t)b * H + h) * L + l) * D + E * lane;
  float kf[E], ss = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    q[dst + i] = qkv[src + i];
    v[dst + i] = qkv[src + 2 * (size_t)H * D + i];
    kf[i] = __bfloat162float(qkv[src + (size_t)H * D + i]);
    ss = fmaf(kf[i], kf[i], ss);
  }
  ss = warp_sum(ss);
  const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) k[dst + i] = __float2bfloat16_rn(kf[i] * inv);
  if (lane == 0) {
    const float a = ab[(size_t)row * 2 * H + h] + (b_a ? b_a[h] : 0.f);
    const float bb = ab[(size_t)row * 2 * H + H + h] + (b_b ? b_b[h] : 0.f);
    const float sp = a > 20.f ? a : log1pf(__expf(a));  // softplus
    const size_t gi = ((size_t)b * H + h) * L + l;
    g[gi] = -(a_scale ? a_scale[h] : 1.f) * sp;
    beta[gi] = 1.f / (1.f + __expf(-bb));
  }
}

// o [B, H, L, d] -> o_flat [B L, H d] (heads side by side), one warp per row
// of d elements
template <int D>
__global__ void __launch_bounds__(256) heads_to_rows_kernel(const __nv_bfloat16* __restrict__ o, int B, int H,
                                                            int L, __nv_bfloat16* __restrict__ of) {
  constexpr int E = D / 32;
  const long long item = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, l, h), h fastest
  if (item >= (long long)B * L * H) return;
  const int lane = threadIdx.x & 31;
  const int h = (int)(item % H);
  const long long row = item / H;
  const long long b = row / L, l = row - b * L;
  const size_t src = (((size_t)b * H + h) * L + l) * D + E * lane;
  const size_t dst = (size_t)row * H * D + (size_t)h * D + E * lane;
#pragma unroll
  for (int i = 0; i < E; ++i) of[dst + i] = o[src + i];
}

// One cuBLAS handle per device; the enqueue of a call's GEMMs holds the
// device's lock (the handle's stream is per-handle state).
struct Blas {
  std::mutex mu;
  bool tried = false;
  cublasHandle_t h = nullptr;
};

Blas* blas_of_current_device() {
  static std::mutex mu;
  static Blas all[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  Blas& b = all[dev];
  if (!b.tried) {
    b.tried = true;
    if (cublasCreate(&b.h) != CUBLAS_STATUS_SUCCESS) b.h = nullptr;
  }
  return b.h ? &b : nullptr;
}

// Row-major C[M, N] = A[M, K] B[K, N] (bf16 operands, fp32 accumulate), as
// the column-major product C^T = B^T A^T.
bool gemm_rm(cublasHandle_t hdl, int M, int N, int K, const void* A, const void* B, void* C,
             cudaDataType_t ctype) {
  const float one = 1.f, zero = 0.f;
  return cublasGemmEx(hdl, CUBLAS_OP_N, CUBLAS_OP_N, N, M, K, &one, B, CUDA_R_16BF, N, A, CUDA_R_16BF, K, &zero,
                      C, ctype, N, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

}  // namespace
}  // namespace nats

using namespace nats;

extern "C" {

size_t nats_x_workspace_size(const nats_dims* dims, int32_t hidden) {
  if (!dims || hidden <= 0 || hidden % 8 != 0 || dims->dtype != NATS_BF16) return 0;
  if (nats_workspace_size(dims) == 0 && (long long)dims->B * dims->H * dims->L > 0) return 0;
  return x_layout(dims, hidden, nullptr, nullptr);
}

nats_status nats_hybrid_fwd_x(const nats_dims* dims, int32_t hidden, const void* x, const void* w_qkv,
                              const void* w_ab, const float* b_a, const float* a_scale, const float* b_b,
                              const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                              const void* w_o, void* y, uint8_t* sel_out, void* workspace,
                              size_t workspace_bytes, nats_stream_t stream) {
  if (!dims) return NATS_ERR_NULL;
  if (dims->dtype != NATS_BF16) return NATS_ERR_DTYPE;
  if (hidden <= 0 || hidden % 8 != 0) return NATS_ERR_SHAPE;
  // shape / value checks of the layer (dims only: the layer's pointers live
  // in the workspace)
  if (nats_workspace_size(dims) == 0 && (long long)dims->B * dims->H * dims->L > 0) {
    const nats_status s = nats_select(dims, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
    return s != NATS_OK ? s : NATS_ERR_SHAPE;
  }
  if ((long long)dims->B * dims->H * dims->L == 0) return NATS_OK;
  if (!x || !w_qkv || !w_ab || !w_s || !w_g || !w_o || !y || !workspace) return NATS_ERR_NULL;
  if (((uintptr_t)x | (uintptr_t)w_qkv | (uintptr_t)w_ab | (uintptr_t)w_o | (uintptr_t)y | (uintptr_t)workspace) & 15)
    return NATS_ERR_ALIGN;
  XWorkspace xw;
  if (workspace_bytes < x_layout(dims, hidden, (char*)workspace, &xw)) return NATS_ERR_WORKSPACE;
  const int B = dims->B, H = dims->H, L = dims->L, D = dims->dk;
  const int BL = B * L, HD = H * D;
  cudaStream_t st = (cudaStream_t)stream;
  Blas* bl = blas_of_current_device();
  if (!bl) return NATS_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(bl->mu);
    if (cublasSetStream(bl->h, st) != CUBLAS_STATUS_SUCCESS) return NATS_ERR_CUDA;
    if (!gemm_rm(bl->h, BL, 3 * HD, hidden, x, w_qkv, xw.qkv, CUDA_R_16BF)) return NATS_ERR_CUDA;
    if (!gemm_rm(bl->h, BL, 2 * H, hidden, x, w_ab, xw.ab, CUDA_R_32F)) return NATS_ERR_CUDA;
  }
  const long long items = (long long)BL * H;
  const unsigned blocks = (unsigned)((items + 7) / 8);
  if (D == 64)
    proj_split_kernel<64><<<blocks, 256, 0, st>>>(xw.qkv, xw.ab, B, H, L, b_a, a_scale, b_b, xw.q, xw.k, xw.v, xw.g,
                                                  xw.beta);
  else
    proj_split_kernel<128><<<blocks, 256, 0, st>>>(xw.qkv, xw.ab, B, H, L, b_a, a_scale, b_b, xw.q, xw.k, xw.v,
                                                   xw.g, xw.beta);
  if (cudaGetLastError() != cudaSuccess) return NATS_ERR_CUDA;
  const nats_status s = nats_hybrid_fwd(dims, xw.q, xw.k, xw.v, xw.g, xw.beta, w_s, b_s, w_g, b_g, nullptr, nullptr,
                                        nullptr, xw.o, sel_out, nullptr, nullptr, nullptr, xw.layer, xw.layer_bytes,
                                        stream);
  if (s != NATS_OK) return s;
  __nv_bfloat16* of = xw.qkv;  // the projected rows are dead by now
  if (D == 64)
    heads_to_rows_kernel<64><<<blocks, 256, 0, st>>>(xw.o, B, H, L, of);
  else
    heads_to_rows_kernel<128><<<blocks, 256, 0, st>>>(xw.o, B, H, L, of);
  if (cudaGetLastError() != cudaSuccess) return NATS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(bl->mu);
  if (cublasSetStream(bl->h, st) != CUBLAS_STATUS_SUCCESS) return NATS_ERR_CUDA;
  if (!gemm_rm(bl->h, BL, hidden, HD, of, w_o, y, CUDA_R_16BF)) return NATS_ERR_CUDA;
  return NATS_OK;
}

}  // extern "C"
