// proj.cu - the layer with its projections: x -> Q, K, V, g, beta (one
// tcgen05 GEMM whose epilogue splits the heads, normalises the keys and
// forms the gates), the layer forward, and the output projection (the same
// GEMM kernel, reading the layer output in its [B, H, L, d] layout).
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 4 (the merge weights come from projections of the
// query); the projections themselves follow the plain Gated DeltaNet form,
// as the reading stated in include/nats.h:
//   [q | k' | v] = bf16(x W_qkv), k = bf16(k' / |k'|) per head,
//   [a | b] = x W_ab, g = -a_scale softplus(a + b_a), beta = sigmoid(b + b_b),
//   y = bf16(o_flat W_o), o_flat[t] = [o_t,0 | o_t,1 | ...] (heads side by side).
#include <cmath>
#include <cstdint>

#include "../../include/nats.h"
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct XWorkspace {
  __nv_bfloat16 *q, *k, *v;  // [B, H, L, d]
  float *g, *beta;           // [B, H, L]
  __nv_bfloat16* o;          // [B, H, L, d] layer output
  void* w_ab_pad;            // [hidden, 2H rounded up to 64] bf16
  int* err;                  // [0] set by a projection GEMM whose bounded wait expired
  void* layer;               // nats_hybrid_fwd workspace
  size_t layer_bytes;
};

size_t x_layout(const nats_dims* d, int hidden, char* base, XWorkspace* w) {
  const size_t BHL = (size_t)d->B * d->H * d->L, D = (size_t)d->dk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  XWorkspace x;
  x.q = (__nv_bfloat16*)take(BHL * D * 2);
  x.k = (__nv_bfloat16*)take(BHL * D * 2);
  x.v = (__nv_bfloat16*)take(BHL * D * 2);
  x.g = (float*)take(BHL * 4);
  x.beta = (float*)take(BHL * 4);
  x.o = (__nv_bfloat16*)take(BHL * D * 2);
  x.w_ab_pad = take(proj_gate_pad_bytes(d->H, hidden));
  x.err = (int*)take(16);
  x.layer_bytes = nats_workspace_size(d);
  x.layer = take(x.layer_bytes);
  if (w) *w = x;
  return off;
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

nats_status nats_x_workspace_check(const nats_dims* dims, int32_t hidden, const void* workspace,
                                   nats_stream_t stream) {
  if (nats_x_workspace_size(dims, hidden) == 0) return dims ? NATS_ERR_SHAPE : NATS_ERR_NULL;
  if ((long long)dims->B * dims->H * dims->L == 0) return NATS_OK;
  if (!workspace) return NATS_ERR_NULL;
  XWorkspace xw;
  x_layout(dims, hidden, (char*)workspace, &xw);
  int flag = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&flag, xw.err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return NATS_ERR_CUDA;
  if (flag) return NATS_ERR_INTERNAL;
  return nats_workspace_check(dims, xw.layer, stream);
}

nats_status nats_hybrid_fwd_x_profiled(const nats_dims* dims, int32_t hidden, const void* x, const void* w_qkv,
                                       const void* w_ab, const float* b_a, const float* a_scale, const float* b_b,
                                       const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                                       const void* w_o, void* y, uint8_t* sel_out, void* workspace,
                                       size_t workspace_bytes, nats_stream_t stream, nats_profile* prof) {
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
  // every flat offset of the projections fits int32 tiling
  if ((long long)dims->B * dims->L > (1LL << 31) - 1 - 128 ||
      3LL * dims->H * dims->dk > (1LL << 31) - 1)
    return NATS_ERR_UNSUPPORTED;
  XWorkspace xw;
  if (workspace_bytes < x_layout(dims, hidden, (char*)workspace, &xw)) return NATS_ERR_WORKSPACE;
  const int B = dims->B, H = dims->H, L = dims->L, D = dims->dk;
  cudaStream_t st = (cudaStream_t)stream;
  auto mark = [&](void* const* ev, int s) -> bool {
    return !prof || !ev[s] || cudaEventRecord((cudaEvent_t)ev[s], st) == cudaSuccess;
  };
  if (cudaMemsetAsync(xw.err, 0, sizeof(int), st) != cudaSuccess) return NATS_ERR_CUDA;
  if (!mark(prof ? prof->start : nullptr, NATS_STAGE_PROJ_IN)) return NATS_ERR_CUDA;
  if (launch_proj_qkv_tc(B, H, L, D, hidden, x, w_qkv, w_ab, xw.w_ab_pad, b_a, a_scale, b_b, xw.q, xw.k, xw.v,
                         xw.g, xw.beta, xw.err, st) != cudaSuccess)
    return NATS_ERR_CUDA;
  if (!mark(prof ? prof->stop : nullptr, NATS_STAGE_PROJ_IN)) return NATS_ERR_CUDA;
  // the layer fills the profile's other stages (and resets its counts)
  const nats_status s = nats_hybrid_fwd_profiled(dims, xw.q, xw.k, xw.v, xw.g, xw.beta, w_s, b_s, w_g, b_g, nullptr,
                                                 nullptr, nullptr, xw.o, sel_out, nullptr, nullptr, nullptr, xw.layer,
                                                 xw.layer_bytes, stream, prof);
  if (s != NATS_OK) return s;
  if (!mark(prof ? prof->start : nullptr, NATS_STAGE_PROJ_OUT)) return NATS_ERR_CUDA;
  if (launch_proj_out_tc(B, H, L, D, hidden, xw.o, w_o, y, xw.err, st) != cudaSuccess) return NATS_ERR_CUDA;
  if (!mark(prof ? prof->stop : nullptr, NATS_STAGE_PROJ_OUT)) return NATS_ERR_CUDA;
  if (prof) {
    prof->launches += 3;  // gate-weight copy, the two GEMMs
    prof->stage_launches[NATS_STAGE_PROJ_IN] = 2;
    prof->stage_launches[NATS_STAGE_PROJ_OUT] = 1;
  }
  return NATS_OK;
}

nats_status nats_hybrid_fwd_x(const nats_dims* dims, int32_t hidden, const void* x, const void* w_qkv,
                              const void* w_ab, const float* b_a, const float* a_scale, const float* b_b,
                              const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                              const void* w_o, void* y, uint8_t* sel_out, void* workspace,
                              size_t workspace_bytes, nats_stream_t stream) {
  return nats_hybrid_fwd_x_profiled(dims, hidden, x, w_qkv, w_ab, b_a, a_scale, b_b, w_s, b_s, w_g, b_g, w_o, y,
                                    sel_out, workspace, workspace_bytes, stream, nullptr);
}

}  // extern "C"
