// no_alloc.cu - nats_hybrid_fwd for callers that cannot allocate device
// memory.
//
// Who needs it: code that runs where cudaMalloc is not an option, for example
// a plugin inside a host application that owns all device memory through its
// own pool (a raw cudaMalloc would bypass that pool and can synchronise the
// whole device), a latency-critical loop that must never block on an
// allocation, or a plain C caller with no allocator of its own that still
// wants to pass only its inputs and outputs.  Such callers cannot provide the
// workspace nats_hybrid_fwd asks for, so this entry point brings its own.
//
// The scratch is one file-scope device array of kNoAllocScratchBytes, created
// when the library is loaded and held on every GPU that loads it until the
// process exits.  Host code cannot pass the array's name to a kernel (in host
// code it names a host-side stand-in, not device memory), so the first call
// on each device looks up its device address with cudaGetSymbolAddress, with
// that device current, and remembers it.  cudaDeviceReset unloads the
// library's device code and with it the array, so the remembered address is
// stale after a reset: the entry point is not for use on a device that the
// process has reset since its first call there.
#include <mutex>

#include "../../include/nats.h"

namespace nats {
nats_status check_fwd_args(const nats_dims* dims, const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* w_s, const float* w_g, const uint8_t* sel_in,
                           const void* out, bool* empty);
}  // namespace nats

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
nats_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NATS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return NATS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return NATS_OK;
}

}  // namespace

extern "C" nats_status nats_hybrid_fwd_noalloc(
    const nats_dims* dims, const void* q, const void* k, const void* v, const float* g, const float* beta,
    const float* w_s, const float* b_s, const float* w_g, const float* b_g, const float* norm_w_soft,
    const float* norm_w_lin, const uint8_t* sel_in, void* out, uint8_t* sel_out, float* state_out,
    float* o_soft_out, float* o_lin_out, nats_stream_t stream) {
  // the checks of nats_hybrid_fwd, in its order, before the size limit
  bool empty = false;
  const nats_status s0 = nats::check_fwd_args(dims, q, k, v, g, beta, w_s, w_g, sel_in, out, &empty);
  if (s0 != NATS_OK || empty) return s0;
  if (nats_workspace_size(dims) > kNoAllocScratchBytes) return NATS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const nats_status s = scratch_address(&scratch);
  if (s != NATS_OK) return s;
  // Nothing in the scratch has to start at zero: every call writes each part
  // of it before reading it (the error flag is cleared by the call itself).
  return nats_hybrid_fwd(dims, q, k, v, g, beta, w_s, b_s, w_g, b_g, norm_w_soft, norm_w_lin, sel_in, out,
                         sel_out, state_out, o_soft_out, o_lin_out, scratch, kNoAllocScratchBytes, stream);
}

extern "C" nats_status nats_noalloc_check(const nats_dims* dims, nats_stream_t stream) {
  if (nats_workspace_size(dims) > kNoAllocScratchBytes) return NATS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const nats_status s = scratch_address(&scratch);
  if (s != NATS_OK) return s;
  return nats_workspace_check(dims, scratch, stream);
}
