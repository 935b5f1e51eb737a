// api.cu - the C ABI of libnats: argument validation, workspace layout and
// the launch sequence of the NAtS-L hybrid attention layer forward.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/nats.h"
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape / dtype / value checks shared by every entry point.
nats_status check_dims(const nats_dims* d) {
  if (!d) return NATS_ERR_NULL;
  if (d->dtype != NATS_BF16 && d->dtype != NATS_F32) return NATS_ERR_DTYPE;
  if (d->B < 0 || d->H < 0 || d->L < 0 || d->dk <= 0 || d->dv <= 0) return NATS_ERR_SHAPE;
  if (d->chunk != kChunk || d->L % kChunk != 0 || d->dk != d->dv) return NATS_ERR_SHAPE;
  if (d->dk != 64 && d->dk != 128) return NATS_ERR_UNSUPPORTED;
  if (!std::isfinite(d->scale) || d->scale < 0.f || !std::isfinite(d->eps) || d->eps < 0.f)
    return NATS_ERR_VALUE;
  // every flat element offset must fit the int64 / int32 grid arithmetic,
  // and every TMA row coordinate a 32-bit int: the largest is a line of the
  // transposed chunk factor U^T, (B H N + c) d
  const long long BH = (long long)d->B * d->H;
  if (BH > (1LL << 31) - 1 || BH * (d->L / kChunk) * d->dk > (1LL << 31) - 1) return NATS_ERR_UNSUPPORTED;
  return NATS_OK;
}

Problem problem_of(const nats_dims* d) {
  Problem p;
  p.B = d->B;
  p.H = d->H;
  p.L = d->L;
  p.d = d->dk;
  p.N = d->L / kChunk;
  p.BH = (long long)d->B * d->H;
  p.scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->dk);
  p.eps = d->eps;
  return p;
}

// Carves the workspace; returns the bytes needed.  `base` may be null
// (size query only).
size_t layout(const Problem& p, char* base, Workspace* ws) {
  const size_t BH = (size_t)p.BH, N = (size_t)p.N, L = (size_t)p.L, D = (size_t)p.d;
  const size_t C = kChunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* ptr = base ? base + off : nullptr;
    off += align_up(bytes);
    return ptr;
  };
  Workspace w;
  w.sel = (uint8_t*)take(BH * N);
  w.nprev = (int32_t*)take(4 * BH * N);
  w.sel_idx = (int32_t*)take(4 * BH * N);
  w.G = (float*)take(4 * BH * L);
  w.W = (float*)take(4 * BH * L * D);
  w.U = (float*)take(4 * BH * L * D);
  w.P = (float*)take(4 * BH * N * C * C);
  w.o_s = (float*)take(4 * BH * L * D);
  w.o_l = (float*)take(4 * BH * L * D);
  w.gate = (float*)take(4 * BH * L);
  w.err = (int*)take(16);
  if (ws) *ws = w;
  return off;
}

// last CUDA error a libnats call on this host thread met
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
// test hook: the launch stage (nats_profile stage id) whose launch the next
// layer forward on this thread replaces by a cudaErrorInvalidValue; -1 none
thread_local int g_fail_stage = -1;

nats_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NATS_OK;
  g_last_cuda_error = e;
  return NATS_ERR_CUDA;
}

// Optional per-stage event records around each launch group.
struct Stages {
  nats_profile* prof;
  cudaStream_t st;
  cudaError_t mark(void* const* ev, int s) const {
    if (!prof || !ev[s]) return cudaSuccess;
    return cudaEventRecord((cudaEvent_t)ev[s], st);
  }
};

#define NATS_STAGE(stg, id, n_launch, expr)                                           \
  do {                                                                                \
    if ((stg).prof && (stg).mark((stg).prof->start, id) != cudaSuccess) return NATS_ERR_CUDA; \
    if (g_fail_stage == (id)) {                                                       \
      g_fail_stage = -1;                                                              \
      return cuda_status(cudaErrorInvalidValue);                                      \
    }                                                                                 \
    if (cuda_status(expr) != NATS_OK) return NATS_ERR_CUDA;                           \
    if ((stg).prof) {                                                                 \
      (stg).prof->launches += (n_launch);                                             \
      (stg).prof->stage_launches[id] += (n_launch);                                   \
      if ((stg).mark((stg).prof->stop, id) != cudaSuccess) return NATS_ERR_CUDA;      \
    }                                                                                 \
  } while (0)

// The Gated DeltaNet scan is sequential in the chunks of a head: one CTA per
// (b, h), so it occupies at most B*H SMs.  The softmax kernel runs
// concurrently on a second stream: the scan is launched on the caller's
// stream right behind the chunk factors, so its CTAs are placed first, and
// the softmax kernel's persistent CTAs, which take tiles dynamically, fill
// the remaining SMs and then the ones the scan releases.  One stream and two
// events per device, created on first use; the fork / join is enqueued under
// a lock so that calls from several host threads do not interleave.
struct Side {
  std::mutex mu;
  bool tried = false;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

Side* side_of_current_device() {
  static std::mutex mu;
  static Side sides[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  Side& sd = sides[dev];
  if (!sd.tried) {
    sd.tried = true;
    if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
      sd.s = nullptr;
      cudaGetLastError();
    }
  }
  return sd.s ? &sd : nullptr;
}

}  // namespace

// Argument checks of the layer forward other than the workspace (shared with
// the allocation-free entry point, so both report the same error first).
// *empty is set when a zero extent makes the call a no-op.
nats_status check_fwd_args(const nats_dims* dims, const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* w_s, const float* w_g, const uint8_t* sel_in,
                           const void* out, bool* empty) {
  *empty = false;
  nats_status s = check_dims(dims);
  if (s != NATS_OK) return s;
  if ((long long)dims->B * dims->H == 0 || dims->L == 0) {
    *empty = true;
    return NATS_OK;
  }
  if (!q || !k || !v || !g || !beta || !w_g || !out) return NATS_ERR_NULL;
  if (!sel_in && !w_s) return NATS_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return NATS_ERR_ALIGN;
  return NATS_OK;
}

}  // namespace nats

using namespace nats;

extern "C" {

const char* nats_status_string(nats_status s) {
  switch (s) {
    case NATS_OK: return "NATS_OK";
    case NATS_ERR_NULL: return "NATS_ERR_NULL: a required pointer is NULL";
    case NATS_ERR_SHAPE: return "NATS_ERR_SHAPE: bad extent (chunk must be 64, L % 64 == 0, dk == dv)";
    case NATS_ERR_DTYPE: return "NATS_ERR_DTYPE: dtype must be NATS_BF16 or NATS_F32";
    case NATS_ERR_ALIGN: return "NATS_ERR_ALIGN: a pointer is not 16-byte aligned";
    case NATS_ERR_WORKSPACE: return "NATS_ERR_WORKSPACE: workspace too small";
    case NATS_ERR_UNSUPPORTED: return "NATS_ERR_UNSUPPORTED: head size must be 64 or 128";
    case NATS_ERR_CUDA: return "NATS_ERR_CUDA: a CUDA call or kernel launch failed";
    case NATS_ERR_INTERNAL: return "NATS_ERR_INTERNAL";
    case NATS_ERR_VALUE: return "NATS_ERR_VALUE: scale / eps must be finite and >= 0";
  }
  return "unknown nats_status";
}

const char* nats_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

void nats_debug_fail_stage(int32_t stage) { g_fail_stage = stage; }

nats_status nats_debug_bounded_wait(int32_t* flag, int64_t limit_ns, nats_stream_t stream) {
  if (!flag) return NATS_ERR_NULL;
  if (limit_ns <= 0 || limit_ns > 1000000000LL) return NATS_ERR_VALUE;
  return cuda_status(launch_bounded_wait(flag, limit_ns, (cudaStream_t)stream));
}

size_t nats_workspace_size(const nats_dims* dims) {
  if (check_dims(dims) != NATS_OK) return 0;
  return layout(problem_of(dims), nullptr, nullptr);
}

nats_status nats_workspace_check(const nats_dims* dims, const void* workspace, nats_stream_t stream) {
  nats_status s = check_dims(dims);
  if (s != NATS_OK) return s;
  const Problem p = problem_of(dims);
  if (p.BH == 0 || p.L == 0) return NATS_OK;
  if (!workspace) return NATS_ERR_NULL;
  Workspace ws;
  layout(p, (char*)workspace, &ws);
  int flag = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&flag, ws.err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return NATS_ERR_CUDA;
  return flag ? NATS_ERR_INTERNAL : NATS_OK;
}

nats_status nats_select(const nats_dims* dims, const void* q, const void* k, const float* w_s,
                        const float* b_s, uint8_t* sel, float* scores, nats_stream_t stream) {
  nats_status s = check_dims(dims);
  if (s != NATS_OK) return s;
  const Problem p = problem_of(dims);
  if (p.BH == 0 || p.L == 0) return NATS_OK;
  if (!q || !k || !w_s || !sel) return NATS_ERR_NULL;
  if (!aligned16(q) || !aligned16(k)) return NATS_ERR_ALIGN;
  return cuda_status(launch_score(p, dims->dtype, q, k, w_s, b_s, sel, scores, (cudaStream_t)stream));
}

nats_status nats_hybrid_fwd_streams(const nats_dims* dims, const void* q, const void* k,
                                    const void* v, const float* g, const float* beta,
                                    const float* w_s, const float* b_s, const float* w_g,
                                    const float* b_g, const float* norm_w_soft,
                                    const float* norm_w_lin, const uint8_t* sel_in, void* out,
                                    uint8_t* sel_out, float* state_out, float* o_soft_out,
                                    float* o_lin_out, float* lse_out, void* workspace, size_t workspace_bytes,
                                    nats_stream_t stream, const nats_streams* streams,
                                    nats_profile* prof) {
  bool empty = false;
  nats_status s = check_fwd_args(dims, q, k, v, g, beta, w_s, w_g, sel_in, out, &empty);
  if (s != NATS_OK) return s;
  if (lse_out && dims->dtype != NATS_BF16) return NATS_ERR_DTYPE;  // the row statistic of the bf16 path
  // caller-owned concurrency: a second stream other than `stream` needs both events
  const bool own_side = streams && streams->side && streams->side != stream;
  if (own_side && (!streams->fork || !streams->join)) return NATS_ERR_NULL;
  const Problem p = problem_of(dims);
  if (prof) {
    prof->launches = 0;
    for (int i = 0; i < NATS_NUM_STAGES; ++i) prof->stage_launches[i] = 0;
  }
  if (empty) return NATS_OK;
  if (!workspace) return NATS_ERR_NULL;
  if (!aligned16(workspace)) return NATS_ERR_ALIGN;
  Workspace ws;
  const size_t need = layout(p, (char*)workspace, &ws);
  if (workspace_bytes < need) return NATS_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const int dt = dims->dtype;
  Stages stg{prof, st};
  // err[0]: bounded-wait flag; err[1]: tile counter of the softmax kernel's
  // dynamic schedule.  Both start at zero before the first kernel runs.
  if (cudaMemsetAsync(ws.err, 0, 2 * sizeof(int), st) != cudaSuccess) return NATS_ERR_CUDA;

  // 1. selection (score layer, or the caller's override).  With bf16 inputs
  //    the chunk-factor kernel scores the chunks from the Q and K it stages.
  const uint8_t* sel = sel_in;
  uint8_t* score_dst = nullptr;
  if (!sel) {
    score_dst = sel_out ? sel_out : ws.sel;
    if (dt != NATS_BF16)
      NATS_STAGE(stg, NATS_STAGE_SCORE, 1, launch_score(p, dt, q, k, w_s, b_s, score_dst, nullptr, st));
    sel = score_dst;
  }
  if (dt == NATS_BF16) {
    // 2. Gated DeltaNet chunk factors, the per-token merge gate (and the selection)
    if (p.d == 128)
      NATS_STAGE(stg, NATS_STAGE_GDN_PREP, 1,
                 launch_gdn_prep_tc(p, q, k, v, g, beta, w_g, b_g, ws.G, ws.W, ws.U, ws.P, ws.gate, w_s, b_s,
                                    score_dst, ws.err, nullptr, st));
    else
      NATS_STAGE(stg, NATS_STAGE_GDN_PREP, 1,
                 launch_gdn_prep_mma(p, q, k, v, g, beta, w_g, b_g, ws.G, ws.W, ws.U, ws.P, ws.gate, w_s, b_s,
                                     score_dst, nullptr, st));
  }
  // 3. compacted softmax-chunk lists (mirrors an overridden selection to sel_out)
  NATS_STAGE(stg, NATS_STAGE_COMPACT, 1,
             launch_compact(p, sel, ws.nprev, ws.sel_idx, (sel_in && sel_out) ? sel_out : nullptr, st));
  if (dt == NATS_BF16) {
    // 4. Gated DeltaNet chunk scan with commit / rollback (caller's stream)
    // 5. softmax branch, concurrently on the side stream (in order on the
    //    caller's stream if that stream could not be made); its epilogue
    //    writes out = w RMSNorm(o_s)
    // o_l goes to the caller's fp32 buffer if asked for, else as bf16 into the
    // workspace (the merge reads half the bytes)
    float* o_l = o_lin_out;
    void* o_l16 = o_lin_out ? nullptr : (void*)ws.o_l;
    // (the caller's second stream and events, or the library's per-device
    // ones, or none: in order on `stream`)
    Side* sd = streams ? nullptr : side_of_current_device();
    {
      std::unique_lock<std::mutex> lk;
      cudaStream_t ss = st;
      cudaEvent_t fork = nullptr, join = nullptr;
      if (own_side) {
        ss = (cudaStream_t)streams->side;
        fork = (cudaEvent_t)streams->fork;
        join = (cudaEvent_t)streams->join;
      } else if (sd) {
        lk = std::unique_lock<std::mutex>(sd->mu);
        ss = sd->s;
        fork = sd->fork;
        join = sd->join;
      }
      if (ss != st && (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(ss, fork, 0) != cudaSuccess))
        return NATS_ERR_CUDA;
      NATS_STAGE(stg, NATS_STAGE_GDN_SCAN, 1,
                 launch_gdn_scan_tc(p, q, k, sel, ws.G, ws.W, ws.U, ws.P, o_l, o_l16, state_out, ws.err, st));
      Stages stg_side{prof, ss};
      NATS_STAGE(stg_side, NATS_STAGE_SOFTMAX, 1,
                 launch_softmax_tc(p, q, k, v, ws.nprev, ws.sel_idx, sel, ws.gate, norm_w_soft, out, o_soft_out,
                                   lse_out, ws.err, ss));
      if (ss != st && (cudaEventRecord(join, ss) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess))
        return NATS_ERR_CUDA;
    }
    // 6. out += (1 - w) RMSNorm(o_l)
    NATS_STAGE(stg, NATS_STAGE_MERGE, 1, launch_merge_lin(p, o_l, o_l16, ws.gate, norm_w_lin, out, st));
  } else {
    // fp32 inputs: softmax branch, Gated DeltaNet branch, then RMSNorm + merge
    float* o_s = o_soft_out ? o_soft_out : ws.o_s;
    NATS_STAGE(stg, NATS_STAGE_SOFTMAX, 1,
               launch_softmax_simt(p, dt, q, k, v, ws.nprev, ws.sel_idx, o_s, st));
    float* o_l = o_lin_out ? o_lin_out : ws.o_l;
    NATS_STAGE(stg, NATS_STAGE_GDN_PREP, 1, launch_gdn_prep_simt(p, dt, q, k, v, g, beta, ws, st));
    NATS_STAGE(stg, NATS_STAGE_GDN_SCAN, 1,
               launch_gdn_scan_simt(p, dt, q, k, sel, ws, o_l, state_out, st));
    NATS_STAGE(stg, NATS_STAGE_MERGE, 1,
               launch_norm_merge(p, dt, o_s, o_l, q, w_g, b_g, norm_w_soft, norm_w_lin, out, st));
  }
  return NATS_OK;
}

nats_status nats_hybrid_fwd_profiled(const nats_dims* dims, const void* q, const void* k,
                                     const void* v, const float* g, const float* beta,
                                     const float* w_s, const float* b_s, const float* w_g,
                                     const float* b_g, const float* norm_w_soft,
                                     const float* norm_w_lin, const uint8_t* sel_in, void* out,
                                     uint8_t* sel_out, float* state_out, float* o_soft_out,
                                     float* o_lin_out, void* workspace, size_t workspace_bytes,
                                     nats_stream_t stream, nats_profile* prof) {
  return nats_hybrid_fwd_streams(dims, q, k, v, g, beta, w_s, b_s, w_g, b_g, norm_w_soft, norm_w_lin, sel_in, out,
                                 sel_out, state_out, o_soft_out, o_lin_out, nullptr, workspace, workspace_bytes,
                                 stream, nullptr, prof);
}

nats_status nats_hybrid_fwd(const nats_dims* dims, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const float* w_s, const float* b_s,
                            const float* w_g, const float* b_g, const float* norm_w_soft,
                            const float* norm_w_lin, const uint8_t* sel_in, void* out,
                            uint8_t* sel_out, float* state_out, float* o_soft_out,
                            float* o_lin_out, void* workspace, size_t workspace_bytes,
                            nats_stream_t stream) {
  return nats_hybrid_fwd_profiled(dims, q, k, v, g, beta, w_s, b_s, w_g, b_g, norm_w_soft,
                                  norm_w_lin, sel_in, out, sel_out, state_out, o_soft_out,
                                  o_lin_out, workspace, workspace_bytes, stream, nullptr);
}

size_t nats_bwd_workspace_size(const nats_dims* dims) {
  if (check_dims(dims) != NATS_OK) return 0;
  return bwd_workspace_bytes(problem_of(dims), dims->dtype);
}

nats_status nats_hybrid_bwd(const nats_dims* dims, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* w_g, const float* b_g, const float* norm_w_soft,
                            const float* norm_w_lin, const uint8_t* sel, const float* o_soft,
                            const float* o_lin, const void* dout, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, float* dw_g, float* db_g, float* dnorm_w_soft, float* dnorm_w_lin,
                            void* workspace, size_t workspace_bytes, nats_stream_t stream) {
  return nats_hybrid_bwd_profiled(dims, q, k, v, g, beta, w_g, b_g, norm_w_soft, norm_w_lin, sel, o_soft, o_lin,
                                  dout, dq, dk, dv, dg, dbeta, dw_g, db_g, dnorm_w_soft, dnorm_w_lin, workspace,
                                  workspace_bytes, stream, nullptr);
}

nats_status nats_hybrid_bwd_profiled(const nats_dims* dims, const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, const float* w_g, const float* b_g,
                                     const float* norm_w_soft, const float* norm_w_lin, const uint8_t* sel,
                                     const float* o_soft, const float* o_lin, const void* dout, float* dq,
                                     float* dk, float* dv, float* dg, float* dbeta, float* dw_g, float* db_g,
                                     float* dnorm_w_soft, float* dnorm_w_lin, void* workspace,
                                     size_t workspace_bytes, nats_stream_t stream, nats_profile* prof) {
  return nats_hybrid_bwd_streams(dims, q, k, v, g, beta, w_g, b_g, norm_w_soft, norm_w_lin, sel, o_soft, o_lin,
                                 nullptr, dout, dq, dk, dv, dg, dbeta, dw_g, db_g, dnorm_w_soft, dnorm_w_lin,
                                 workspace, workspace_bytes, stream, nullptr, prof);
}

nats_status nats_hybrid_bwd_streams(const nats_dims* dims, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* w_g, const float* b_g,
                                    const float* norm_w_soft, const float* norm_w_lin, const uint8_t* sel,
                                    const float* o_soft, const float* o_lin, const float* lse, const void* dout,
                                    float* dq,
                                    float* dk, float* dv, float* dg, float* dbeta, float* dw_g, float* db_g,
                                    float* dnorm_w_soft, float* dnorm_w_lin, void* workspace,
                                    size_t workspace_bytes, nats_stream_t stream, const nats_streams* streams,
                                    nats_profile* prof) {
  if (prof) {
    prof->launches = 0;
    for (int i = 0; i < NATS_NUM_STAGES; ++i) prof->stage_launches[i] = 0;
  }
  nats_status s = check_dims(dims);
  if (s != NATS_OK) return s;
  const Problem p = problem_of(dims);
  if (p.BH == 0 || p.L == 0) return NATS_OK;
  if (!q || !k || !v || !g || !beta || !w_g || !sel || !o_soft || !o_lin || !dout || !dq || !dk || !dv || !dg ||
      !dbeta || !workspace)
    return NATS_ERR_NULL;
  const void* ptrs[] = {q, k, v, o_soft, o_lin, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return NATS_ERR_ALIGN;
  if (lse && !aligned16(lse)) return NATS_ERR_ALIGN;
  // caller-owned concurrency: a second stream other than `stream` needs both events
  const bool own_side = streams && streams->side && streams->side != stream;
  if (own_side && (!streams->fork || !streams->join)) return NATS_ERR_NULL;
  if (workspace_bytes < bwd_workspace_bytes(p, dims->dtype)) return NATS_ERR_WORKSPACE;
  // bf16 layers: the Gated DeltaNet state work runs on a second stream (the
  // caller's, or the library's per-device one; in order on `stream` if
  // neither is given or the library's could not be made)
  cudaStream_t ss = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::unique_lock<std::mutex> lk;
  if (own_side) {
    ss = (cudaStream_t)streams->side;
    fork = (cudaEvent_t)streams->fork;
    join = (cudaEvent_t)streams->join;
  } else if (!streams && dims->dtype == NATS_BF16) {
    if (Side* sd = side_of_current_device()) {
      lk = std::unique_lock<std::mutex>(sd->mu);
      ss = sd->s;
      fork = sd->fork;
      join = sd->join;
    }
  }
  const nats_status r = cuda_status(launch_hybrid_bwd(
      p, dims->dtype, q, k, v, g, beta, w_g, b_g, norm_w_soft, norm_w_lin, sel, o_soft, o_lin, dout, dq, dk, dv, dg,
      dbeta, dw_g, db_g, dnorm_w_soft, dnorm_w_lin, workspace, (cudaStream_t)stream, prof ? prof->start : nullptr,
      prof ? prof->stop : nullptr, prof ? prof->stage_launches : nullptr, ss, fork, join,
      dims->dtype == NATS_BF16 ? lse : nullptr));
  if (prof)
    for (int i = 0; i < NATS_BWD_NUM_STAGES; ++i) prof->launches += prof->stage_launches[i];
  return r;
}

nats_status nats_score_bwd(const nats_dims* dims, const void* q, const void* k, const float* w_s, const float* b_s,
                           const uint8_t* sel, const void* out, const void* dout, float* dq, float* dk, float* dw_s,
                           float* db_s, nats_stream_t stream) {
  nats_status s = check_dims(dims);
  if (s != NATS_OK) return s;
  const Problem p = problem_of(dims);
  if (!q || !k || !w_s || !sel || !out || !dout || !dq || !dk || !dw_s || !db_s) return NATS_ERR_NULL;
  const void* ptrs[] = {q, k, out, dout, dq, dk};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return NATS_ERR_ALIGN;
  return cuda_status(launch_score_bwd(p, dims->dtype, q, k, w_s, b_s, sel, out, dout, dq, dk, dw_s, db_s,
                                      (cudaStream_t)stream));
}

nats_status nats_decode_step(const nats_dims* dims, int64_t t, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* w_s, const float* b_s,
                             const float* w_g, const float* b_g, const float* norm_w_soft,
                             const float* norm_w_lin, const nats_decode_state* state, void* out,
                             uint8_t* sel_out, float* o_soft_out, float* o_lin_out, nats_stream_t stream) {
  if (!dims) return NATS_ERR_NULL;
  nats_dims d = *dims;
  d.L = 0;  // not used in decode mode
  nats_status s = check_dims(&d);
  if (s != NATS_OK) return s;
  if (t < 0) return NATS_ERR_VALUE;
  const Problem p = problem_of(&d);
  if (p.BH == 0) return NATS_OK;
  if (!q || !k || !v || !g || !beta || !w_s || !w_g || !state || !out) return NATS_ERR_NULL;
  const nats_decode_state& st = *state;
  if (!st.S || !st.S0 || !st.ck || !st.cv || !st.psum || !st.kv_k || !st.kv_v || !st.n_kv || !st.err)
    return NATS_ERR_NULL;
  const void* ptrs[] = {q, k, v, out, st.S, st.S0, st.ck, st.cv, st.psum, st.kv_k, st.kv_v};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return NATS_ERR_ALIGN;
  if (st.cap < (long long)kChunk * (t / kChunk + 1)) return NATS_ERR_WORKSPACE;
  return cuda_status(launch_decode_step(p, d.dtype, t, q, k, v, g, beta, w_s, b_s, w_g, b_g, norm_w_soft,
                                        norm_w_lin, st.S, st.S0, st.ck, st.cv, st.psum, st.kv_k, st.kv_v, st.n_kv,
                                        st.cap, out, sel_out, o_soft_out, o_lin_out, st.err,
                                        (cudaStream_t)stream));
}

}  // extern "C"
