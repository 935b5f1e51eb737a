// kernels.h - host-side launchers of the libnats kernels (internal).
#pragma once

#include "common.cuh"

namespace nats {

// dtype: 0 = bf16, 1 = fp32 (nats_dtype).

cudaError_t launch_score(const Problem& p, int dtype, const void* q, const void* k, const float* w_s,
                         const float* b_s, uint8_t* sel, float* scores, cudaStream_t st);

cudaError_t launch_compact(const Problem& p, const uint8_t* sel, int32_t* nprev, int32_t* sel_idx,
                           uint8_t* sel_copy, cudaStream_t st);

// bf16 softmax branch; its epilogue writes out = w RMSNorm(o_s) (bf16) with
// the per-token gate w; o_s (fp32 diagnostics) may be null, and so may
// lse_out (fp32 [BH, L]: each row's log2-sum-exp2 of its scores times
// scale log2 e, the backward pass's row statistic).
cudaError_t launch_softmax_tc(const Problem& p, const void* q, const void* k, const void* v,
                              const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel,
                              const float* gate, const float* nw_s, void* out, float* o_s, float* lse_out,
                              int* err, cudaStream_t st);

cudaError_t launch_softmax_simt(const Problem& p, int dtype, const void* q, const void* k,
                                const void* v, const int32_t* nprev, const int32_t* sel_idx,
                                float* o_s, cudaStream_t st);

cudaError_t launch_gdn_prep_simt(const Problem& p, int dtype, const void* q, const void* k,
                                 const void* v, const float* g, const float* beta,
                                 const Workspace& ws, cudaStream_t st);

cudaError_t launch_gdn_scan_simt(const Problem& p, int dtype, const void* q, const void* k,
                                 const uint8_t* sel, const Workspace& ws, float* o_l,
                                 float* state_out, cudaStream_t st);

// bf16 chunk factors of the Gated DeltaNet branch plus the per-token merge
// gate; T_out (or null) receives T = (I + A)^{-1} of every chunk, fp32
// [BH, N, C, C], zero above the diagonal.
cudaError_t launch_gdn_prep_mma(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* w_g, const float* b_g, float* G, void* W16,
                                void* U16, void* P16, float* gate, const float* w_s, const float* b_s,
                                uint8_t* sel_out, float* T_out, cudaStream_t st);

// The same factors (d = 128) from the persistent tcgen05 pipeline; err[0] is
// set if one of its bounded waits expires.
cudaError_t launch_gdn_prep_tc(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* w_g, const float* b_g, float* G, void* W16,
                               void* U16, void* P16, float* gate, const float* w_s, const float* b_s,
                               uint8_t* sel_out, int* err, float* T_out, cudaStream_t st);

// bf16 chunk scan: o_l (fp32 [BH, L, dv]); state_out may be null; s0_out
// (or null) receives every chunk's start state, fp32 [BH, N, dv, dk].
cudaError_t launch_gdn_scan_tc(const Problem& p, const void* q, const void* k, const uint8_t* sel, const float* G,
                               const void* W16, const void* UT16, const void* P16, float* o_l, void* o_l16,
                               float* state_out, int* err, cudaStream_t st, float* s0_out = nullptr);

// One decode step of the layer (dtype 0 = bf16, 1 = fp32), one CTA per (b, h).
cudaError_t launch_decode_step(const Problem& p, int dtype, long long t, const void* q, const void* k,
                               const void* v, const float* g, const float* beta, const float* w_s,
                               const float* b_s, const float* w_g, const float* b_g, const float* nw_s,
                               const float* nw_l, float* S, float* S0, void* ck, void* cv, float* psum,
                               void* kv_k, void* kv_v, int32_t* n_kv, long long cap, void* out,
                               uint8_t* sel_out, float* o_s_out, float* o_l_out, int* err, cudaStream_t st);

// Backward pass at a given selection (backward.cu): its scratch bytes, and
// the launches (norm + merge, softmax dq and dk / dv, Gated DeltaNet adjoint,
// per-token combine).  ev_start / ev_stop (NATS_BWD_STAGE_* ids, entries may
// be NULL) are recorded around each stage, launches[stage] counts its kernels.
size_t bwd_workspace_bytes(const Problem& p, int dtype);
cudaError_t launch_hybrid_bwd(const Problem& p, int dtype, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* w_g, const float* b_g,
                              const float* nws, const float* nwl, const uint8_t* sel, const float* o_s,
                              const float* o_l, const void* dout, float* dq, float* dk, float* dv, float* dg,
                              float* dbeta, float* dw_g, float* db_g, float* dnws, float* dnwl, void* ws,
                              cudaStream_t st, void* const* ev_start = nullptr, void* const* ev_stop = nullptr,
                              int32_t* launches = nullptr, cudaStream_t side = nullptr, cudaEvent_t fork = nullptr,
                              cudaEvent_t join = nullptr, const float* lse_in = nullptr);

// The score layer's gradient under the straight-through surrogate
// (score_bwd.cu): zeroes dw_s, db_s, then sums into them and adds the score
// layer's share into dq, dk.
cudaError_t launch_score_bwd(const Problem& p, int dtype, const void* q, const void* k, const float* w_s,
                             const float* b_s, const uint8_t* sel, const void* out, const void* dout, float* dq,
                             float* dk, float* dw_s, float* db_s, cudaStream_t st);

// Chunkwise Gated DeltaNet adjoint of bf16 layers (gdn_bwd_chunk.cu): its
// scratch, carved from the backward workspace.
struct GdnBwdScratch {
  float* S0;    // [BH, N, dk, dv] chunk-start states, transposed (the forward recompute writes them)
  float* dSC;   // [BH, N, dk, dv] gradient of each committed chunk's end state, transposed
  float* G;     // [BH, L] in-chunk cumulative log-decay
  float* Li;    // [BH, N, C, C] (I + diag(beta) A)^{-1} (the forward's chunk-factor kernel stores it)
  float* P;     // [BH, N, C, C] lower(e^{G_i - G_j} scale q_i . k_j)
  void* W16;    // [BH, L, dk] fp16: Linv diag(beta gamma) K  \  each times its chunk's
  void* Qe16;   // [BH, L, dk] fp16: diag(gamma) Q~ - P W      >  power-of-two scale
  void* Kt16;   // [BH, L, dk] fp16: diag(gamma_C / gamma) K  /   (sc)
  float* sc;    // [BH, N, 4] the scales of W, Q_eff, K~
};
// the adjoint's chunk factors (one kernel; it reads q, k, g, beta and Linv
// and writes only the scratch: G, P, W, Q_eff, K~ and their scales)
cudaError_t launch_gdn_bwd_factors(const Problem& p, const void* q, const void* k, const float* g,
                                   const float* beta, const GdnBwdScratch& w, cudaStream_t st);
// the reverse state-gradient scan (one kernel, after the factors; it reads
// them, the selection and dO, and writes dS_C of every committed chunk)
cudaError_t launch_gdn_bwd_reverse_scan(const Problem& p, const uint8_t* sel, const float* dO,
                                        const GdnBwdScratch& w, cudaStream_t st);
// every per-chunk product of the adjoint, after the factors, the reverse
// scan and the chunk-start states S0 (one kernel, on tcgen05 for d = 128;
// dq, dk, dv accumulate, dg and dbeta are overwritten; err[0] is set if a
// bounded wait expires)
cudaError_t launch_gdn_bwd_products(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                                    const float* beta, const uint8_t* sel, const float* dO, const GdnBwdScratch& w,
                                    float* dq, float* dk, float* dv, float* dg, float* dbeta, int* err,
                                    cudaStream_t st);

// Softmax branch of the backward pass on tcgen05 (softmax_bwd_tc.cu), bf16
// layers: lse (fp32 [BH, L], exp2 domain) and dq (+=), then dk, dv (=); the
// compacted softmax-chunk lists (nprev, sel_idx) as the forward builds them;
// lse_in (or null) is the forward's row statistic, which then replaces the
// query-tile kernel's first pass (lse is not written); err[0] is set if a
// bounded wait expires.
cudaError_t launch_softmax_bwd_tc(const Problem& p, const void* q, const void* k, const void* v, const void* dos,
                                  const float* delta, const int32_t* nprev, const int32_t* sel_idx,
                                  const uint8_t* sel, float* lse, const float* lse_in, float* dq, float* dk,
                                  float* dv, int* err, cudaStream_t st);

// The projections around the layer on tcgen05 (gemm_tc.cu).  QKV: x W_qkv
// into the layer's q, k (normalised per head), v [B, H, L, d] and x W_ab into
// g, beta [B, H, L]; w_ab_pad is scratch of proj_gate_pad_bytes(H, hidden).
// Out: y = o_flat W_o, o read from its [B, H, L, d] layout.  err[0] is set if
// a bounded wait expires.
size_t proj_gate_pad_bytes(int H, int hidden);
cudaError_t launch_proj_qkv_tc(int B, int H, int L, int d, int hidden, const void* x, const void* w_qkv,
                               const void* w_ab, void* w_ab_pad, const float* b_a, const float* a_scale,
                               const float* b_b, void* q, void* k, void* v, float* g, float* beta, int* err,
                               cudaStream_t st);
cudaError_t launch_proj_out_tc(int B, int H, int L, int d, int hidden, const void* o, const void* w_o, void* y,
                               int* err, cudaStream_t st);

// Native Hybrid Attention (nha.cu): workspace bytes, the two launches (slot
// state scan, unless w >= L; the attention), and the bounded-wait flag.
size_t nha_workspace_bytes(long long BH, int L);
// ev_start / ev_stop (or null): cudaEvent_t handles recorded around the
// slot scan [0] and the attention [1]; *launches counts the kernels.
cudaError_t launch_nha_fwd(long long BH, int L, int window, float scale, const void* q, const void* k, const void* v,
                           const float* log_alpha, void* out, void* ws, cudaStream_t st, void* const* ev_start,
                           void* const* ev_stop, int* launches);
int* nha_err_flag(void* ws, long long BH, int L);

// Test hook: one bounded wait that runs out after limit_ns and sets *flag.
cudaError_t launch_bounded_wait(int* flag, long long limit_ns, cudaStream_t st);

// bf16 path: out (holding w RMSNorm(o_s)) += (1 - w) RMSNorm(o_l).
cudaError_t launch_merge_lin(const Problem& p, const float* o_l, const void* o_l16, const float* gate,
                             const float* nw_l, void* out, cudaStream_t st);

cudaError_t launch_norm_merge(const Problem& p, int dtype, const float* o_s, const float* o_l,
                              const void* q, const float* w_g, const float* b_g, const float* nw_s,
                              const float* nw_l, void* out, cudaStream_t st);

}  // namespace nats
