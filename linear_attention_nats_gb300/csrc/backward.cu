// backward.cu - the layer's backward pass at the forward's selection:
// the gradient of <dout, out> with respect to q, k, v, g, beta, W_g, b_g and
// the two RMSNorm weights ("Neural Attention Search Linear (NAtS-L)",
// technical summary, "Kernmechanismen" items 3 and 4; item 5 says the
// selection is learned end to end but gives no estimator for the argmax: the
// score layer's surrogate gradient is a separate call, score_bwd.cu).
//
// Stages, every result in fp32:
//   1. norm + merge, one warp per token: with N_x = o_x r_x w_x,
//      r_x = (mean(o_x^2) + eps)^(-1/2), out = w N_s + (1 - w) N_l and
//      w = sigmoid(q . W_g + b_g):
//        dN_s = w dout, dN_l = (1 - w) dout, dz = w (1 - w) <dout, N_s - N_l>,
//        do_x = r_x (w_x dN_x) - o_x r_x^3 <w_x dN_x, o_x> / d,
//      dq = dz W_g (the gate's share), and the weight gradients (dW_g,
//      db_g, the norm weights) summed per CTA, then atomically;
//   2. softmax branch, from the row log-sum-exp: P_tj = exp(s_tj - lse_t),
//      dS_tj = P_tj (do_s,t . v_j - do_s,t . o_s,t); bf16 layers on tcgen05
//      (softmax_bwd_tc.cu); fp32 layers here: a row pass (one warp per
//      query) takes lse_t and dq_t += scale sum_j dS_tj k_j, a key pass (one
//      warp per key) dk_j = scale sum_t dS_tj q_t and dv_j = sum_t P_tj do_s,t
//      over the queries that see key j (the rest of its chunk, and every
//      later query when its chunk chose softmax);
//   3. Gated DeltaNet.  bf16 layers: the chunk-start states recomputed by the
//      forward's own kernels, then the chunkwise adjoint (gdn_bwd_chunk.cu);
//      the recompute and the adjoint's chunk factors and reverse scan run on
//      a second stream beside stage 2.  fp32 layers, one CTA per (b, h): the
//      forward is replayed for the chunk-start states, then the adjoint runs
//      backwards token by token.  Per token, with
//      u = S_{t-1} k, e = v - a u, S_t = a S_{t-1} + beta e k^T and
//      o_t = S_t (scale q):
//        dS_t += do_t (scale q)^T, dq += scale S_t^T do_t (formed as
//        a S_{t-1}^T do_t + beta <e, do_t> k, so S_t is not needed),
//        x = dS_t k, de = beta x, dbeta = <e, x>, dv = de,
//        dk = beta dS_t^T e - a S_{t-1}^T de,
//        da = <dS_t, S_{t-1}> - <u, de>, dg = a da,
//        dS_{t-1} = a dS_t - a de k^T.
//      A chunk that chose softmax was rolled back: the state after it is its
//      start state, so the gradient arriving there passes to the start
//      unchanged and the tokens inside start from zero.  The states inside a
//      chunk are replayed into scratch before its tokens are reversed.  The
//      state rows are split between two CTAs per head; a last kernel adds
//      the halves' column sums and scalars per token.
#include <type_traits>

#include "../../include/nats.h"
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int kMergeRows = 64;  // token rows per CTA of the merge stage

template <int E>
__device__ __forceinline__ void row_load(const float* p, float (&o)[E]) {
#pragma unroll
  for (int x = 0; x < E; ++x) o[x] = p[x];
}
template <int E>
__device__ __forceinline__ void row_load(const __nv_bfloat16* p, float (&o)[E]) {
#pragma unroll
  for (int x = 0; x < E; ++x) o[x] = __bfloat162float(p[x]);
}
// E (2 or 4) consecutive elements at an E-aligned offset, one vector access
template <int E>
__device__ __forceinline__ void vec_load(const float* p, float (&o)[E]) {
  if constexpr (E == 4) {
    const float4 v = *(const float4*)p;
    o[0] = v.x, o[1] = v.y, o[2] = v.z, o[3] = v.w;
  } else {
    const float2 v = *(const float2*)p;
    o[0] = v.x, o[1] = v.y;
  }
}
template <int E>
__device__ __forceinline__ void vec_load(const __nv_bfloat16* p, float (&o)[E]) {
  if constexpr (E == 4) {
    const uint2 v = *(const uint2*)p;
    const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)&v.x), b = __bfloat1622float2(*(const __nv_bfloat162*)&v.y);
    o[0] = a.x, o[1] = a.y, o[2] = b.x, o[3] = b.y;
  } else {
    const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)p);
    o[0] = a.x, o[1] = a.y;
  }
}
template <int E>
__device__ __forceinline__ void vec_store(float* p, const float (&o)[E]) {
  if constexpr (E == 4)
    *(float4*)p = make_float4(o[0], o[1], o[2], o[3]);
  else
    *(float2*)p = make_float2(o[0], o[1]);
}
template <int E>
__device__ __forceinline__ void vec_store(__nv_bfloat16* p, const float (&o)[E]) {
  if constexpr (E == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
    uint2 v;
    v.x = *(const uint32_t*)&a;
    v.y = *(const uint32_t*)&b;
    *(uint2*)p = v;
  } else {
    *(__nv_bfloat162*)p = __floats2bfloat162_rn(o[0], o[1]);
  }
}

// ------------------------------------------------------------ 1. merge
template <typename T, int D>
__global__ void __launch_bounds__(256) merge_bwd_kernel(
    const T* __restrict__ q, const T* __restrict__ dout, const float* __restrict__ o_s,
    const float* __restrict__ o_l, const float* __restrict__ w_g, const float* __restrict__ b_g,
    const float* __restrict__ nws, const float* __restrict__ nwl, int H, int L, float eps,
    float* __restrict__ d_os, __nv_bfloat16* __restrict__ d_os16, float* __restrict__ d_ol,
    float* __restrict__ delta, float* __restrict__ dq, float* __restrict__ dw_g, float* __restrict__ db_g,
    float* __restrict__ dnws, float* __restrict__ dnwl) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_head = L / kMergeRows;
  const long long bh = blockIdx.x / per_head;
  const int h = (int)(bh % H);
  const int row0 = (int)(blockIdx.x % per_head) * kMergeRows;
  __shared__ float red[8][3][D];
  __shared__ float red_b[8];
  float wg[E], ws[E], wl[E];
#pragma unroll
  for (int x = 0; x < E; ++x) {
    const int f = lane * E + x;
    wg[x] = w_g[(long long)h * D + f];
    ws[x] = nws ? nws[f] : 1.f;
    wl[x] = nwl ? nwl[f] : 1.f;
  }
  const float bg = b_g ? b_g[h] : 0.f;
  float a_wg[E], a_ns[E], a_nl[E], a_bg = 0.f;
#pragma unroll
  for (int x = 0; x < E; ++x) a_wg[x] = a_ns[x] = a_nl[x] = 0.f;
  for (int r = warp; r < kMergeRows; r += 8) {
    const long long t = bh * L + row0 + r;
    float os[E], ol[E], R[E], qv[E];
    vec_load<E>(o_s + t * D + lane * E, os);
    vec_load<E>(o_l + t * D + lane * E, ol);
    vec_load<E>(dout + t * D + lane * E, R);
    vec_load<E>(q + t * D + lane * E, qv);
    float ss = 0.f, sl = 0.f, z = 0.f;
#pragma unroll
    for (int x = 0; x < E; ++x) {
      ss = fmaf(os[x], os[x], ss);
      sl = fmaf(ol[x], ol[x], sl);
      z = fmaf(qv[x], wg[x], z);
    }
    ss = warp_sum(ss);
    sl = warp_sum(sl);
    z = warp_sum(z) + bg;
    const float rs = rsqrtf(ss / D + eps), rl = rsqrtf(sl / D + eps);
    const float w = 1.f / (1.f + expf(-z));
    float dw = 0.f, gs = 0.f, gl = 0.f;  // <dout, N_s - N_l>, <w_s dN_s, o_s>, <w_l dN_l, o_l>
#pragma unroll
    for (int x = 0; x < E; ++x) {
      dw = fmaf(R[x], os[x] * rs * ws[x] - ol[x] * rl * wl[x], dw);
      gs = fmaf(ws[x] * w * R[x], os[x], gs);
      gl = fmaf(wl[x] * (1.f - w) * R[x], ol[x], gl);
    }
    dw = warp_sum(dw);
    gs = warp_sum(gs);
    gl = warp_sum(gl);
    const float dz = dw * w * (1.f - w);
    float dl = 0.f, g_s[E], g_l[E], gq[E];
#pragma unroll
    for (int x = 0; x < E; ++x) {
      g_s[x] = rs * ws[x] * w * R[x] - os[x] * rs * rs * rs * gs / D;
      g_l[x] = rl * wl[x] * (1.f - w) * R[x] - ol[x] * rl * rl * rl * gl / D;
      gq[x] = dz * wg[x];
      dl = fmaf(g_s[x], os[x], dl);
      a_wg[x] = fmaf(dz, qv[x], a_wg[x]);
      a_ns[x] = fmaf(w * R[x], os[x] * rs, a_ns[x]);
      a_nl[x] = fmaf((1.f - w) * R[x], ol[x] * rl, a_nl[x]);
    }
    // d o_s in fp32 for the fp32 path, in bf16 for the tensor-core softmax backward
    if (d_os16)
      vec_store<E>(d_os16 + t * D + lane * E, g_s);
    else
      vec_store<E>(d_os + t * D + lane * E, g_s);
    vec_store<E>(d_ol + t * D + lane * E, g_l);
    vec_store<E>(dq + t * D + lane * E, gq);
    dl = warp_sum(dl);
    if (lane == 0) delta[t] = dl;
    a_bg += dz;
  }
  // weight gradients: the CTA's warps summed, then one atomic per element
#pragma unroll
  for (int x = 0; x < E; ++x) {
    red[warp][0][lane * E + x] = a_wg[x];
    red[warp][1][lane * E + x] = a_ns[x];
    red[warp][2][lane * E + x] = a_nl[x];
  }
  if (lane == 0) red_b[warp] = a_bg;
  __syncthreads();
  for (int f = threadIdx.x; f < 3 * D; f += blockDim.x) {
    const int which = f / D, c = f % D;
    float s = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s += red[w8][which][c];
    float* dst = which == 0 ? (dw_g ? dw_g + (long long)h * D : nullptr) : which == 1 ? dnws : dnwl;
    if (dst) atomicAdd(dst + c, s);
  }
  if (threadIdx.x == 0 && db_g) {
    float s = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s += red_b[w8];
    atomicAdd(db_g + h, s);
  }
}

// ---------------------------------------------------- 2. softmax branch
// The keys a query row t of chunk c sees: every key of the earlier chunks
// that chose softmax, then its own chunk up to t.  fn(j) for each, in order.
template <typename F>
__device__ __forceinline__ void for_each_key(const uint8_t* sel_h, int t, F&& fn) {
  const int c = t / kChunk;
  for (int cj = 0; cj < c; ++cj)
    if (sel_h[cj] == 0)
      for (int j = cj * kChunk; j < (cj + 1) * kChunk; ++j) fn(j);
  for (int j = c * kChunk; j <= t; ++j) fn(j);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) softmax_bwd_rows_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const uint8_t* __restrict__ sel,
    const float* __restrict__ d_os, const float* __restrict__ delta, long long rows, int L, int N, float scale,
    float* __restrict__ lse, float* __restrict__ dq) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + warp;
  if (row >= rows) return;  // warp-uniform
  const long long bh = row / L;
  const int t = (int)(row % L);
  const T* kh = k + bh * L * D;
  const T* vh = v + bh * L * D;
  const uint8_t* sel_h = sel + bh * N;
  float qv[E], dov[E];
  row_load<E>(q + row * D + lane * E, qv);
  row_load<E>(d_os + row * D + lane * E, dov);
  // pass 1: log-sum-exp of the row's scores
  float m = -INFINITY, s = 0.f;
  for_each_key(sel_h, t, [&](int j) {
    float kv[E];
    row_load<E>(kh + (long long)j * D + lane * E, kv);
    float p = 0.f;
#pragma unroll
    for (int x = 0; x < E; ++x) p = fmaf(qv[x], kv[x], p);
    const float sc = warp_sum(p) * scale;
    if (sc > m) {
      s = s * expf(m - sc) + 1.f;
      m = sc;
    } else {
      s += expf(sc - m);
    }
  });
  const float l = m + logf(s);
  const float dt = delta[row];
  // pass 2: dq_t = scale sum_j P_tj (do_t . v_j - delta_t) k_j
  float acc[E];
#pragma unroll
  for (int x = 0; x < E; ++x) acc[x] = 0.f;
  for_each_key(sel_h, t, [&](int j) {
    float kv[E], vv[E];
    row_load<E>(kh + (long long)j * D + lane * E, kv);
    row_load<E>(vh + (long long)j * D + lane * E, vv);
    float p = 0.f, dp = 0.f;
#pragma unroll
    for (int x = 0; x < E; ++x) {
      p = fmaf(qv[x], kv[x], p);
      dp = fmaf(dov[x], vv[x], dp);
    }
    const float P = expf(warp_sum(p) * scale - l);
    const float ds = P * (warp_sum(dp) - dt);
#pragma unroll
    for (int x = 0; x < E; ++x) acc[x] = fmaf(ds, kv[x], acc[x]);
  });
#pragma unroll
  for (int x = 0; x < E; ++x) dq[row * D + lane * E + x] += scale * acc[x];
  if (lane == 0) lse[row] = l;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) softmax_bwd_keys_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const uint8_t* __restrict__ sel,
    const float* __restrict__ d_os, const float* __restrict__ delta, const float* __restrict__ lse,
    long long rows, int L, int N, float scale, float* __restrict__ dk, float* __restrict__ dv) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + warp;
  if (row >= rows) return;  // warp-uniform
  const long long bh = row / L;
  const int j = (int)(row % L), cj = j / kChunk;
  const long long h0 = bh * L;
  float kv[E], vv[E];
  row_load<E>(k + row * D + lane * E, kv);
  row_load<E>(v + row * D + lane * E, vv);
  // the queries that see key j: the rest of its chunk, then every later
  // query if the chunk chose softmax
  const int t_end = sel[bh * N + cj] == 0 ? L : (cj + 1) * kChunk;
  float ak[E], av[E];
#pragma unroll
  for (int x = 0; x < E; ++x) ak[x] = av[x] = 0.f;
  for (int t = j; t < t_end; ++t) {
    float qv[E], dov[E];
    row_load<E>(q + (h0 + t) * D + lane * E, qv);
    row_load<E>(d_os + (h0 + t) * D + lane * E, dov);
    float p = 0.f, dp = 0.f;
#pragma unroll
    for (int x = 0; x < E; ++x) {
      p = fmaf(qv[x], kv[x], p);
      dp = fmaf(dov[x], vv[x], dp);
    }
    const float P = expf(warp_sum(p) * scale - lse[h0 + t]);
    const float ds = P * (warp_sum(dp) - delta[h0 + t]);
#pragma unroll
    for (int x = 0; x < E; ++x) {
      ak[x] = fmaf(ds, qv[x], ak[x]);
      av[x] = fmaf(P, dov[x], av[x]);
    }
  }
#pragma unroll
  for (int x = 0; x < E; ++x) {
    dk[row * D + lane * E + x] = scale * ak[x];
    dv[row * D + lane * E + x] = av[x];
  }
}

// --------------------------------------------------- 3. Gated DeltaNet
// The rows of the state are independent under the delta rule, so a head's
// d rows are split between kRowSplit CTAs of 512 threads.  Thread (warp w,
// lane l) holds rows [w RW, w RW + RW) of its CTA's half x columns
// [l CW, l CW + CW).  Column sums and scalars are per-half partials, added
// by gdn_bwd_combine_kernel.  Each token's vectors are read into registers
// two steps ahead, and in the reverse sweep each thread copies its elements
// of the state two tokens back into a three-slot shared-memory ring
// (cp.async), so global latency hides behind the arithmetic of two tokens.
constexpr int kGdnThreads = 512;
constexpr int kRowSplit = 2;

template <int D>
struct GdnBwd {
  static constexpr int RH = D / kRowSplit;  // rows per CTA
  static constexpr int RW = RH / 16;        // rows per warp
  static constexpr int CW = D / 32;         // columns per lane
  // a token's vectors: k, scale q, v and do of the CTA's rows, a, beta
  static constexpr int TOK = 2 * D + 2 * RH + 2;
  // shared memory (floats)
  static constexpr int offTok = 0;                    // [2][TOK]
  static constexpr int offU = offTok + 2 * TOK;       // [kChunk][RH] u_t of the replayed chunk
  static constexpr int offColA = offU + kChunk * RH;  // [16][D]
  static constexpr int offColB = offColA + 16 * D;    // [16][D]
  static constexpr int offRed = offColB + 16 * D;     // [16][3]
  static constexpr int offSt = offRed + 64;            // [3][RH][D] states before the coming tokens
  static constexpr int kFloats = offSt + 3 * RH * D;
  static constexpr int kBytes = kFloats * 4;
};

// asynchronous copy of `bytes` (8 or 16) global -> shared by this thread
template <int BYTES>
__device__ __forceinline__ void cp_async(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  if constexpr (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename T, int D>
__global__ void __launch_bounds__(kGdnThreads, 1) gdn_bwd_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, const uint8_t* __restrict__ sel, const float* __restrict__ d_ol, int L,
    int N, float scale, float* __restrict__ Sc, float* __restrict__ Tk, float* __restrict__ dSx,
    float* __restrict__ pcol, float* __restrict__ psc, float* __restrict__ dv) {
  using G = GdnBwd<D>;
  constexpr int RH = G::RH, RW = G::RW, CW = G::CW, TOK = G::TOK;
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long bh = blockIdx.x / kRowSplit;
  const int part = (int)(blockIdx.x % kRowSplit);
  const int row0 = part * RH;  // first state row of this CTA
  const long long h0 = bh * L;
  const uint8_t* sel_h = sel + bh * N;
  float* sc_h = Sc + bh * (long long)N * D * D;        // chunk-start states
  float* tk_h = Tk + bh * (long long)kChunk * D * D;   // states after each token of one chunk
  float* dsx_h = dSx + bh * (long long)D * D;
  // this half's partials: column sums [L][2 D] and scalars [L][4]
  float* pc = pcol + ((long long)part * (long long)(gridDim.x / kRowSplit) + bh) * L * 2 * D;
  float* ps = psc + ((long long)part * (long long)(gridDim.x / kRowSplit) + bh) * L * 4;
  const int r0 = warp * RW, c0 = lane * CW;  // within the half / the row
  auto el = [&](int i, int j) { return (long long)(row0 + r0 + i) * D + c0 + j; };
  auto ld = [&](const float* M, float (&X)[RW][CW]) {
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int j = 0; j < CW; ++j) X[i][j] = M[el(i, j)];
  };
  auto st = [&](float* M, const float (&X)[RW][CW]) {
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int j = 0; j < CW; ++j) M[el(i, j)] = X[i][j];
  };
  // this thread's element of token t's vectors (threads >= TOK: none)
  auto fetch = [&](int t) -> float {
    const long long r = h0 + t;
    if (tid < D) return to_f32(k[r * D + tid]);
    if (tid < 2 * D) return scale * to_f32(q[r * D + tid - D]);
    if (tid < 2 * D + RH) return to_f32(v[r * D + row0 + tid - 2 * D]);
    if (tid < 2 * D + 2 * RH) return d_ol[r * D + row0 + tid - 2 * D - RH];
    if (tid == 2 * D + 2 * RH) return expf(g[r]);
    if (tid == 2 * D + 2 * RH + 1) return beta[r];
    return 0.f;
  };
  auto tbuf = [&](int b) { return sm + G::offTok + b * TOK; };
  auto put = [&](int b, float x) {
    if (tid < TOK) tbuf(b)[tid] = x;
  };
  auto row_dot = [&](const float (&X)[RW][CW], const float* y, float (&out)[RW]) {
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      float p = 0.f;
#pragma unroll
      for (int j = 0; j < CW; ++j) p = fmaf(X[i][j], y[c0 + j], p);
      out[i] = warp_sum(p);
    }
  };
  // one forward token step on this half of S; u = S_{t-1} k of its rows
  auto fwd_step = [&](float (&S)[RW][CW], const float* tb, float (&u)[RW]) {
    const float* kt = tb;
    const float* vt = tb + 2 * D;
    const float a = tb[2 * D + 2 * RH], bt = tb[2 * D + 2 * RH + 1];
    row_dot(S, kt, u);
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const float coef = bt * (vt[r0 + i] - a * u[i]);
#pragma unroll
      for (int j = 0; j < CW; ++j) S[i][j] = fmaf(a, S[i][j], coef * kt[c0 + j]);
    }
  };

  // phase A: the chunk-start states
  int b = 0;
  {
    float S[RW][CW];
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int j = 0; j < CW; ++j) S[i][j] = 0.f;
    put(b, fetch(0));
    float pfa = L > 1 ? fetch(1) : 0.f;  // the next token's element, read a step ago
    __syncthreads();
    for (int t = 0; t < L; ++t) {
      const int c = t / kChunk;
      if (t % kChunk == 0) st(sc_h + (long long)c * D * D, S);
      const float pfb = t + 2 < L ? fetch(t + 2) : 0.f;
      float u[RW];
      fwd_step(S, tbuf(b), u);
      if (t % kChunk == kChunk - 1 && sel_h[c] == 0) ld(sc_h + (long long)c * D * D, S);  // rollback
      put(b ^ 1, pfa);
      pfa = pfb;
      __syncthreads();
      b ^= 1;
    }
  }

  // phase B: the adjoint, chunk by chunk from the last
  float dS[RW][CW];
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int j = 0; j < CW; ++j) dS[i][j] = 0.f;
  for (int c = N - 1; c >= 0; --c) {
    const int t0 = c * kChunk;
    const bool rolled_back = sel_h[c] == 0;
    float* sc_c = sc_h + (long long)c * D * D;
    // replay the chunk: the state after each token (but the last), and u_t
    {
      float S[RW][CW];
      ld(sc_c, S);
      put(b, fetch(t0));
      float pfa = fetch(t0 + 1);
      __syncthreads();
      for (int i = 0; i < kChunk; ++i) {
        const float pfb = i + 2 < kChunk ? fetch(t0 + i + 2) : 0.f;
        float u[RW];
        fwd_step(S, tbuf(b), u);
        if (lane == 0)
#pragma unroll
          for (int x = 0; x < RW; ++x) sm[G::offU + i * RH + r0 + x] = u[x];
        if (i + 1 < kChunk) st(tk_h + (long long)i * D * D, S);
        put(b ^ 1, pfa);
        pfa = pfb;
        __syncthreads();
        b ^= 1;
      }
    }
    // the gradient arriving at the state after the chunk: through the
    // tokens, or (rolled back) straight to the chunk start
    if (rolled_back) {
      st(dsx_h, dS);
#pragma unroll
      for (int i = 0; i < RW; ++i)
#pragma unroll
        for (int j = 0; j < CW; ++j) dS[i][j] = 0.f;
    }
    // the state before token i: after token i - 1, or the chunk start
    auto before = [&](int i) -> const float* { return i > 0 ? tk_h + (long long)(i - 1) * D * D : sc_c; };
    // this thread's elements of the state before token i, into ring slot i % 3
    auto stage = [&](int i) {
      const float* src = before(i);
      float* dst = sm + G::offSt + (i % 3) * RH * D;
#pragma unroll
      for (int x = 0; x < RW; ++x) cp_async<CW * 4>(dst + (r0 + x) * D + c0, src + el(x, 0));
    };
    stage(kChunk - 1);
    cp_async_commit();
    stage(kChunk - 2);
    cp_async_commit();
    put(b, fetch(t0 + kChunk - 1));
    float pfa = fetch(t0 + kChunk - 2);
    __syncthreads();
    for (int i = kChunk - 1; i >= 0; --i) {
      const int t = t0 + i;
      // two steps ahead: token i - 2's element and the state before it
      const float pfb = i >= 2 ? fetch(t - 2) : 0.f;
      if (i >= 2) stage(i - 2);
      cp_async_commit();
      cp_async_wait<2>();  // this thread's copy of the state before token i has landed
      float Sb[RW][CW];
      {
        const float* src = sm + G::offSt + (i % 3) * RH * D;
#pragma unroll
        for (int x = 0; x < RW; ++x)
#pragma unroll
          for (int j = 0; j < CW; ++j) Sb[x][j] = src[(r0 + x) * D + c0 + j];
      }
      const float* tb = tbuf(b);
      const float* kt = tb;
      const float* qt = tb + D;
      const float* vt = tb + 2 * D;
      const float* dot = tb + 2 * D + RH;
      const float a = tb[2 * D + 2 * RH], bt = tb[2 * D + 2 * RH + 1];
      // dS_t += do_t (scale q_t)^T; S_{t-1}^T do_t (column sums)
      float colA[CW], colB[CW];
#pragma unroll
      for (int j = 0; j < CW; ++j) colA[j] = colB[j] = 0.f;
#pragma unroll
      for (int x = 0; x < RW; ++x) {
        const float dor = dot[r0 + x];
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          dS[x][j] = fmaf(dor, qt[c0 + j], dS[x][j]);
          colA[j] = fmaf(Sb[x][j], dor, colA[j]);
        }
      }
      float xr[RW];
      row_dot(dS, kt, xr);
      float p_da = 0.f, p_db = 0.f, p_ed = 0.f;
#pragma unroll
      for (int x = 0; x < RW; ++x) {
        const float u = sm[G::offU + i * RH + r0 + x];
        const float e = vt[r0 + x] - a * u;
        const float de = bt * xr[x];
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          colB[j] = fmaf(bt * e, dS[x][j], colB[j]);
          colB[j] = fmaf(-a * de, Sb[x][j], colB[j]);
          p_da = fmaf(dS[x][j], Sb[x][j], p_da);
        }
        if (lane == 0) {
          p_da -= u * de;
          p_db = fmaf(e, xr[x], p_db);
          p_ed = fmaf(e, dot[r0 + x], p_ed);
          dv[(h0 + t) * D + row0 + r0 + x] += de;
        }
        // dS_{t-1} = a dS_t - a de k^T
#pragma unroll
        for (int j = 0; j < CW; ++j) dS[x][j] = a * fmaf(-de, kt[c0 + j], dS[x][j]);
      }
      p_da = warp_sum(p_da);
#pragma unroll
      for (int j = 0; j < CW; ++j) {
        sm[G::offColA + warp * D + c0 + j] = colA[j];
        sm[G::offColB + warp * D + c0 + j] = colB[j];
      }
      if (lane == 0) {
        sm[G::offRed + 3 * warp] = p_da;
        sm[G::offRed + 3 * warp + 1] = p_db;
        sm[G::offRed + 3 * warp + 2] = p_ed;
      }
      __syncthreads();
      // this half's partials of token t
      if (tid < 2 * D) {
        const int off = tid < D ? G::offColA + tid : G::offColB + tid - D;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) sum += sm[off + w * D];
        pc[(long long)t * 2 * D + tid] = sum;
      } else if (tid < 2 * D + 3) {
        const int which = tid - 2 * D;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) sum += sm[G::offRed + 3 * w + which];
        ps[(long long)t * 4 + which] = sum;
      }
      put(b ^ 1, pfa);
      pfa = pfb;
      __syncthreads();
      b ^= 1;
    }
    if (rolled_back) {
      float X[RW][CW];
      ld(dsx_h, X);
#pragma unroll
      for (int i = 0; i < RW; ++i)
#pragma unroll
        for (int j = 0; j < CW; ++j) dS[i][j] += X[i][j];
    }
  }
}

// The halves' partials of each token combined: S_t^T do_t = a S_{t-1}^T do_t
// + beta <e, do_t> k_t gives dq, the column sums of dk add up, and
// dg = a da, dbeta.  One warp per token.
template <typename T, int D>
__global__ void __launch_bounds__(256) gdn_bwd_combine_kernel(
    const T* __restrict__ k, const float* __restrict__ g, const float* __restrict__ beta,
    const float* __restrict__ pcol, const float* __restrict__ psc, long long rows, float scale,
    float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dg, float* __restrict__ dbeta) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * 8 + warp;
  if (r >= rows) return;  // warp-uniform
  const float a = expf(g[r]), bt = beta[r];
  float da = 0.f, db = 0.f, ed = 0.f;
#pragma unroll
  for (int h = 0; h < kRowSplit; ++h) {
    const float* s4 = psc + ((long long)h * rows + r) * 4;
    da += s4[0];
    db += s4[1];
    ed += s4[2];
  }
  float kv[E];
  row_load<E>(k + r * D + lane * E, kv);
#pragma unroll
  for (int x = 0; x < E; ++x) {
    const int f = lane * E + x;
    float ca = 0.f, cb = 0.f;
#pragma unroll
    for (int h = 0; h < kRowSplit; ++h) {
      const float* pr = pcol + ((long long)h * rows + r) * 2 * D;
      ca += pr[f];
      cb += pr[D + f];
    }
    dq[r * D + f] += scale * fmaf(a, ca, bt * ed * kv[x]);
    dk[r * D + f] += cb;
  }
  if (lane == 0) {
    dg[r] = a * da;
    dbeta[r] = db;
  }
}

}  // namespace

// The backward workspace, carved in one order for the size query and the
// launch (base == nullptr: sizes only).
struct BwdLayout {
  float *d_os, *d_ol, *delta, *lse;
  __nv_bfloat16* d_os16;
  // fp32 layers: the token-serial adjoint
  float *Sc, *Tk, *dSx, *pcol, *psc;
  // bf16 layers: the forward recompute of the chunk-start states, then the
  // chunkwise adjoint
  int32_t *nprev, *sel_idx;
  float *fG, *fgate;
  void *fW, *fU, *fP, *fol16;
  int* ferr;
  GdnBwdScratch cw;
};

static size_t bwd_layout(const Problem& p, int dtype, uint8_t* base, BwdLayout* o) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* ptr = base ? base + off : nullptr;
    off += (bytes + 255) & ~(size_t)255;
    return ptr;
  };
  const size_t rows = (size_t)p.BH * p.L, dd = (size_t)p.d * p.d, chunks = (size_t)p.BH * p.N;
  BwdLayout l{};
  if (dtype != 0)
    l.d_os = (float*)take(rows * p.d * 4);             // d o_s
  else
    l.d_os16 = (__nv_bfloat16*)take(rows * p.d * 2);   // d o_s in bf16 (the operand of the tensor-core products)
  l.d_ol = (float*)take(rows * p.d * 4);               // d o_l
  l.delta = (float*)take(rows * 4);
  l.lse = (float*)take(rows * 4);
  if (dtype != 0) {
    l.Sc = (float*)take(chunks * dd * 4);                       // chunk-start states
    l.Tk = (float*)take((size_t)p.BH * kChunk * dd * 4);        // states inside the chunk being reversed
    l.dSx = (float*)take((size_t)p.BH * dd * 4);                // gradient held over a rolled-back chunk
    l.pcol = (float*)take((size_t)kRowSplit * rows * 2 * p.d * 4);  // the state halves' column sums per token
    l.psc = (float*)take((size_t)kRowSplit * rows * 4 * 4);     // and their scalars
  } else {
    l.nprev = (int32_t*)take(chunks * 4);    // compacted softmax-chunk lists
    l.sel_idx = (int32_t*)take(chunks * 4);
    l.fG = (float*)take(rows * 4);        // forward chunk factors (recomputed)
    l.fW = take(rows * p.d * 2);
    l.fU = take(rows * p.d * 2);
    l.fP = take(rows * kChunk * 2);
    l.fgate = (float*)take(rows * 4);
    l.fol16 = take(rows * p.d * 2);       // the recompute's o_l (not used)
    l.ferr = (int*)take(16);
    GdnBwdScratch& w = l.cw;
    w.S0 = (float*)take(chunks * dd * 4);
    w.dSC = (float*)take(chunks * dd * 4);
    w.G = (float*)take(rows * 4);
    w.Li = (float*)take(rows * kChunk * 4);
    w.P = (float*)take(rows * kChunk * 4);
    w.W16 = take(rows * p.d * 2);
    w.Qe16 = take(rows * p.d * 2);
    w.Kt16 = take(rows * p.d * 2);
    w.sc = (float*)take(chunks * 4 * 4);
  }
  if (o) *o = l;
  return off;
}

size_t bwd_workspace_bytes(const Problem& p, int dtype) { return bwd_layout(p, dtype, nullptr, nullptr); }

cudaError_t launch_hybrid_bwd(const Problem& p, int dtype, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* w_g, const float* b_g,
                              const float* nws, const float* nwl, const uint8_t* sel, const float* o_s,
                              const float* o_l, const void* dout, float* dq, float* dk, float* dv, float* dg,
                              float* dbeta, float* dw_g, float* db_g, float* dnws, float* dnwl, void* ws,
                              cudaStream_t st, void* const* ev_start, void* const* ev_stop, int32_t* launches,
                              cudaStream_t side, cudaEvent_t fork, cudaEvent_t join, const float* lse_in) {
  if (p.BH == 0 || p.L == 0) return cudaSuccess;
  auto mark_on = [&](void* const* ev, int s, cudaStream_t on) -> cudaError_t {
    return (ev && ev[s]) ? cudaEventRecord((cudaEvent_t)ev[s], on) : cudaSuccess;
  };
  auto mark = [&](void* const* ev, int s) -> cudaError_t { return mark_on(ev, s, st); };
  auto count = [&](int s, int n) {
    if (launches) launches[s] += n;
  };
  const long long rows = (long long)p.BH * p.L;
  BwdLayout lay;
  bwd_layout(p, dtype, (uint8_t*)ws, &lay);
  float* d_os = lay.d_os;
  float* d_ol = lay.d_ol;
  __nv_bfloat16* d_os16 = lay.d_os16;
  float* delta = lay.delta;
  float* lse = lay.lse;
  float* Sc = lay.Sc;
  float* Tk = lay.Tk;
  float* dSx = lay.dSx;
  float* pcol = lay.pcol;
  float* psc = lay.psc;
  // weight gradients are sums over the launch: zeroed first
  cudaError_t e = cudaSuccess;
  if (dw_g) e = cudaMemsetAsync(dw_g, 0, (size_t)p.H * p.d * 4, st);
  if (e == cudaSuccess && db_g) e = cudaMemsetAsync(db_g, 0, (size_t)p.H * 4, st);
  if (e == cudaSuccess && dnws) e = cudaMemsetAsync(dnws, 0, (size_t)p.d * 4, st);
  if (e == cudaSuccess && dnwl) e = cudaMemsetAsync(dnwl, 0, (size_t)p.d * 4, st);
  if (e == cudaSuccess && lay.ferr) e = cudaMemsetAsync(lay.ferr, 0, 16, st);  // bounded-wait flag of the tcgen05 kernels
  if (e != cudaSuccess) return e;
  auto run = [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    const T* qt = (const T*)q;
    const T* kt = (const T*)k;
    const T* vt = (const T*)v;
    constexpr bool tc = std::is_same<T, __nv_bfloat16>::value;  // bf16: the softmax branch on tensor cores
    // bf16 layers with a second stream: the chunk-start states' recompute
    // and the adjoint's chunk factors need only the inputs and the selection
    // and write only scratch, so they start on the second stream before the
    // merge stage; the reverse scan (it reads d o_l) waits for the merge.
    // That stream's work is the longer of the two branches', and the softmax
    // branch's CTAs fill the SMs its scans (chains over the chunks: 1 and 2
    // CTAs per head) leave idle.
    const bool two = tc && side && side != st && fork && join;
    const cudaStream_t ss = two ? side : st;
    auto state_work = [&]() -> cudaError_t {
      cudaError_t e3 = mark_on(ev_start, NATS_BWD_STAGE_GDN, ss);
      if constexpr (tc) {
        // the chunk-start states, from the forward's chunk factors and scan
        // (the same kernels as the forward; the selection is given), and
        // every chunk's Linv = (I + diag(beta) A)^{-1} in fp32 on the way
        if (e3 == cudaSuccess)
          e3 = D == 128 ? launch_gdn_prep_tc(p, q, k, v, g, beta, w_g, b_g, lay.fG, lay.fW, lay.fU, lay.fP,
                                             lay.fgate, nullptr, nullptr, nullptr, lay.ferr, lay.cw.Li, ss)
                        : launch_gdn_prep_mma(p, q, k, v, g, beta, w_g, b_g, lay.fG, lay.fW, lay.fU, lay.fP,
                                              lay.fgate, nullptr, nullptr, nullptr, lay.cw.Li, ss);
        if (e3 == cudaSuccess)
          e3 = launch_gdn_scan_tc(p, q, k, sel, lay.fG, lay.fW, lay.fU, lay.fP, nullptr, lay.fol16, nullptr,
                                  lay.ferr, ss, lay.cw.S0);
        // the adjoint's chunk factors
        if (e3 == cudaSuccess) e3 = launch_gdn_bwd_factors(p, q, k, g, beta, lay.cw, ss);
        if (e3 == cudaSuccess) count(NATS_BWD_STAGE_GDN, 3);
      }
      return e3;
    };
    cudaError_t e2 = cudaSuccess;
    if (two && ((e2 = cudaEventRecord(fork, st)) != cudaSuccess || (e2 = cudaStreamWaitEvent(ss, fork, 0)) != cudaSuccess ||
                (e2 = state_work()) != cudaSuccess))
      return e2;
    if ((e2 = mark(ev_start, NATS_BWD_STAGE_MERGE)) != cudaSuccess) return e2;
    merge_bwd_kernel<T, D><<<(unsigned)(rows / kMergeRows), 256, 0, st>>>(
        qt, (const T*)dout, o_s, o_l, w_g, b_g, nws, nwl, p.H, p.L, p.eps, d_os, tc ? d_os16 : nullptr, d_ol,
        delta, dq, dw_g, db_g, dnws, dnwl);
    count(NATS_BWD_STAGE_MERGE, 1);
    if ((e2 = mark(ev_stop, NATS_BWD_STAGE_MERGE)) != cudaSuccess) return e2;
    if constexpr (tc) {
      auto softmax_stage = [&]() -> cudaError_t {
        cudaError_t e3 = mark(ev_start, NATS_BWD_STAGE_SOFTMAX);
        if (e3 == cudaSuccess) e3 = launch_compact(p, sel, lay.nprev, lay.sel_idx, nullptr, st);
        if (e3 == cudaSuccess)
          e3 = launch_softmax_bwd_tc(p, q, k, v, d_os16, delta, lay.nprev, lay.sel_idx, sel, lse, lse_in, dq, dk,
                                     dv, lay.ferr, st);
        if (e3 != cudaSuccess) return e3;
        count(NATS_BWD_STAGE_SOFTMAX, 4);  // compaction, query tiles, local and retained key tiles
        return mark(ev_stop, NATS_BWD_STAGE_SOFTMAX);
      };
      auto reverse_scan = [&]() -> cudaError_t {
        cudaError_t e3 = launch_gdn_bwd_reverse_scan(p, sel, d_ol, lay.cw, ss);
        if (e3 != cudaSuccess) return e3;
        count(NATS_BWD_STAGE_GDN, 1);
        return mark_on(ev_stop, NATS_BWD_STAGE_GDN, ss);
      };
      if (two) {
        // the reverse scan after the merge (the fork event is recorded again:
        // a wait takes the event's latest record)
        if ((e2 = cudaEventRecord(fork, st)) != cudaSuccess || (e2 = cudaStreamWaitEvent(ss, fork, 0)) != cudaSuccess ||
            (e2 = reverse_scan()) != cudaSuccess || (e2 = softmax_stage()) != cudaSuccess ||
            (e2 = cudaEventRecord(join, ss)) != cudaSuccess || (e2 = cudaStreamWaitEvent(st, join, 0)) != cudaSuccess)
          return e2;
      } else if ((e2 = softmax_stage()) != cudaSuccess || (e2 = state_work()) != cudaSuccess ||
                 (e2 = reverse_scan()) != cudaSuccess) {
        return e2;
      }
      // every per-chunk product of the adjoint: dq, dk, dv, dg, dbeta
      if ((e2 = mark(ev_start, NATS_BWD_STAGE_COMBINE)) != cudaSuccess) return e2;
      if ((e2 = launch_gdn_bwd_products(p, q, k, v, g, beta, sel, d_ol, lay.cw, dq, dk, dv, dg, dbeta, lay.ferr,
                                        st)) != cudaSuccess)
        return e2;
      count(NATS_BWD_STAGE_COMBINE, 1);
    } else {
      if ((e2 = mark(ev_start, NATS_BWD_STAGE_SOFTMAX)) != cudaSuccess) return e2;
      softmax_bwd_rows_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(qt, kt, vt, sel, d_os, delta,
                                                                               rows, p.L, p.N, p.scale, lse, dq);
      softmax_bwd_keys_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(
          qt, kt, vt, sel, d_os, delta, lse, rows, p.L, p.N, p.scale, dk, dv);
      count(NATS_BWD_STAGE_SOFTMAX, 2);
      if ((e2 = mark(ev_stop, NATS_BWD_STAGE_SOFTMAX)) != cudaSuccess) return e2;
      if ((e2 = mark(ev_start, NATS_BWD_STAGE_GDN)) != cudaSuccess) return e2;
      constexpr int smem = GdnBwd<D>::kBytes;
      static const cudaError_t attr =
          cudaFuncSetAttribute(gdn_bwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (attr != cudaSuccess) return attr;
      gdn_bwd_kernel<T, D><<<(unsigned)(p.BH * kRowSplit), kGdnThreads, smem, st>>>(
          qt, kt, vt, g, beta, sel, d_ol, p.L, p.N, p.scale, Sc, Tk, dSx, pcol, psc, dv);
      count(NATS_BWD_STAGE_GDN, 1);
      if ((e2 = mark(ev_stop, NATS_BWD_STAGE_GDN)) != cudaSuccess) return e2;
      if ((e2 = mark(ev_start, NATS_BWD_STAGE_COMBINE)) != cudaSuccess) return e2;
      gdn_bwd_combine_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(kt, g, beta, pcol, psc, rows,
                                                                              p.scale, dq, dk, dg, dbeta);
      count(NATS_BWD_STAGE_COMBINE, 1);
    }
    if ((e2 = mark(ev_stop, NATS_BWD_STAGE_COMBINE)) != cudaSuccess) return e2;
    return cudaGetLastError();
  };
  using bf = __nv_bfloat16;
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (dtype == 0) return p.d == 64 ? run(bf(), D64()) : run(bf(), D128());
  return p.d == 64 ? run(0.f, D64()) : run(0.f, D128());
}

}  // namespace nats
