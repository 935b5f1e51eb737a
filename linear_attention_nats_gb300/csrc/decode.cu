// decode.cu - the NAtS-L layer in decode mode: one new token per (b, h) per
// launch ("Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" items 1, 3 and 4, read token by token).
//
// A cluster of kSplit CTAs of 128 threads per (b, h), sharing the head's
// work, so that a step is one wave of small CTAs over the whole GPU (four
// per SM):
//   1. the token's q, k, v to shared memory (every CTA); CTA 0 appends k, v
//      to the chunk's keys / values at position p = t % chunk.  The
//      CTA's state rows are requested first, then thread 0 starts the copies
//      of the CTA's keys (below);
//   2. softmax over the keys held in memory (the retained keys of earlier
//      softmax chunks, then the chunk's keys before the token) in blocks of
//      32, which the cluster's CTAs claim one at a time from a counter in
//      CTA 0's shared memory (distributed shared memory atomics), so that a
//      CTA whose copies land sooner takes more of them: one thread copies a
//      claimed block's key and value rows (contiguous runs) into a ring of
//      shared-memory stages with bulk async copies, up to three stages in
//      flight, completing on an mbarrier; each warp scores eight rows of a
//      stage, lanes over the d
//      features, the eight dot products summed over the warp by halving
//      (nine shuffles), online softmax, P V.  The token itself (the last
//      key) is scored by one warp of the last CTA from shared memory;
//   3. Gated DeltaNet on the CTA's d / kSplit rows of the fp32 state (read
//      before the key copies are issued, updated after the keys):
//      S <- a S (I - beta k k^T) + beta v k^T, i.e. row i of S becomes
//      a S_i + beta (v_i - a S_i . k) k^T, and o_l = S (scale q); the rows of
//      o_l go to CTA 0's shared memory (distributed shared memory), and so
//      does the CTA's softmax (max, sum, partial output), before a cluster
//      barrier; the new rows are stored after it;
//   4. CTA 0: the kSplit partials combined, RMSNorm of both branches and the
//      query-gated sum; the running [q; k] sum of the chunk;
//   5. when the token completes the chunk: every CTA computes the chunk's
//      score and selection (the same arithmetic, so the same result) and
//      applies it to its own state rows and its share of the chunk's keys
//      and values: softmax appends them to the retained ones and restores
//      the state to the chunk start, Gated DeltaNet keeps the state as the
//      new chunk start.
// Every wait is bounded: a copy that does not land in time sets *err and
// the step finishes without it.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kSplit = 8;                  // CTAs per (b, h): a thread-block cluster
constexpr int kKeysPerStage = 8 * kWarps;  // eight rows per warp and stage

// The ring of key / value stages in dynamic shared memory.
template <typename T, int D>
struct Ring {
  static constexpr int kRow = D * (int)sizeof(T);        // bytes of one key (value) row
  static constexpr int kHalf = kKeysPerStage * kRow;     // the key rows of a stage
  static constexpr int kStage = 2 * kHalf;               // then its value rows
  static constexpr int kStages = kStage <= 16384 ? 3 : 2;
  static constexpr int kBytes = kStages * kStage;
};

template <int N>
__device__ __forceinline__ void load_n(const float* p, float (&o)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 v = *(const float4*)(p + i);
    o[i] = v.x, o[i + 1] = v.y, o[i + 2] = v.z, o[i + 3] = v.w;
  }
}
template <int N>
__device__ __forceinline__ void load_n(const __nv_bfloat16* p, float (&o)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 8) {
    const uint4 u = *(const uint4*)(p + i);
    const __nv_bfloat162* h2 = (const __nv_bfloat162*)&u;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 f = __bfloat1622float2(h2[x]);
      o[i + 2 * x] = f.x, o[i + 2 * x + 1] = f.y;
    }
  }
}
// E (2 or 4) consecutive elements
template <int E>
__device__ __forceinline__ void load_e(const float* p, float (&o)[E]) {
#pragma unroll
  for (int x = 0; x < E; ++x) o[x] = p[x];
}
template <int E>
__device__ __forceinline__ void load_e(const __nv_bfloat16* p, float (&o)[E]) {
#pragma unroll
  for (int x = 0; x < E; ++x) o[x] = __bfloat162float(p[x]);
}

// E consecutive elements kept in their storage form (the rows of a batch in
// flight), converted when used
template <typename T, int E>
struct Raw;
template <>
struct Raw<__nv_bfloat16, 4> {
  uint2 r;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { r = *(const uint2*)p; }
  __device__ __forceinline__ void zero() { r = make_uint2(0, 0); }
  __device__ __forceinline__ void get(float (&o)[4]) const {
    o[0] = __uint_as_float(r.x << 16), o[1] = __uint_as_float(r.x & 0xffff0000u);
    o[2] = __uint_as_float(r.y << 16), o[3] = __uint_as_float(r.y & 0xffff0000u);
  }
};
template <>
struct Raw<__nv_bfloat16, 2> {
  uint32_t r;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { r = *(const uint32_t*)p; }
  __device__ __forceinline__ void zero() { r = 0; }
  __device__ __forceinline__ void get(float (&o)[2]) const {
    o[0] = __uint_as_float(r << 16), o[1] = __uint_as_float(r & 0xffff0000u);
  }
};
template <>
struct Raw<float, 4> {
  float4 r;
  __device__ __forceinline__ void load(const float* p) { r = *(const float4*)p; }
  __device__ __forceinline__ void zero() { r = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&o)[4]) const { o[0] = r.x, o[1] = r.y, o[2] = r.z, o[3] = r.w; }
};
template <>
struct Raw<float, 2> {
  float2 r;
  __device__ __forceinline__ void load(const float* p) { r = *(const float2*)p; }
  __device__ __forceinline__ void zero() { r = make_float2(0.f, 0.f); }
  __device__ __forceinline__ void get(float (&o)[2]) const { o[0] = r.x, o[1] = r.y; }
};

// sums of three per-thread values over the CTA (every thread gets them)
__device__ __forceinline__ void block_sum3(float& a, float& b, float& c, float (*red)[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  c = warp_sum(c);
  if (lane == 0) red[warp][0] = a, red[warp][1] = b, red[warp][2] = c;
  __syncthreads();
  a = b = c = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) a += red[w][0], b += red[w][1], c += red[w][2];
  __syncthreads();
}

// programmatic dependent launch: let the next kernel of the stream be
// scheduled now; wait for the previous one to complete (its writes visible)
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T, int D>
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads, 4) decode_step_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, const float* __restrict__ w_s, const float* __restrict__ b_s,
    const float* __restrict__ w_g, const float* __restrict__ b_g, const float* __restrict__ nw_s,
    const float* __restrict__ nw_l, int H, int C, int p, float scale, float eps, float* __restrict__ S,
    float* __restrict__ S0, T* __restrict__ ck, T* __restrict__ cv, float* __restrict__ psum,
    T* __restrict__ kv_k, T* __restrict__ kv_v, int32_t* __restrict__ n_kv, long long cap, T* __restrict__ out,
    uint8_t* __restrict__ sel_out, float* __restrict__ o_s_out, float* __restrict__ o_l_out, int* err) {
  static_assert(D % 32 == 0 && D <= 128 && D % kSplit == 0, "shape");
  using R = Ring<T, D>;
  constexpr int RPC = D / kSplit;       // state rows per CTA
  constexpr int TPR = kThreads / RPC;   // threads per state row
  constexpr int CPT = D / TPR;          // state columns per thread
  constexpr int E = D / 32;             // features per lane in the softmax
  static_assert(TPR <= 32 && CPT % 4 == 0, "state split");
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long bh = blockIdx.x / kSplit;
  const int h = (int)(bh % H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[R::kStages];
  __shared__ __align__(16) float qs[D], ks[D], vs[D], os[D], ol[D];
  __shared__ float wm[kWarps], wl[kWarps];
  __shared__ float red[kWarps][3];
  __shared__ __align__(16) float part_o[kSplit][D];  // CTA 0: the cluster's partial outputs
  __shared__ float part_m[kSplit], part_l[kSplit];
  __shared__ int sel_sh;
  __shared__ int claim;            // CTA 0's: the next block of 32 keys to hand out
  __shared__ int blk[R::kStages];  // the block in each slot (-1: none was left)

  if (tid == 0) {
    for (int i = 0; i < R::kStages; ++i) tc::mbar_init(&full[i], 1);
    tc::fence_barrier_init();
    claim = 0;
  }
  launch_dependents();
  cluster.sync();  // CTA 0's counter is set and every CTA of the cluster runs
  // nothing before this point reads global memory: every input, the state
  // included, may be written by the preceding kernel of the stream
  wait_prerequisites();

  // this CTA's state rows, read first (used after the keys, by which time
  // they have long arrived; read after the copies they would queue behind
  // them)
  const int srow_i = rank * RPC + tid / TPR, spart = tid % TPR;
  float* srow = S + (bh * D + srow_i) * D + spart * CPT;
  float sv[CPT];
  load_n<CPT>(srow, sv);

  // the hi = nr + p keys held in memory, nr retained then p of the chunk,
  // in blocks of 32 that the cluster's CTAs claim one at a time from CTA 0's
  // counter (a CTA whose copies land sooner takes more blocks)
  const int nr = n_kv[bh];
  const int hi = nr + p;
  const int nblk = (hi + kKeysPerStage - 1) / kKeysPerStage;
  int* claim0 = cluster.map_shared_rank(&claim, 0);
  const T* Kr = kv_k + bh * cap * D;
  const T* Vr = kv_v + bh * cap * D;
  const T* Kc = ck + bh * C * D;
  const T* Vc = cv + bh * C * D;
  // stage s: a claimed block into slot s % kStages (the retained rows and the
  // chunk's rows are two contiguous runs); false when none was left, the
  // slot then completes with no copy and blk = -1 ends the CTA's loop
  auto issue = [&](int s) -> bool {
    const int slot = s % R::kStages;
    uint8_t* kb = ring + slot * R::kStage;
    uint8_t* vb = kb + R::kHalf;
    uint64_t* bar = &full[slot];
    const int b = atomicAdd(claim0, 1);
    if (b >= nblk) {
      blk[slot] = -1;
      tc::mbar_arrive(bar);
      return false;
    }
    blk[slot] = b;
    const int a0 = b * kKeysPerStage, a1 = min(a0 + kKeysPerStage, hi);
    const int m = min(max(nr, a0), a1);  // [a0, m) retained, [m, a1) of the chunk
    tc::mbar_arrive_expect_tx(bar, (uint32_t)((a1 - a0) * 2 * R::kRow));
    if (m > a0) {
      tc::bulk_load_1d(kb, Kr + (long long)a0 * D, (uint32_t)((m - a0) * R::kRow), bar);
      tc::bulk_load_1d(vb, Vr + (long long)a0 * D, (uint32_t)((m - a0) * R::kRow), bar);
    }
    if (a1 > m) {
      tc::bulk_load_1d(kb + (m - a0) * R::kRow, Kc + (long long)(m - nr) * D, (uint32_t)((a1 - m) * R::kRow), bar);
      tc::bulk_load_1d(vb + (m - a0) * R::kRow, Vc + (long long)(m - nr) * D, (uint32_t)((a1 - m) * R::kRow), bar);
    }
    return true;
  };
  int issued = 0;    // stages issued (thread 0)
  bool more = true;  // blocks may be left (thread 0)
  if (tid == 0)
    for (; issued < R::kStages && more; ++issued) more = issue(issued);

  // 1. the token
  if (tid < D) {
    const T kt = k[bh * D + tid], vt = v[bh * D + tid];
    qs[tid] = to_f32(q[bh * D + tid]);
    ks[tid] = to_f32(kt);
    vs[tid] = to_f32(vt);
    if (rank == 0) {
      ck[(bh * C + p) * D + tid] = kt;
      cv[(bh * C + p) * D + tid] = vt;
    }
  }
  const float a = __expf(g[bh]), bt = beta[bh];
  // operands of the epilogue and of the chunk's selection, read now so that
  // no global load follows the cluster barrier
  constexpr int PE = (2 * D + kThreads - 1) / kThreads;  // running-sum entries per thread
  const bool last = p == C - 1;
  float psv[PE], ws0[PE], ws1[PE];
#pragma unroll
  for (int i = 0; i < PE; ++i) {
    const int e = tid + i * kThreads;
    psv[i] = ws0[i] = ws1[i] = 0.f;
    if (e < 2 * D && (rank == 0 || last)) psv[i] = psum[bh * 2 * D + e];
    if (e < 2 * D && last) {
      ws0[i] = w_s[((long long)h * 2 + 0) * 2 * D + e];
      ws1[i] = w_s[((long long)h * 2 + 1) * 2 * D + e];
    }
  }
  float wg = 0.f, nws = 1.f, nwl = 1.f, bg = 0.f;
  if (rank == 0 && tid < D) {
    wg = w_g[(long long)h * D + tid];
    if (nw_s) nws = nw_s[tid];
    if (nw_l) nwl = nw_l[tid];
    if (b_g) bg = b_g[h];
  }
  __syncthreads();  // also: the barriers are initialised

  // 2. softmax over the CTA's keys
  float qv[E];
#pragma unroll
  for (int x = 0; x < E; ++x) qv[x] = qs[lane * E + x];
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int x = 0; x < E; ++x) acc[x] = 0.f;
  using RV = Raw<T, E>;
  // the 8 keys from j0 (valid below hi): scores (partial dot products summed
  // over the warp by halving: lane (b4 b3 b2 . .) ends with key 4 b4 + 2 b3 +
  // b2), online softmax, P V
  auto batch = [&](int j0, const RV (&kb)[8], const RV (&vb)[8]) {
    float dp[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float kk[E];
      kb[u].get(kk);
      dp[u] = 0.f;
#pragma unroll
      for (int x = 0; x < E; ++x) dp[u] = fmaf(qv[x], kk[x], dp[u]);
    }
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float d4[4], d2[2];
#pragma unroll
    for (int u = 0; u < 4; ++u) d4[u] = (b4 ? dp[4 + u] : dp[u]) + __shfl_xor_sync(0xffffffffu, b4 ? dp[u] : dp[4 + u], 16);
#pragma unroll
    for (int u = 0; u < 2; ++u) d2[u] = (b3 ? d4[2 + u] : d4[u]) + __shfl_xor_sync(0xffffffffu, b3 ? d4[u] : d4[2 + u], 8);
    float d1 = (b2 ? d2[1] : d2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? d2[0] : d2[1], 4);
    d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
    d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
    const int ku = 4 * (lane >> 4) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
    const float sc = (j0 + ku < hi) ? d1 * scale : -INFINITY;
    float mb = sc;
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
    const float mn = fmaxf(m, mb);
    const float alpha = __expf(m - mn);  // 0 on the first batch (m = -inf)
    const float pu = (j0 + ku < hi) ? __expf(sc - mn) : 0.f;
    float ps = pu;
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int x = 0; x < E; ++x) acc[x] *= alpha;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float pw = __shfl_sync(0xffffffffu, pu, ((u >> 2) << 4) | (((u >> 1) & 1) << 3) | ((u & 1) << 2));
      float vv[E];
      vb[u].get(vv);
#pragma unroll
      for (int x = 0; x < E; ++x) acc[x] = fmaf(pw, vv[x], acc[x]);
    }
  };
  bool ok = true;
  int s = 0;
  for (;; ++s) {
    const int slot = s % R::kStages;
    const bool wok = __all_sync(0xffffffffu, tc::mbar_wait(&full[slot], (uint32_t)((s / R::kStages) & 1), err));
    const int b = wok ? blk[slot] : -1;  // written by thread 0 before the slot's arrival
    if (b >= 0 && b * kKeysPerStage + 8 * warp < hi) {
      const uint8_t* kb = ring + slot * R::kStage + 8 * warp * R::kRow;
      const uint8_t* vb = kb + R::kHalf;
      const int j0 = b * kKeysPerStage + 8 * warp;
      RV kr[8], vr[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < hi) {
          kr[u].load((const T*)(kb + u * R::kRow) + lane * E);
          vr[u].load((const T*)(vb + u * R::kRow) + lane * E);
        } else {
          kr[u].zero();
          vr[u].zero();
        }
      }
      batch(j0, kr, vr);
    }
    ok = __syncthreads_and(wok) != 0;  // the slot is read by every warp
    if (!ok || b < 0) break;
    if (tid == 0 && more) more = issue(issued++);
  }
  if (!ok && tid == 0) {
    // a copy did not land in time: wait (bounded) for those still in flight
    // into this CTA's shared memory before it is released
    for (int i = s; i < issued; ++i)
      tc::mbar_wait(&full[i % R::kStages], (uint32_t)((i / R::kStages) & 1), err);
  }
  // the token (the last key), from shared memory
  if (rank == kSplit - 1 && warp == 0) {
    float dp = 0.f;
#pragma unroll
    for (int x = 0; x < E; ++x) dp = fmaf(qv[x], ks[lane * E + x], dp);
    const float sc = warp_sum(dp) * scale;
    const float mn = fmaxf(m, sc);
    const float alpha = __expf(m - mn), pw = __expf(sc - mn);
    l = l * alpha + pw;
    m = mn;
#pragma unroll
    for (int x = 0; x < E; ++x) acc[x] = fmaf(pw, vs[lane * E + x], acc[x] * alpha);
  }

  // 3. Gated DeltaNet on this CTA's state rows
  {
    float u = 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) u = fmaf(sv[j], ks[spart * CPT + j], u);
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
    const float coef = bt * (vs[srow_i] - a * u);
    float r = 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      sv[j] = fmaf(a, sv[j], coef * ks[spart * CPT + j]);
      r = fmaf(sv[j], qs[spart * CPT + j], r);
    }
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (spart == 0) *cluster.map_shared_rank(&ol[srow_i], 0) = r * scale;
  }
  __syncthreads();  // the ring is free: the warps' partials go there
  float* wo = (float*)ring;  // [kWarps][D]
  if (lane == 0) wm[warp] = m, wl[warp] = l;
#pragma unroll
  for (int x = 0; x < E; ++x) wo[warp * D + lane * E + x] = acc[x];
  __syncthreads();
  // this CTA's (max, sum, unnormalised output) into CTA 0's shared memory
  if (tid < D) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = wm[w] == -INFINITY ? 0.f : __expf(wm[w] - M);
      L = fmaf(wl[w], f, L);
      o = fmaf(wo[w * D + tid], f, o);
    }
    *cluster.map_shared_rank(&part_o[rank][tid], 0) = o;
    if (tid == 0) {
      *cluster.map_shared_rank(&part_m[rank], 0) = M;
      *cluster.map_shared_rank(&part_l[rank], 0) = L;
    }
  }

  // the chunk's score and selection at its last token (every CTA, from the
  // running sum read before the barrier, after which CTA 0 rewrites it)
#pragma unroll
  for (int i = 0; i < PE; ++i) {
    const int e = tid + i * kThreads;
    if (e < 2 * D) psv[i] += e < D ? qs[e] : ks[e - D];
  }
  if (last) {
    float s0 = 0.f, s1 = 0.f, unused = 0.f;
#pragma unroll
    for (int i = 0; i < PE; ++i) {
      s0 = fmaf(ws0[i], psv[i], s0);
      s1 = fmaf(ws1[i], psv[i], s1);
    }
    block_sum3(s0, s1, unused, red);
    if (tid == 0) {
      const float a0 = s0 / C + (b_s ? b_s[2 * h] : 0.f);
      const float a1 = s1 / C + (b_s ? b_s[2 * h + 1] : 0.f);
      sel_sh = (a0 >= a1) ? 0 : 1;
    }
  }
  cluster.sync();
  if (!ok && tid == 0) atomicExch(err, 1);

  // the new state rows, stored after the barrier (whose release would
  // otherwise wait for them); at the chunk's last token Gated DeltaNet also
  // makes them the new chunk start, softmax puts the rows back to the chunk
  // start instead (each thread its own columns)
  {
    float* s0row = S0 + (bh * D + srow_i) * D + spart * CPT;
    const bool rollback = last && sel_sh == 0;
    if (rollback) load_n<CPT>(s0row, sv);
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
      const float4 x = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
      *(float4*)(srow + j) = x;
      if (last && !rollback) *(float4*)(s0row + j) = x;
    }
  }

  if (rank == 0) {
    // 4. the partials combined; RMSNorm of each branch and the query-gated sum
    if (tid < D) {
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kSplit; ++r) M = fmaxf(M, part_m[r]);
      float L = 0.f, o = 0.f;
#pragma unroll
      for (int r = 0; r < kSplit; ++r) {
        const float f = part_m[r] == -INFINITY ? 0.f : __expf(part_m[r] - M);
        L = fmaf(part_l[r], f, L);
        o = fmaf(part_o[r][tid], f, o);
      }
      os[tid] = o / L;
    }
    float ss_s = 0.f, ss_l = 0.f, z = 0.f;
    if (tid < D) {
      ss_s = os[tid] * os[tid];
      ss_l = ol[tid] * ol[tid];
      z = qs[tid] * wg;
    }
    block_sum3(ss_s, ss_l, z, red);
    if (tid < D) {
      const float w = 1.f / (1.f + __expf(-(z + bg)));
      const float ns = os[tid] * rsqrtf(ss_s / D + eps) * nws;
      const float nl = ol[tid] * rsqrtf(ss_l / D + eps) * nwl;
      out[bh * D + tid] = from_f32<T>(w * ns + (1.f - w) * nl);
      if (o_s_out) o_s_out[bh * D + tid] = os[tid];
      if (o_l_out) o_l_out[bh * D + tid] = ol[tid];
    }
    // the chunk's running [q; k] sum (restarted after its last token)
#pragma unroll
    for (int i = 0; i < PE; ++i) {
      const int e = tid + i * kThreads;
      if (e < 2 * D) psum[bh * 2 * D + e] = last ? 0.f : psv[i];
    }
  }
  if (!last) return;

  // 5. softmax: this CTA's share of the chunk's keys / values joins the
  //    retained ones (the last one is this token)
  const int sel = sel_sh;
  if (sel == 0) {
    constexpr int RC = kChunk / kSplit;  // chunk rows per CTA
    for (int e = tid; e < RC * D; e += kThreads) {
      const int j = rank * RC + e / D, c = e % D;
      const long long dst = (bh * cap + nr + j) * D + c;
      kv_k[dst] = j == C - 1 ? from_f32<T>(ks[c]) : Kc[(long long)j * D + c];
      kv_v[dst] = j == C - 1 ? from_f32<T>(vs[c]) : Vc[(long long)j * D + c];
    }
    if (rank == 0 && tid == 0) n_kv[bh] = nr + C;
  }
  if (rank == 0 && tid == 0 && sel_out) sel_out[bh] = (uint8_t)sel;
}

// one (dtype, d) instantiation: its ring is dynamic shared memory, and the
// largest carveout keeps four CTAs per SM (attributes set once per kernel)
template <typename T, int D>
cudaError_t launch_one(const Problem& p, int pos, const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                       const float* nw_s, const float* nw_l, float* S, float* S0, void* ck, void* cv,
                       float* psum, void* kv_k, void* kv_v, int32_t* n_kv, long long cap, void* out,
                       uint8_t* sel_out, float* o_s_out, float* o_l_out, int* err, cudaStream_t st) {
  constexpr int smem = Ring<T, D>::kBytes;
  static const cudaError_t attr = [] {
    cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_step_kernel<T, D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  // programmatic stream serialization: the kernel may start while the
  // previous one in the stream finishes (it waits for it before reading)
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.BH * kSplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_step_kernel<T, D>, (const T*)q, (const T*)k, (const T*)v, g, beta, w_s,
                            b_s, w_g, b_g, nw_s, nw_l, (int)p.H, (int)kChunk, pos, p.scale, p.eps, S, S0, (T*)ck,
                            (T*)cv, psum, (T*)kv_k, (T*)kv_v, n_kv, cap, (T*)out, sel_out, o_s_out, o_l_out, err);
}

}  // namespace

cudaError_t launch_decode_step(const Problem& p, int dtype, long long t, const void* q, const void* k,
                               const void* v, const float* g, const float* beta, const float* w_s,
                               const float* b_s, const float* w_g, const float* b_g, const float* nw_s,
                               const float* nw_l, float* S, float* S0, void* ck, void* cv, float* psum,
                               void* kv_k, void* kv_v, int32_t* n_kv, long long cap, void* out,
                               uint8_t* sel_out, float* o_s_out, float* o_l_out, int* err, cudaStream_t st) {
  if (p.BH == 0) return cudaSuccess;
  const int pos = (int)(t % kChunk);
  using bf = __nv_bfloat16;
  auto* fn = dtype == 0 ? (p.d == 64 ? launch_one<bf, 64> : launch_one<bf, 128>)  // NATS_BF16
                        : (p.d == 64 ? launch_one<float, 64> : launch_one<float, 128>);
  return fn(p, pos, q, k, v, g, beta, w_s, b_s, w_g, b_g, nw_s, nw_l, S, S0, ck, cv, psum, kv_k, kv_v, n_kv, cap,
            out, sel_out, o_s_out, o_l_out, err, st);
}

}  // namespace nats
