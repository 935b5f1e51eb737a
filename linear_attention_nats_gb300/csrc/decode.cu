// decode.cu - the NAtS-L layer in decode mode: one new token per (b, h) per
// launch ("Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" items 1, 3 and 4, read token by token).
//
// A cluster of kSplit CTAs (256 threads each) per (b, h); the keys are split
// between the cluster's CTAs, which keeps many more loads in flight than
// one CTA per head:
//   1. the token's q, k, v to shared memory (every CTA); CTA 0 appends k, v
//      to the chunk's keys / values at position p = t % chunk;
//   2. CTA 0: Gated DeltaNet, S <- a S (I - beta k k^T) + beta v k^T, i.e.
//      row i of S becomes a S_i + beta (v_i - a S_i . k) k^T, and
//      o_l = S (scale q), 256 / d threads per state row (fp32 state in
//      global memory);
//   3. CTAs 1 .. kSplit - 1: softmax over their share of the keys (the
//      retained keys of earlier softmax chunks, then the chunk's keys up to
//      the token): a warp takes its keys in batches of eight, lanes split the
//      d features (one coalesced 256-byte row per key), the next batch's rows
//      are loaded while the current one is scored; the eight dot products
//      are summed over the warp by halving (nine shuffles); the CTA's warps
//      are combined and its (max, sum, partial output) goes into CTA 0's
//      shared memory (distributed shared memory) before a cluster barrier;
//   4. CTA 0: the kSplit partials combined, RMSNorm of both branches and the
//      query-gated sum;
//   5. CTA 0: the running [q; k] sum of the chunk; when the token completes
//      the chunk: the chunk score and selection; softmax appends the chunk's
//      keys and values to the retained ones and restores the state to the
//      chunk start, Gated DeltaNet keeps the state as the new chunk start.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSplit = 8;  // CTAs per (b, h) (a thread-block cluster): CTA 0 the state, CTAs 1.. the keys

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

template <typename T, int D>
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads, 1) decode_step_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, const float* __restrict__ w_s, const float* __restrict__ b_s,
    const float* __restrict__ w_g, const float* __restrict__ b_g, const float* __restrict__ nw_s,
    const float* __restrict__ nw_l, int H, int C, int p, float scale, float eps, float* __restrict__ S,
    float* __restrict__ S0, T* __restrict__ ck, T* __restrict__ cv, float* __restrict__ psum,
    T* __restrict__ kv_k, T* __restrict__ kv_v, int32_t* __restrict__ n_kv, long long cap, T* __restrict__ out,
    uint8_t* __restrict__ sel_out, float* __restrict__ o_s_out, float* __restrict__ o_l_out) {
  static_assert(D % 32 == 0 && D <= 128, "shape");
  constexpr int CPT = 32;              // state columns per thread
  constexpr int TPR = D / CPT;         // threads per state row
  constexpr int RPP = kThreads / TPR;  // state rows per pass
  constexpr int E = D / 32;            // features per lane in the softmax
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long bh = blockIdx.x / kSplit;
  const int h = (int)(bh % H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ __align__(16) float qs[D], ks[D], vs[D], os[D], ol[D];
  __shared__ __align__(16) float wo[kWarps][D];
  __shared__ float wm[kWarps], wl[kWarps];
  __shared__ float red[kWarps][3];
  __shared__ __align__(16) float part_o[kSplit][D];  // CTA 0: the cluster's partial outputs
  __shared__ float part_m[kSplit], part_l[kSplit];
  __shared__ int sel_sh;

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
  __syncthreads();

  // 2. Gated DeltaNet state update and readout (CTA 0)
  if (rank == 0) {
#pragma unroll 1
    for (int row0 = 0; row0 < D; row0 += RPP) {
      const int row = row0 + tid / TPR, part = tid % TPR;
      if (RPP > D && row >= D) break;  // (d = 64: half the threads have no row); warp-uniform
      float* srow = S + (bh * D + row) * D + part * CPT;
      float sv[CPT];
      load_n<CPT>(srow, sv);
      float u = 0.f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) u = fmaf(sv[j], ks[part * CPT + j], u);
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
      const float coef = bt * (vs[row] - a * u);
      float r = 0.f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        sv[j] = fmaf(a, sv[j], coef * ks[part * CPT + j]);
        r = fmaf(sv[j], qs[part * CPT + j], r);
      }
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
#pragma unroll
      for (int j = 0; j < CPT; j += 4)
        *(float4*)(srow + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
      if (part == 0) ol[row] = r * scale;
    }
  }

  // 3. softmax over the retained keys and the chunk's keys up to the token
  {
    const int nr = n_kv[bh];
    const int n = nr + p + 1;  // key n - 1 is this token (taken from shared memory)
    // keys [lo, hi) of this CTA (CTA 0 has none), [wlo, whi) of this warp
    const int nk = kSplit - 1, kr_ = rank - 1;
    const int lo = rank == 0 ? 0 : (int)((long long)n * kr_ / nk), hi = rank == 0 ? 0 : (int)((long long)n * (kr_ + 1) / nk);
    const int wlo = lo + (int)((long long)(hi - lo) * warp / kWarps), whi = lo + (int)((long long)(hi - lo) * (warp + 1) / kWarps);
    const T* Kr = kv_k + bh * cap * D;
    const T* Vr = kv_v + bh * cap * D;
    const T* Kc = ck + bh * C * D;
    const T* Vc = cv + bh * C * D;
    float qv[E];
#pragma unroll
    for (int x = 0; x < E; ++x) qv[x] = qs[lane * E + x];
    float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
    for (int x = 0; x < E; ++x) acc[x] = 0.f;
    // lane's E features of key / value row j, in storage form (zeros past
    // the end of the warp's keys; this token's from the inputs)
    using RV = Raw<T, E>;
    auto fetch = [&](int j, RV (&kb)[8], RV (&vb)[8], int u) {
      if (j >= whi) {
        kb[u].zero();
        vb[u].zero();
      } else if (j == n - 1) {
        kb[u].load(k + bh * D + lane * E);
        vb[u].load(v + bh * D + lane * E);
      } else {
        const long long off = (j < nr ? (long long)j : (long long)(j - nr)) * D + lane * E;
        kb[u].load((j < nr ? Kr : Kc) + off);
        vb[u].load((j < nr ? Vr : Vc) + off);
      }
    };
    auto fetch8 = [&](int j0, RV (&kb)[8], RV (&vb)[8]) {
#pragma unroll
      for (int u = 0; u < 8; ++u) fetch(j0 + u, kb, vb, u);
    };
    // the 8 keys from j0: scores (partial dot products summed over the warp
    // by halving: lane (b4 b3 b2 . .) ends with key 4 b4 + 2 b3 + b2), online
    // softmax, P V
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
      const float sc = (j0 + ku < whi) ? d1 * scale : -INFINITY;
      float mb = sc;
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
      const float mn = fmaxf(m, mb);
      const float alpha = __expf(m - mn);  // 0 on the first batch (m = -inf)
      const float pu = (j0 + ku < whi) ? __expf(sc - mn) : 0.f;
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
    // two batches of rows in flight: the next one loads while one is scored
    RV k0[8], v0[8], k1[8], v1[8];
    if (wlo < whi) fetch8(wlo, k0, v0);
    for (int j0 = wlo; j0 < whi; j0 += 16) {
      fetch8(j0 + 8, k1, v1);
      batch(j0, k0, v0);
      if (j0 + 8 >= whi) break;
      fetch8(j0 + 16, k0, v0);
      batch(j0 + 8, k1, v1);
    }
    if (lane == 0) wm[warp] = m, wl[warp] = l;
#pragma unroll
    for (int x = 0; x < E; ++x) wo[warp][lane * E + x] = acc[x];
    __syncthreads();
    // this CTA's (max, sum, unnormalised output) into CTA 0's shared memory
    float* po = cluster.map_shared_rank(&part_o[rank][0], 0);
    if (tid < D) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w]);
      float L = 0.f, o = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = wm[w] == -INFINITY ? 0.f : __expf(wm[w] - M);
        L = fmaf(wl[w], f, L);
        o = fmaf(wo[w][tid], f, o);
      }
      po[tid] = o;
      if (tid == 0) {
        *cluster.map_shared_rank(&part_m[rank], 0) = M;
        *cluster.map_shared_rank(&part_l[rank], 0) = L;
      }
    }
    cluster.sync();
    if (rank != 0) return;  // only CTA 0's shared memory is read after the barrier
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
    __syncthreads();
  }

  // 4. RMSNorm of each branch and the query-gated sum
  {
    float ss_s = 0.f, ss_l = 0.f, z = 0.f;
    if (tid < D) {
      ss_s = os[tid] * os[tid];
      ss_l = ol[tid] * ol[tid];
      z = qs[tid] * w_g[(long long)h * D + tid];
    }
    block_sum3(ss_s, ss_l, z, red);
    if (tid < D) {
      const float w = 1.f / (1.f + __expf(-(z + (b_g ? b_g[h] : 0.f))));
      const float ns = os[tid] * rsqrtf(ss_s / D + eps) * (nw_s ? nw_s[tid] : 1.f);
      const float nl = ol[tid] * rsqrtf(ss_l / D + eps) * (nw_l ? nw_l[tid] : 1.f);
      out[bh * D + tid] = from_f32<T>(w * ns + (1.f - w) * nl);
      if (o_s_out) o_s_out[bh * D + tid] = os[tid];
      if (o_l_out) o_l_out[bh * D + tid] = ol[tid];
    }
  }

  // 5. the chunk's [q; k] sum; at the chunk's last token the selection,
  //    then commit or rollback
  float ps = 0.f;
  if (tid < 2 * D) {
    ps = psum[bh * 2 * D + tid] + (tid < D ? qs[tid] : ks[tid - D]);
    psum[bh * 2 * D + tid] = ps;
  }
  if (p != C - 1) return;
  {
    float s0 = 0.f, s1 = 0.f, unused = 0.f;
    if (tid < 2 * D) {
      s0 = w_s[((long long)h * 2 + 0) * 2 * D + tid] * ps;
      s1 = w_s[((long long)h * 2 + 1) * 2 * D + tid] * ps;
    }
    block_sum3(s0, s1, unused, red);
    if (tid == 0) {
      const float a0 = s0 / C + (b_s ? b_s[2 * h] : 0.f);
      const float a1 = s1 / C + (b_s ? b_s[2 * h + 1] : 0.f);
      sel_sh = (a0 >= a1) ? 0 : 1;
    }
    __syncthreads();  // also: every thread's state row is written
  }
  const int sel = sel_sh;
  if (tid < 2 * D) psum[bh * 2 * D + tid] = 0.f;
  float* Sh = S + bh * D * D;
  float* S0h = S0 + bh * D * D;
  if (sel == 0) {
    // softmax: the chunk's keys / values join the retained ones; the state
    // returns to the chunk start
    const int nr = n_kv[bh];
    T* dk = kv_k + (bh * cap + nr) * D;
    T* dv = kv_v + (bh * cap + nr) * D;
    const T* sk = ck + bh * C * D;
    const T* sv = cv + bh * C * D;
    for (int e = tid; e < C * D; e += kThreads) {
      dk[e] = sk[e];
      dv[e] = sv[e];
    }
    for (int e = tid; e < D * D / 4; e += kThreads) ((float4*)Sh)[e] = ((const float4*)S0h)[e];
    __syncthreads();
    if (tid == 0) n_kv[bh] = nr + C;
  } else {
    // Gated DeltaNet: the state is committed and starts the next chunk
    for (int e = tid; e < D * D / 4; e += kThreads) ((float4*)S0h)[e] = ((const float4*)Sh)[e];
  }
  if (tid == 0 && sel_out) sel_out[bh] = (uint8_t)sel;
}

}  // namespace

cudaError_t launch_decode_step(const Problem& p, int dtype, long long t, const void* q, const void* k,
                               const void* v, const float* g, const float* beta, const float* w_s,
                               const float* b_s, const float* w_g, const float* b_g, const float* nw_s,
                               const float* nw_l, float* S, float* S0, void* ck, void* cv, float* psum,
                               void* kv_k, void* kv_v, int32_t* n_kv, long long cap, void* out,
                               uint8_t* sel_out, float* o_s_out, float* o_l_out, cudaStream_t st) {
  if (p.BH == 0) return cudaSuccess;
  const int pos = (int)(t % kChunk);
  auto run = [&](auto kern, auto tag) -> cudaError_t {
    using T = decltype(tag);
    kern<<<(unsigned)(p.BH * kSplit), kThreads, 0, st>>>(
        (const T*)q, (const T*)k, (const T*)v, g, beta, w_s, b_s, w_g, b_g, nw_s, nw_l, p.H, kChunk, pos,
        p.scale, p.eps, S, S0, (T*)ck, (T*)cv, psum, (T*)kv_k, (T*)kv_v, n_kv, cap, (T*)out, sel_out, o_s_out,
        o_l_out);
    return cudaGetLastError();
  };
  if (dtype == 0) {  // NATS_BF16
    return p.d == 64 ? run(decode_step_kernel<__nv_bfloat16, 64>, __nv_bfloat16())
                     : run(decode_step_kernel<__nv_bfloat16, 128>, __nv_bfloat16());
  }
  return p.d == 64 ? run(decode_step_kernel<float, 64>, 0.f) : run(decode_step_kernel<float, 128>, 0.f);
}

}  // namespace nats
