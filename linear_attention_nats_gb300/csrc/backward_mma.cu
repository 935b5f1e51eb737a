// backward_mma.cu - softmax branch of the backward pass on warp-level
// tensor-core MMAs (bf16 operands, fp32 accumulators), for bf16 layers
// ("Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: query t of chunk c sees every key of the earlier
// chunks that chose softmax and its own chunk up to itself).
//
// Work is in 64 x 64 blocks (a query chunk against a key chunk it sees):
//   S = Q K^T scale, P = exp(S - lse), dP = dO V^T, dS = P (dP - delta),
//   dQ = dS K scale, dK = dS^T Q scale, dV = P^T dO,
// with lse the row log-sum-exp and delta_t = do_s,t . o_s,t.
//   query kernel: one CTA (4 warps x 16 query rows) per (b, h, query chunk)
//     walks the key chunks it sees twice: first for lse (online max / sum),
//     then for dQ, accumulated in registers and added to dq once;
//   key kernel: one CTA (4 warps x 16 key rows) per (b, h, key chunk) walks
//     the query chunks that see it (its own, then all later ones if the
//     chunk chose softmax) and accumulates dK, dV in registers, S^T and dP^T
//     taken in two 32-query halves.
// dO enters as bf16 (rounded once by the norm stage); P and dS are rounded
// to bf16 as the second products' operands.  Operands are staged with
// cp.async into rows skewed by 16 bytes (conflict-free ldmatrix).
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int kC = kChunk;

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// D(16x8 fp32) += A(16x16 bf16, row) B(16x8 bf16, col)
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D>
struct Tile {
  static constexpr int RS = D + 8;             // bf16 row stride
  static constexpr int kBytes = kC * RS * 2;   // one 64-row tile
};

// 64 rows x D bf16 from global (row stride D) into a skewed tile, by 128 threads
template <int D>
__device__ __forceinline__ void load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  constexpr int CPR = D / 8;  // 16-byte pieces per row
  for (int x = threadIdx.x; x < kC * CPR; x += 128) {
    const int r = x / CPR, c = x % CPR;
    cp16(dst + r * Tile<D>::RS + 8 * c, src + (long long)r * D + 8 * c);
  }
}

// A fragment (16 x 16, rows m0.., k 16 ks..) of a row-major tile
template <int RS>
__device__ __forceinline__ void frag_a(const __nv_bfloat16* X, int m0, int ks, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm4(saddr(X + (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 16 * ks + 8 * (lane >> 4)), a);
}
// B fragments of n-tiles 2 jp, 2 jp + 1 for X^T, X row-major [n][k] (rows 16 jp..)
template <int RS>
__device__ __forceinline__ void frag_bt(const __nv_bfloat16* X, int jp, int ks, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm4(saddr(X + (16 * jp + (lane & 7) + 8 * (lane >> 4)) * RS + 16 * ks + 8 * ((lane >> 3) & 1)), b);
}
// B fragments of n-tiles 2 np, 2 np + 1 for X row-major [k][n] (k rows 16 ks..)
template <int RS>
__device__ __forceinline__ void frag_b(const __nv_bfloat16* X, int ks, int np, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm4t(saddr(X + (16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 16 * np + 8 * (lane >> 4)), b);
}
// A fragment for k-step kk from two accumulator n-tiles (2 kk, 2 kk + 1)
__device__ __forceinline__ void acc_to_a(const float (&c0)[4], const float (&c1)[4], uint32_t (&a)[4]) {
  a[0] = pack2(c0[0], c0[1]);
  a[1] = pack2(c0[2], c0[3]);
  a[2] = pack2(c1[0], c1[1]);
  a[3] = pack2(c1[2], c1[3]);
}

// ------------------------------------------------------------ dQ and lse
template <int D>
__global__ void __launch_bounds__(128) softmax_bwd_dq_mma_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const __nv_bfloat16* __restrict__ dos, const float* __restrict__ delta, const uint8_t* __restrict__ sel, int L,
    int N, float scale, float* __restrict__ lse, float* __restrict__ dq) {
  using Tl = Tile<D>;
  constexpr int RS = Tl::RS;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* Qs = (__nv_bfloat16*)smem;
  __nv_bfloat16* Os = (__nv_bfloat16*)(smem + Tl::kBytes);
  __nv_bfloat16* Ks = (__nv_bfloat16*)(smem + 2 * Tl::kBytes);
  __nv_bfloat16* Vs = (__nv_bfloat16*)(smem + 3 * Tl::kBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const long long bh = blockIdx.x / N;
  const int ci = (int)(blockIdx.x % N);
  const long long r0 = bh * L + (long long)ci * kC;  // first row of the query chunk
  const uint8_t* sel_h = sel + bh * N;
  const int m0 = 16 * warp;
  load_tile<D>(Qs, q + r0 * D);
  load_tile<D>(Os, dos + r0 * D);
  // rows gq and gq + 8 of this warp's 16
  const int qa = m0 + gq, qb = qa + 8;
  const float dla = delta[r0 + qa], dlb = delta[r0 + qb];

  // S = Q K_j^T scale for this warp's rows, masked on the diagonal chunk
  auto scores = [&](bool diag, float (&s)[8][4]) {
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) s[n][x] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      frag_a<RS>(Qs, m0, ks, a);
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t b[4];
        frag_bt<RS>(Ks, jp, ks, b);
        mma(s[2 * jp], a, b[0], b[1]);
        mma(s[2 * jp + 1], a, b[2], b[3]);
      }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int key = 8 * n + 2 * cq + (x & 1), row = x < 2 ? qa : qb;
        s[n][x] = (diag && key > row) ? -INFINITY : s[n][x] * scale;
      }
  };
  // the key chunks row chunk ci sees: softmax chunks before it, then itself
  auto next_chunk = [&](int cj) {  // first visible chunk >= cj (ci at most)
    while (cj < ci && sel_h[cj] != 0) ++cj;
    return cj;
  };

  // pass 1: log-sum-exp of rows qa, qb
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
  for (int cj = next_chunk(0); cj <= ci; cj = next_chunk(cj + 1)) {
    load_tile<D>(Ks, k + (bh * L + (long long)cj * kC) * D);
    cp_wait();
    __syncthreads();
    float s[8][4];
    scores(cj == ci, s);
    float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      xa = fmaxf(xa, fmaxf(s[n][0], s[n][1]));
      xb = fmaxf(xb, fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, o));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, o));
    }
    const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
    float ea = 0.f, eb = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      ea += expf(s[n][0] - na) + expf(s[n][1] - na);
      eb += expf(s[n][2] - nb) + expf(s[n][3] - nb);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      ea += __shfl_xor_sync(0xffffffffu, ea, o);
      eb += __shfl_xor_sync(0xffffffffu, eb, o);
    }
    la = la * expf(ma - na) + ea;
    lb = lb * expf(mb - nb) + eb;
    ma = na;
    mb = nb;
    __syncthreads();  // Ks is reloaded next
  }
  const float lsa = ma + logf(la), lsb = mb + logf(lb);
  if (cq == 0) {
    lse[r0 + qa] = lsa;
    lse[r0 + qb] = lsb;
  }

  // pass 2: dQ = sum_j dS_j K_j
  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int x = 0; x < 4; ++x) acc[n][x] = 0.f;
  for (int cj = next_chunk(0); cj <= ci; cj = next_chunk(cj + 1)) {
    const long long kr = bh * L + (long long)cj * kC;
    load_tile<D>(Ks, k + kr * D);
    load_tile<D>(Vs, v + kr * D);
    cp_wait();
    __syncthreads();
    float s[8][4], dp[8][4];
    scores(cj == ci, s);
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) dp[n][x] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      frag_a<RS>(Os, m0, ks, a);
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t b[4];
        frag_bt<RS>(Vs, jp, ks, b);
        mma(dp[2 * jp], a, b[0], b[1]);
        mma(dp[2 * jp + 1], a, b[2], b[3]);
      }
    }
    // dS = P (dP - delta), in place of s
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float p = expf(s[n][x] - (x < 2 ? lsa : lsb));
        s[n][x] = p * (dp[n][x] - (x < 2 ? dla : dlb));
      }
    // dQ += dS K_j (k-dim = the 64 keys)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      acc_to_a(s[2 * kk], s[2 * kk + 1], a);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b[4];
        frag_b<RS>(Ks, kk, np, b);
        mma(acc[2 * np], a, b[0], b[1]);
        mma(acc[2 * np + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();  // Ks, Vs are reloaded next
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int f = 8 * n + 2 * cq;
    float* da = dq + (r0 + qa) * D + f;
    float* db = dq + (r0 + qb) * D + f;
    da[0] += scale * acc[n][0];
    da[1] += scale * acc[n][1];
    db[0] += scale * acc[n][2];
    db[1] += scale * acc[n][3];
  }
}

// ------------------------------------------------------------- dK and dV
template <int D>
__global__ void __launch_bounds__(128) softmax_bwd_dkv_mma_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const __nv_bfloat16* __restrict__ dos, const float* __restrict__ delta, const float* __restrict__ lse,
    const uint8_t* __restrict__ sel, int L, int N, float scale, float* __restrict__ dk, float* __restrict__ dv) {
  using Tl = Tile<D>;
  constexpr int RS = Tl::RS;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* Ks = (__nv_bfloat16*)smem;
  __nv_bfloat16* Vs = (__nv_bfloat16*)(smem + Tl::kBytes);
  __nv_bfloat16* Qs = (__nv_bfloat16*)(smem + 2 * Tl::kBytes);
  __nv_bfloat16* Os = (__nv_bfloat16*)(smem + 3 * Tl::kBytes);
  float* lses = (float*)(smem + 4 * Tl::kBytes);
  float* dls = lses + kC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const long long bh = blockIdx.x / N;
  const int cj = (int)(blockIdx.x % N);
  const long long k0 = bh * L + (long long)cj * kC;  // first row of the key chunk
  const int m0 = 16 * warp;
  const int ka = m0 + gq, kb = ka + 8;  // this thread's key rows
  load_tile<D>(Ks, k + k0 * D);
  load_tile<D>(Vs, v + k0 * D);
  float adk[D / 8][4], adv[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int x = 0; x < 4; ++x) adk[n][x] = adv[n][x] = 0.f;
  // the query chunks that see key chunk cj: itself, then every later one if
  // it chose softmax
  const int ci_end = sel[bh * N + cj] == 0 ? N : cj + 1;
  for (int ci = cj; ci < ci_end; ++ci) {
    const long long r0 = bh * L + (long long)ci * kC;
    load_tile<D>(Qs, q + r0 * D);
    load_tile<D>(Os, dos + r0 * D);
    if (threadIdx.x < kC) {
      lses[threadIdx.x] = lse[r0 + threadIdx.x];
      dls[threadIdx.x] = delta[r0 + threadIdx.x];
    }
    cp_wait();
    __syncthreads();
    const bool diag = ci == cj;
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {  // queries 32 hq .. 32 hq + 31
      float st[4][4], dpt[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int x = 0; x < 4; ++x) st[n][x] = dpt[n][x] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t ak[4], av[4];
        frag_a<RS>(Ks, m0, ks, ak);
        frag_a<RS>(Vs, m0, ks, av);
#pragma unroll
        for (int jq = 0; jq < 2; ++jq) {
          uint32_t bq[4], bo[4];
          frag_bt<RS>(Qs, 2 * hq + jq, ks, bq);
          frag_bt<RS>(Os, 2 * hq + jq, ks, bo);
          mma(st[2 * jq], ak, bq[0], bq[1]);
          mma(st[2 * jq + 1], ak, bq[2], bq[3]);
          mma(dpt[2 * jq], av, bo[0], bo[1]);
          mma(dpt[2 * jq + 1], av, bo[2], bo[3]);
        }
      }
      // P^T and dS^T, in place
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int qc = 32 * hq + 8 * n + 2 * cq + (x & 1), key = x < 2 ? ka : kb;
          const float p = (diag && key > qc) ? 0.f : expf(st[n][x] * scale - lses[qc]);
          st[n][x] = p;
          dpt[n][x] = p * (dpt[n][x] - dls[qc]);
        }
      // dV += P^T dO, dK += dS^T Q (k-dim = the half's 32 queries)
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t ap[4], as[4];
        acc_to_a(st[2 * kk], st[2 * kk + 1], ap);
        acc_to_a(dpt[2 * kk], dpt[2 * kk + 1], as);
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t bo[4], bq[4];
          frag_b<RS>(Os, 2 * hq + kk, np, bo);
          frag_b<RS>(Qs, 2 * hq + kk, np, bq);
          mma(adv[2 * np], ap, bo[0], bo[1]);
          mma(adv[2 * np + 1], ap, bo[2], bo[3]);
          mma(adk[2 * np], as, bq[0], bq[1]);
          mma(adk[2 * np + 1], as, bq[2], bq[3]);
        }
      }
    }
    __syncthreads();  // Qs, Os, lse, delta are reloaded next
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int f = 8 * n + 2 * cq;
    *(float2*)(dk + (k0 + ka) * D + f) = make_float2(scale * adk[n][0], scale * adk[n][1]);
    *(float2*)(dk + (k0 + kb) * D + f) = make_float2(scale * adk[n][2], scale * adk[n][3]);
    *(float2*)(dv + (k0 + ka) * D + f) = make_float2(adv[n][0], adv[n][1]);
    *(float2*)(dv + (k0 + kb) * D + f) = make_float2(adv[n][2], adv[n][3]);
  }
}

template <int D>
cudaError_t run(const Problem& p, const void* q, const void* k, const void* v, const void* dos, const float* delta,
                const uint8_t* sel, float* lse, float* dq, float* dk, float* dv, cudaStream_t st) {
  constexpr int smem_q = 4 * Tile<D>::kBytes;
  constexpr int smem_k = 4 * Tile<D>::kBytes + 2 * kC * 4;
  static const cudaError_t attr = [] {
    cudaError_t e = cudaFuncSetAttribute(softmax_bwd_dq_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_q);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(softmax_bwd_dkv_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_k);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  const unsigned grid = (unsigned)(p.BH * p.N);
  using bf = __nv_bfloat16;
  softmax_bwd_dq_mma_kernel<D><<<grid, 128, smem_q, st>>>((const bf*)q, (const bf*)k, (const bf*)v, (const bf*)dos,
                                                          delta, sel, p.L, p.N, p.scale, lse, dq);
  softmax_bwd_dkv_mma_kernel<D><<<grid, 128, smem_k, st>>>((const bf*)q, (const bf*)k, (const bf*)v,
                                                           (const bf*)dos, delta, lse, sel, p.L, p.N, p.scale, dk, dv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_bwd_mma(const Problem& p, const void* q, const void* k, const void* v, const void* dos,
                                   const float* delta, const uint8_t* sel, float* lse, float* dq, float* dk,
                                   float* dv, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run<64>(p, q, k, v, dos, delta, sel, lse, dq, dk, dv, st)
                   : run<128>(p, q, k, v, dos, delta, sel, lse, dq, dk, dv, st);
}

}  // namespace nats
