// gdn_bwd_chunk.cu - the Gated DeltaNet branch of the backward pass in
// chunkwise form (bf16 layers).
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" items 3 and 5: the linear state is pseudo-updated through
// every chunk and rolled back after a chunk that chose softmax; the layer is
// trained end to end.  Per chunk (C = 64 tokens; G the in-chunk cumulative
// log-decay, gamma = e^G; Q~ = scale q; S0 the state at the chunk start,
// dv x dk) the forward is
//   A[i, j] = e^{G_i - G_j} k_i . k_j (j < i),  Linv = (I + diag(beta) A)^{-1}
//   Vh = V - diag(gamma) K S0^T,   U = Linv diag(beta) Vh
//   P[i, j] = e^{G_i - G_j} q~_i . k_j (j <= i),   O = diag(gamma) Q~ S0^T + P U
//   S_C = gamma_C S0 + U^T K~,  K~ = diag(gamma_C / gamma) K   (committed chunks)
// and, with dO the gradient of O and dS_C that of S_C (zero for a chunk that
// is rolled back, and for the last one), its adjoint is
//   dU = P^T dO + K~ dS_C^T,  Y = Linv^T dU,  dVh = diag(beta) Y = dV
//   dS0 = dS_C (gamma_C I - K~^T W) + dO^T Q_eff
//       with W = Linv diag(beta gamma) K, Q_eff = diag(gamma) Q~ - P W
//   dP = lower(dO U^T),  dL = -strict_lower(Y U^T),  dA = diag(beta) dL
//   dQ~ = (dP . R) K + diag(gamma) dO S0
//   dK  = (dP . R)^T Q~ + (A~ + A~^T) K - diag(gamma) dVh S0 + diag(gamma_C / gamma) U dS_C
//   dbeta_i = Y_i . Vh_i + sum_j dL_ij A_ij
//   dG = row sums - column sums of dP.P and dA.A, + gamma_i (dO S0)_i . q~_i
//        - gamma_i (dVh S0)_i . k_i - (U dS_C)_j . K~_j, and at the last token
//        sum_j (U dS_C)_j . K~_j + gamma_C <dS_C, S0>;  dg = reverse cumsum of dG
// (R[i, j] = e^{G_i - G_j}, A~ = dA . R).  The state gradient runs backwards
// over the chunks: dS_c = dS0 of chunk c with dS_C = dS_{c+1} for a committed
// chunk, dS_{c+1} + dO^T Q_eff for a rolled-back one.
//
// Kernels (after the forward scan has written every chunk's S0; S0 and
// dS_C are stored transposed, [dk][dv], so that both scans write them as
// whole lines):
//   gdn_bwd_prep_kernel   per chunk: G, P (fp32), W, Q_eff, K~ (fp16, scaled), from
//                         Linv as the forward's chunk-factor kernel stores it
//   gdn_bwd_scan_kernel   per (b, h, 64 state rows): the reverse scan, writing
//                         dS_C of every committed chunk (fp32)
//   gdn_bwd_fused_kernel  per chunk, every product above: Vh, U, dU, Y, the
//                         C x C products; dq, dk, dv updated once each, dbeta
//                         and dg written
// Products run on warp-level tensor cores with fp32 accumulation over fp16
// operand tiles read through ldmatrix (m16n8k16), each tile scaled by its
// own power of two so that its largest entry sits below 2^15 (fp16 range is
// never exceeded, its 11-bit precision matches tf32); the reverse scan keeps
// its state gradient in fp32 and feeds it, X = dS K~^T and dO to the
// products as fp16 rows, each at its own power-of-two scale (taken within a
// quad of threads: no block-wide reduction on the chain).
// The chunk-factor and scan kernels have 8 warps, the fused kernel 16; a C x D
// output is split into 16-row strips (warp w & 3) and column halves (8
// warps) or quarters (16 warps) (warp w >> 2).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

constexpr int C = kChunk;
using bf16 = __nv_bfloat16;

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}

// f(row, col, value, index into the tile) for every accumulator element
// base[r][c] += acc (rows m0.., columns n0..; row stride D), two adjacent
// columns per 8-byte access, the loads of four column groups issued before
// their stores
template <int NT, int D>
__device__ __forceinline__ void acc_add_global(const float (&acc)[NT][4], int m0, int n0, float* base) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  constexpr int GJ = NT < 4 ? NT : 4;
#pragma unroll
  for (int j0 = 0; j0 < NT; j0 += GJ) {
    float2 old[GJ][2];
#pragma unroll
    for (int j = 0; j < GJ; ++j) {
      const int c0 = n0 + 8 * (j0 + j) + 2 * t;
      old[j][0] = *(const float2*)(base + (size_t)(m0 + g) * D + c0);
      old[j][1] = *(const float2*)(base + (size_t)(m0 + g + 8) * D + c0);
    }
#pragma unroll
    for (int j = 0; j < GJ; ++j) {
      const int c0 = n0 + 8 * (j0 + j) + 2 * t;
      const float* a = acc[j0 + j];
      *(float2*)(base + (size_t)(m0 + g) * D + c0) = make_float2(old[j][0].x + a[0], old[j][0].y + a[1]);
      *(float2*)(base + (size_t)(m0 + g + 8) * D + c0) = make_float2(old[j][1].x + a[2], old[j][1].y + a[3]);
    }
  }
}

template <int NT, class F>
__device__ __forceinline__ void each(const float (&acc)[NT][4], int m0, int n0, F f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c0 = n0 + 8 * j + 2 * t;
    f(m0 + g, c0, acc[j][0], j, 0);
    f(m0 + g, c0 + 1, acc[j][1], j, 1);
    f(m0 + g + 8, c0, acc[j][2], j, 2);
    f(m0 + g + 8, c0 + 1, acc[j][3], j, 3);
  }
}

// per-row partial sums of a thread (its rows m0 + g and m0 + g + 8) summed
// over the quad and added into dst[row]
__device__ __forceinline__ void add_rows(float lo, float hi, int m0, float* dst) {
  lo += __shfl_xor_sync(0xffffffffu, lo, 1);
  lo += __shfl_xor_sync(0xffffffffu, lo, 2);
  hi += __shfl_xor_sync(0xffffffffu, hi, 1);
  hi += __shfl_xor_sync(0xffffffffu, hi, 2);
  const int lane = threadIdx.x & 31;
  if ((lane & 3) == 0) {
    atomicAdd(dst + m0 + (lane >> 2), lo);
    atomicAdd(dst + m0 + (lane >> 2) + 8, hi);
  }
}

// per-column partial sums (columns n0 + 8 j + 2 t + e) summed over the eight
// row groups of the warp and added into dst[col]
template <int NT>
__device__ __forceinline__ void add_cols(float (&v)[NT][2], int n0, float* dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float x = v[j][e];
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      if (lane < 4) atomicAdd(dst + n0 + 8 * j + 2 * lane + e, x);
    }
}

template <int D>
struct Tiles {
  static constexpr int FS = D + 4;  // fp32 row stride of C x D and D x D tiles
  static constexpr int BS = D + 8;  // bf16 row stride of C x D tiles
};

// a hint: bring `bytes` (a multiple of 16, 16-byte aligned) at p into L2
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

// the chunk's cumulative log-decay G (from Gb) and gamma, beta into shared memory
__device__ __forceinline__ void load_scalars(const float* Gb, const float* beta, size_t row0, float* sG, float* sGam,
                                             float* sB) {
  if (threadIdx.x < C) {
    const float G = Gb[row0 + threadIdx.x];
    sG[threadIdx.x] = G;
    sGam[threadIdx.x] = __expf(G);
    sB[threadIdx.x] = beta[row0 + threadIdx.x];
  }
}

// ---------------------------------------------------------- fp16 operands
using half = __half;

template <int COLS>
struct H {
  static constexpr int ld = COLS + 8;  // row stride (halves): 16-byte rows, ldmatrix without bank conflicts
  static constexpr int bytes(int rows) { return rows * ld * 2; }
};

__device__ __forceinline__ void ldsm4(const half* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void ldsm4t(const half* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc[j] (rows m0 .. m0 + 15, columns n0 + 8 j .. + 7) += sum_k A(i, k) B(k, n)
// over fp16 tiles: A stored [m][k] (AT false) or [k][m] (AT true), B stored
// [n][k] (BT false) or [k][n] (BT true); NT even, K a multiple of 16
template <int NT, int K, bool AT, bool BT>
__device__ __forceinline__ void hmm(float (&acc)[NT][4], int m0, int n0, const half* A, int lda, const half* B,
                                    int ldb) {
  static_assert(NT % 2 == 0, "pairs of n8 tiles");
  const int lane = threadIdx.x & 31, mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4];
    if (!AT)
      ldsm4(A + (m0 + (lane & 15)) * lda + k0 + 8 * (lane >> 4), a);
    else
      ldsm4t(A + (k0 + (mi >> 1) * 8 + r8) * lda + m0 + (mi & 1) * 8, a);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      uint32_t b[4];
      if (!BT)
        ldsm4(B + (n0 + 8 * j + (mi >> 1) * 8 + r8) * ldb + k0 + (mi & 1) * 8, b);
      else
        ldsm4t(B + (k0 + (mi & 1) * 8 + r8) * ldb + n0 + 8 * j + (mi >> 1) * 8, b);
      mma16(acc[j], a, b[0], b[1]);
      mma16(acc[j + 1], a, b[2], b[3]);
    }
  }
}

// A power of two s with m s < 2^15 (1 for m = 0 or not finite).
__device__ __forceinline__ float pow2_scale(float m) {
  if (!(m > 0.f) || !(m < INFINITY)) return 1.f;
  int e = ((__float_as_int(m) >> 23) & 0xff) - 127;  // m in [2^e, 2^(e+1)) for normal m
  e = min(max(e, -100), 100);
  return __int_as_float((127 + 14 - e) << 23);
}

// The scales of NS tiles from every thread's partial maxima m[u] of |x| (a
// block-wide collective over NTH threads; red: NS x NTH / 32 floats of
// shared memory).
template <int NS, int NTH>
__device__ __forceinline__ void block_scalesN(float (&m)[NS], float* red, float (&s)[NS]) {
  constexpr int NW = NTH / 32;
#pragma unroll
  for (int u = 0; u < NS; ++u) m[u] = warp_max(m[u]);
  __syncthreads();  // red is free again
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int u = 0; u < NS; ++u) red[u * NW + (threadIdx.x >> 5)] = m[u];
  __syncthreads();
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    float r = red[u * NW];
#pragma unroll
    for (int w = 1; w < NW; ++w) r = fmaxf(r, red[u * NW + w]);
    s[u] = pow2_scale(r);
  }
}

// The scale of a tile from every thread's partial max |x| (a block-wide
// collective; red: NTH / 32 floats of shared memory).
template <int NTH = 256>
__device__ __forceinline__ float block_scale(float m, float* red) {
  float mm[1] = {m}, s[1];
  block_scalesN<1, NTH>(mm, red, s);
  return s[0];
}

__device__ __forceinline__ float max4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}
__device__ __forceinline__ uint2 half4(float4 v, float s) {
  const __half2 a = __floats2half2_rn(v.x * s, v.y * s), b = __floats2half2_rn(v.z * s, v.w * s);
  return make_uint2(*(const uint32_t*)&a, *(const uint32_t*)&b);
}

// fp32 ROWS x COLS (row stride src_ld; global or shared) -> scaled fp16 tile;
// returns the scale.  f(r, c, v) may rewrite each value first.
template <int ROWS, int COLS, int NTH = 256, class F>
__device__ __forceinline__ float tile_h(const float* src, int src_ld, half* dst, float* red, F f) {
  constexpr int V = ROWS * COLS / 4 / NTH;
  static_assert(V >= 1 && ROWS * COLS % (4 * NTH) == 0, "tile");
  float4 v[V];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int x = threadIdx.x + NTH * i, r = x / (COLS / 4), c = 4 * (x % (COLS / 4));
    v[i] = *(const float4*)(src + (size_t)r * src_ld + c);
    v[i].x = f(r, c, v[i].x);
    v[i].y = f(r, c + 1, v[i].y);
    v[i].z = f(r, c + 2, v[i].z);
    v[i].w = f(r, c + 3, v[i].w);
    m = fmaxf(m, max4(v[i]));
  }
  const float s = block_scale<NTH>(m, red);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int x = threadIdx.x + NTH * i, r = x / (COLS / 4), c = 4 * (x % (COLS / 4));
    *(uint2*)(dst + r * H<COLS>::ld + c) = half4(v[i], s);
  }
  return s;
}
template <int ROWS, int COLS, int NTH = 256>
__device__ __forceinline__ float tile_h(const float* src, int src_ld, half* dst, float* red) {
  return tile_h<ROWS, COLS, NTH>(src, src_ld, dst, red, [](int, int, float x) { return x; });
}

// A tile held in registers between its loads and its scaled store, so that
// the loads of several tiles are in flight together and their scales come
// from one block-wide reduction (block_scales2).
template <int D, int NTH = 256>
struct BF16Tile {  // bf16 C x D (row stride D) -> scaled fp16 tile
  static constexpr int V = C * D / 8 / NTH;
  uint4 v[V];
  float m;
  __device__ __forceinline__ void load(const bf16* src) {
    m = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = threadIdx.x + NTH * i, r = x / (D / 8), c = 8 * (x % (D / 8));
      v[i] = *(const uint4*)(src + (size_t)r * D + c);
    }
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const __nv_bfloat162* h2 = (const __nv_bfloat162*)&v[i];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h2[u]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  __device__ __forceinline__ void store(half* dst, float s) const {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = threadIdx.x + NTH * i, r = x / (D / 8), c = 8 * (x % (D / 8));
      const __nv_bfloat162* h2 = (const __nv_bfloat162*)&v[i];
      uint4 o;
      uint32_t* o32 = (uint32_t*)&o;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h2[u]);
        const __half2 hh = __floats2half2_rn(f.x * s, f.y * s);
        o32[u] = *(const uint32_t*)&hh;
      }
      *(uint4*)(dst + r * H<D>::ld + c) = o;
    }
  }
};
// The scales of two tiles from every thread's partial maxima (a block-wide
// collective; red: 16 floats of shared memory).
__device__ __forceinline__ void block_scales2(float m1, float m2, float* red, float& s1, float& s2) {
  m1 = warp_max(m1);
  m2 = warp_max(m2);
  __syncthreads();  // red is free again
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = m1;
    red[8 + (threadIdx.x >> 5)] = m2;
  }
  __syncthreads();
  float r1 = red[0], r2 = red[8];
#pragma unroll
  for (int w = 1; w < 8; ++w) r1 = fmaxf(r1, red[w]), r2 = fmaxf(r2, red[8 + w]);
  s1 = pow2_scale(r1);
  s2 = pow2_scale(r2);
}

// accumulators (rows m0.., columns n0..) -> scaled fp16 tile (a block-wide
// collective: every thread calls it); returns the scale
template <int NT, int COLS, int NTH = 256>
__device__ __forceinline__ float acc_h(const float (&acc)[NT][4], int m0, int n0, half* dst, float* red) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(acc[j][e]));
  const float s = block_scale<NTH>(m, red);
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c0 = n0 + 8 * j + 2 * t;
    *(__half2*)(dst + (m0 + g) * H<COLS>::ld + c0) = __floats2half2_rn(acc[j][0] * s, acc[j][1] * s);
    *(__half2*)(dst + (m0 + g + 8) * H<COLS>::ld + c0) = __floats2half2_rn(acc[j][2] * s, acc[j][3] * s);
  }
  return s;
}

// fp16 C x D rows (global, row stride D) -> the padded tile, asynchronously
template <int D, int NTH = 256>
__device__ __forceinline__ void copy_h(half* dst, const half* src) {
  for (int x = threadIdx.x; x < C * D / 8; x += NTH) {
    const int r = x / (D / 8), c8 = 8 * (x % (D / 8));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst + r * H<D>::ld + c8)),
                 "l"(src + (size_t)r * D + c8)
                 : "memory");
  }
}
__device__ __forceinline__ void copy_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int NT, class F>
__device__ __forceinline__ void each_mut(float (&acc)[NT][4], int m0, int n0, F f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c0 = n0 + 8 * j + 2 * t;
    acc[j][0] = f(m0 + g, c0, acc[j][0], j, 0);
    acc[j][1] = f(m0 + g, c0 + 1, acc[j][1], j, 1);
    acc[j][2] = f(m0 + g + 8, c0, acc[j][2], j, 2);
    acc[j][3] = f(m0 + g + 8, c0 + 1, acc[j][3], j, 3);
  }
}

// ------------------------------------------------------------------ prep
template <int D>
struct PrepSm {
  static constexpr int offQ = 0;                              // fp16 [C][D + 8]
  static constexpr int offK = offQ + H<D>::bytes(C);
  static constexpr int offW = offK + H<D>::bytes(C);
  static constexpr int offL = offW + H<D>::bytes(C);          // fp16 [C][C + 8]: Linv diag(beta gamma)
  static constexpr int offPh = offL + H<C>::bytes(C);         // fp16 [C][C + 8]: P
  static constexpr int offV = offPh + H<C>::bytes(C);         // G, gamma, beta, reduction
  static constexpr int kBytes = offV + 3 * C * 4 + 64;
};

// Linv comes from the forward's chunk-factor kernel (rerun for the
// chunk-start states), which forms it by its blocked inverse.
template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_prep_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k,
                                                           const float* __restrict__ g,
                                                           const float* __restrict__ beta, int L, int N, float scale,
                                                           float* __restrict__ Gb, const float* __restrict__ Li,
                                                           float* __restrict__ P_out, half* __restrict__ W16,
                                                           half* __restrict__ Qe16, half* __restrict__ Kt16,
                                                           float* __restrict__ sc_out) {
  using S = PrepSm<D>;
  constexpr int NT = D / 16, LD = H<D>::ld, LC = H<C>::ld;
  extern __shared__ __align__(16) uint8_t sm[];
  half* hQ = (half*)(sm + S::offQ);
  half* hK = (half*)(sm + S::offK);
  half* hW = (half*)(sm + S::offW);
  half* hL = (half*)(sm + S::offL);
  half* hP = (half*)(sm + S::offPh);
  float* sG = (float*)(sm + S::offV);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* red = sB + C;
  const long long chunk = blockIdx.x;
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)(chunk % N) * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {  // in-chunk cumulative log-decay: two tokens per lane, then a warp scan
    const float x0 = g[row0 + 2 * lane], x1 = g[row0 + 2 * lane + 1];
    float s = x0 + x1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sG[2 * lane] = s - x1;
    sG[2 * lane + 1] = s;
    sGam[2 * lane] = __expf(s - x1);
    sGam[2 * lane + 1] = __expf(s);
    Gb[row0 + 2 * lane] = s - x1;
    Gb[row0 + 2 * lane + 1] = s;
  }
  if (tid < C) sB[tid] = beta[row0 + tid];
  float sq, sk;
  {  // q and k: both tiles' loads in flight at once, one reduction (its barriers also publish sG, sB)
    BF16Tile<D> tq, tk;
    tq.load(q + row0 * D);
    tk.load(k + row0 * D);
    block_scales2(tq.m, tk.m, red, sq, sk);
    tq.store(hQ, sq);
    tk.store(hK, sk);
  }
  // Linv diag(beta gamma) (the W product's operand)
  const float sl = tile_h<C, C>(Li + (size_t)chunk * C * C, C, hL, red,
                                [&](int, int m, float x) { return x * sB[m] * sGam[m]; });
  __syncthreads();
  // P (lower, diagonal included)
  float sp;
  {
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
    float qk[4][4];
    zero(qk);
    hmm<4, D, false, false>(qk, m0, n0, hQ, LD, hK, LD);
    const float iqk = scale / (sq * sk);
    each_mut(qk, m0, n0, [&](int i, int j, float v, int, int) {
      return j <= i ? __expf(sG[i] - sG[j]) * v * iqk : 0.f;
    });
    {  // P to memory, two columns per 8-byte store
      const int g = lane >> 2, t = lane & 3;
      float* pd = P_out + (size_t)chunk * C * C;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c0 = n0 + 8 * j + 2 * t;
        *(float2*)(pd + (m0 + g) * C + c0) = make_float2(qk[j][0], qk[j][1]);
        *(float2*)(pd + (m0 + g + 8) * C + c0) = make_float2(qk[j][2], qk[j][3]);
      }
    }
    sp = acc_h<4, C>(qk, m0, n0, hP, red);
  }
  __syncthreads();
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
  // W = Linv diag(beta gamma) K
  float acc[NT][4];
  zero(acc);
  hmm<NT, C, false, true>(acc, m0, n0, hL, LC, hK, LD);
  {
    const float iw = 1.f / (sl * sk);
    each_mut(acc, m0, n0, [&](int, int, float v, int, int) { return v * iw; });
  }
  const float sw = acc_h<NT, D>(acc, m0, n0, hW, red);
  __syncthreads();
  // W and K~ for the reverse scan: fp16 rows as staged (K~ = the K tile
  // times gamma_C / gamma <= 1, at the K tile's scale)
  for (int x = tid; x < C * D / 8; x += 256) {
    const int i = x / (D / 8), c8 = 8 * (x % (D / 8));
    *(uint4*)(W16 + (row0 + i) * D + c8) = *(const uint4*)(hW + i * LD + c8);
    const float f = sGam[C - 1] / sGam[i];
    const __half2* k2 = (const __half2*)(hK + i * LD + c8);
    uint4 o;
    __half2* o2 = (__half2*)&o;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 kf = __half22float2(k2[u]);
      o2[u] = __floats2half2_rn(kf.x * f, kf.y * f);
    }
    *(uint4*)(Kt16 + (row0 + i) * D + c8) = o;
  }
  // Q_eff = diag(gamma) Q~ - P W (fp16, at its own scale)
  zero(acc);
  hmm<NT, C, false, true>(acc, m0, n0, hP, LC, hW, LD);
  {
    const float ipw = 1.f / (sp * sw), iq = scale / sq;
    each_mut(acc, m0, n0, [&](int i, int n, float v, int, int) {
      return sGam[i] * iq * __half2float(hQ[i * LD + n]) - v * ipw;
    });
    float mq = 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) mq = fmaxf(mq, fabsf(acc[j][e]));
    const float sqe = block_scale(mq, red);
    each(acc, m0, n0, [&](int i, int n, float v, int j, int e) {  // pairs (n, n + 1)
      if ((e & 1) == 0) *(__half2*)(Qe16 + (row0 + i) * D + n) = __floats2half2_rn(v * sqe, acc[j][e + 1] * sqe);
    });
    if (tid == 0) {
      sc_out[chunk * 4 + 0] = sw;
      sc_out[chunk * 4 + 1] = sqe;
      sc_out[chunk * 4 + 2] = sk;
    }
  }
}

// ------------------------------------------------------------------ scan
constexpr int RB = 64;  // state-gradient rows per CTA (BH x D / 64 CTAs: one wave at the layer's sizes)

// acc[j] (rows m0 .. m0 + 15, columns n0 + 8 j .. + 7) += sum_k A(i, k) B(k, n)
// with A fp32 in shared memory, [m][k] (AT false; row stride = 8 mod 32
// words: conflict-free 8-byte loads) or [k][m] (AT true; row stride = 4 mod
// 16 words), and B fp16 as in hmm.  Each row of A enters as fp16 at its own
// power-of-two scale (the four threads of a quad hold the whole row, so the
// scale takes two shuffles, no barrier); u_lo and u_hi return the inverse
// scales of the thread's rows m0 + g and m0 + g + 8, by which the caller
// multiplies the accumulator rows.
template <int NT, int K, bool AT, bool BT>
__device__ __forceinline__ void rmm(float (&acc)[NT][4], float& u_lo, float& u_hi, int m0, int n0, const float* A,
                                    int lda, const half* B, int ldb) {
  static_assert(NT % 2 == 0 && K % 16 == 0, "pairs of n8 tiles, k16 blocks");
  constexpr int KB = K / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, mi = lane >> 3, r8 = lane & 7;
  // x[kb]: row g at k = 2t, 2t + 1, 2t + 8, 2t + 9 of block kb, then row g + 8
  float x[KB][8];
  float mlo = 0.f, mhi = 0.f;
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    const int k = 16 * kb + 2 * t;
    if (!AT) {
      const float* r_lo = A + (m0 + g) * lda + k;
      const float* r_hi = A + (m0 + g + 8) * lda + k;
      const float2 p0 = *(const float2*)r_lo, p1 = *(const float2*)(r_lo + 8);
      const float2 q0 = *(const float2*)r_hi, q1 = *(const float2*)(r_hi + 8);
      x[kb][0] = p0.x, x[kb][1] = p0.y, x[kb][2] = p1.x, x[kb][3] = p1.y;
      x[kb][4] = q0.x, x[kb][5] = q0.y, x[kb][6] = q1.x, x[kb][7] = q1.y;
    } else {
      const int kk[4] = {k, k + 1, k + 8, k + 9};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[kb][e] = A[kk[e] * lda + m0 + g];
        x[kb][4 + e] = A[kk[e] * lda + m0 + g + 8];
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mlo = fmaxf(mlo, fabsf(x[kb][e]));
      mhi = fmaxf(mhi, fabsf(x[kb][4 + e]));
    }
  }
  mlo = fmaxf(mlo, __shfl_xor_sync(0xffffffffu, mlo, 1));
  mlo = fmaxf(mlo, __shfl_xor_sync(0xffffffffu, mlo, 2));
  mhi = fmaxf(mhi, __shfl_xor_sync(0xffffffffu, mhi, 1));
  mhi = fmaxf(mhi, __shfl_xor_sync(0xffffffffu, mhi, 2));
  const float slo = pow2_scale(mlo), shi = pow2_scale(mhi);
  u_lo = 1.f / slo;
  u_hi = 1.f / shi;
  auto pack = [](float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  };
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    const int k0 = 16 * kb;
    uint32_t a[4];
    a[0] = pack(x[kb][0] * slo, x[kb][1] * slo);
    a[1] = pack(x[kb][4] * shi, x[kb][5] * shi);
    a[2] = pack(x[kb][2] * slo, x[kb][3] * slo);
    a[3] = pack(x[kb][6] * shi, x[kb][7] * shi);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      uint32_t b[4];
      if (!BT)
        ldsm4(B + (n0 + 8 * j + (mi >> 1) * 8 + r8) * ldb + k0 + (mi & 1) * 8, b);
      else
        ldsm4t(B + (k0 + (mi & 1) * 8 + r8) * ldb + n0 + 8 * j + (mi >> 1) * 8, b);
      mma16(acc[j], a, b[0], b[1]);
      mma16(acc[j + 1], a, b[2], b[3]);
    }
  }
}

template <int D>
struct ScanSm {
  static constexpr int kTile = H<D>::bytes(C);   // fp16 [C][D + 8]
  static constexpr int OL = RB + 4;              // fp32 [C][RB + 4]: dO columns of the CTA's rows
  static constexpr int kO = C * OL * 4;
  static constexpr int kStage = 3 * kTile + kO;  // K~, W, Q_eff, dO
  static constexpr int FS = D + 8;               // fp32 [RB][D + 8]: the state gradient
  static constexpr int XS = C + 8;               // fp32 [RB][C + 8]: X = -dS K~^T
  static constexpr int offS = 2 * kStage;
  static constexpr int offX = offS + RB * FS * 4;
  static constexpr int kBytes = offX + RB * XS * 4;
};


// The state gradient, backwards over the chunks of one head, RB rows per
// CTA (the rows are independent): dS_C of chunk c is the state gradient
// before its step; then dS <- gamma_C dS - (dS K~^T) W + dO^T Q_eff for a
// committed chunk, dS + dO^T Q_eff for a rolled-back one.  dS stays fp32 in
// shared memory and enters the products as fp16 rows at their own scales, as
// do X and dO^T; K~, W and Q_eff are the chunk-factor kernel's fp16 tiles at
// their stored scales.
// Two barriers a step: the step's stage is complete and the last update
// visible (then the next stage's copies start: every read of the stage they
// overwrite is behind that barrier), and X complete.  The update writes the
// next chunk's dS_C (when it is committed) from registers.
template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_scan_kernel(const half* __restrict__ Kt16,
                                                           const half* __restrict__ W16,
                                                           const half* __restrict__ Qe16,
                                                           const float* __restrict__ sc,
                                                           const float* __restrict__ dO, const float* __restrict__ Gb,
                                                           const uint8_t* __restrict__ sel, int L, int N,
                                                           float* __restrict__ dSC) {
  using S = ScanSm<D>;
  constexpr int FS = S::FS, XS = S::XS, OL = S::OL, LD = H<D>::ld;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sdS = (float*)(sm + S::offS);
  float* sX = (float*)(sm + S::offX);
  constexpr int splits = D / RB;
  const long long bh = blockIdx.x / splits;
  const int r0 = (blockIdx.x % splits) * RB;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, g = lane >> 2, t = lane & 3;
  for (int x = tid; x < RB * FS; x += 256) sdS[x] = 0.f;
  auto stage_ptr = [&](int st, int which) { return sm + st * S::kStage + which * S::kTile; };
  auto prefetch = [&](int c) {
    const int st = c & 1;
    const size_t row0 = (size_t)bh * L + (size_t)c * C;
    const half* srcs[3] = {Kt16, W16, Qe16};
#pragma unroll
    for (int w3 = 0; w3 < 3; ++w3) {
      half* dst = (half*)stage_ptr(st, w3);
      for (int x = tid; x < C * D / 8; x += 256) {
        const int r = x / (D / 8), c8 = x % (D / 8);
        cp16(dst + r * LD + 8 * c8, srcs[w3] + (row0 + r) * D + 8 * c8);
      }
    }
    float* dO_s = (float*)stage_ptr(st, 3);
    for (int x = tid; x < C * RB / 4; x += 256) {
      const int r = x / (RB / 4), c4 = x % (RB / 4);
      cp16(dO_s + r * OL + 4 * c4, dO + (row0 + r) * D + r0 + 4 * c4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if (N > 0) prefetch(N - 1);
  // the step's selection, scales and end-of-chunk log-decay, read one step
  // ahead (a global load on the chain costs as much as a product)
  struct StepScalars {
    bool lin;
    float sw, sqe, skt, GC;
  };
  auto step_scalars = [&](int c) {
    StepScalars s;
    const long long ch = bh * N + c;
    s.lin = sel[ch] != 0;
    s.sw = sc[ch * 4];
    s.sqe = sc[ch * 4 + 1];
    s.skt = sc[ch * 4 + 2];
    s.GC = Gb[(size_t)bh * L + (size_t)c * C + C - 1];
    return s;
  };
  StepScalars nx = step_scalars(N > 0 ? N - 1 : 0);
  for (int c = N - 1; c >= 0; --c) {
    const StepScalars cur = nx;
    if (c > 0) nx = step_scalars(c - 1);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (c > 0) prefetch(c - 1);
    const int st = c & 1;
    const half* hKt = (const half*)stage_ptr(st, 0);
    const half* hW = (const half*)stage_ptr(st, 1);
    const half* hQe = (const half*)stage_ptr(st, 2);
    const float* sO = (const float*)stage_ptr(st, 3);
    const bool lin = cur.lin;
    if (lin) {  // X = -dS K~^T (RB x C)
      const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
      float acc[4][4];
      zero(acc);
      float ulo, uhi;
      rmm<4, D, false, false>(acc, ulo, uhi, m0, n0, sdS, FS, hKt, LD);
      const float ilo = -ulo / cur.skt, ihi = -uhi / cur.skt;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c0 = n0 + 8 * j + 2 * t;
        *(float2*)(sX + (m0 + g) * XS + c0) = make_float2(acc[j][0] * ilo, acc[j][1] * ilo);
        *(float2*)(sX + (m0 + g + 8) * XS + c0) = make_float2(acc[j][2] * ihi, acc[j][3] * ihi);
      }
    }
    __syncthreads();
    {  // dS <- gamma_C dS + X W + dO^T Q_eff (committed), dS + dO^T Q_eff (rolled back)
      constexpr int NT = D / 16;
      const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
      float a1[NT][4], a2[NT][4];
      zero(a1);
      zero(a2);
      float u1[2] = {0.f, 0.f}, u2[2];
      if (lin) rmm<NT, C, false, true>(a1, u1[0], u1[1], m0, n0, sX, XS, hW, LD);
      rmm<NT, C, true, true>(a2, u2[0], u2[1], m0, n0, sO, OL, hQe, LD);
      const float gC = lin ? __expf(cur.GC) : 1.f;
      const float f1[2] = {u1[0] / cur.sw, u1[1] / cur.sw}, f2[2] = {u2[0] / cur.sqe, u2[1] / cur.sqe};
      // dS_C of chunk c - 1 (when committed), stored transposed ([dk][dv])
      // like the chunk-start states: 8 consecutive rows of a column make one
      // whole 32-byte sector
      float* dst = (c > 0 && nx.lin) ? dSC + (size_t)(bh * N + c - 1) * D * D + r0 : nullptr;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c0 = n0 + 8 * j + 2 * t;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = m0 + g + 8 * hr;
          float2* p = (float2*)(sdS + i * FS + c0);
          const float2 o = *p;
          const float2 v = make_float2(gC * o.x + a1[j][2 * hr] * f1[hr] + a2[j][2 * hr] * f2[hr],
                                       gC * o.y + a1[j][2 * hr + 1] * f1[hr] + a2[j][2 * hr + 1] * f2[hr]);
          *p = v;
          if (dst) {
            dst[(size_t)c0 * D + i] = v.x;
            dst[(size_t)(c0 + 1) * D + i] = v.y;
          }
        }
      }
    }
  }
}

// ------------------------------------------ every per-chunk product, fused
// One CTA of 16 warps per chunk holds all of the chunk's operand tiles in
// shared memory (fp16, each at its own power-of-two scale) and takes every
// product of the adjoint in turn, so that dq, dk and dv are each updated
// once, dbeta and dg written once, and no per-chunk intermediate goes
// through global memory.  A C x D output is split into 16-row strips
// (warp w & 3) and column quarters (warp w >> 2); a C x C output likewise.
template <int D>
struct FusedSm {
  static constexpr int offS = 0;                        // fp16 [D][D + 8]: S0 ([dk][dv])
  static constexpr int offT = offS + H<D>::bytes(D);    // dS_C ([dk][dv])
  static constexpr int offQ = offT + H<D>::bytes(D);    // fp16 [C][D + 8]: q
  static constexpr int offK = offQ + H<D>::bytes(C);    // k
  static constexpr int offV = offK + H<D>::bytes(C);    // v (bf16 as loaded), then Vh
  static constexpr int offO = offV + H<D>::bytes(C);    // dO
  static constexpr int offU = offO + H<D>::bytes(C);    // U
  static constexpr int offD = offU + H<D>::bytes(C);    // dU, then Y
  static constexpr int offL = offD + H<D>::bytes(C);    // fp16 [C][C + 8]: Linv
  static constexpr int offLb = offL + H<C>::bytes(C);   // Linv diag(beta)
  static constexpr int offP = offLb + H<C>::bytes(C);   // P, then dP . R
  static constexpr int offA = offP + H<C>::bytes(C);    // A~
  static constexpr int offVec = offA + H<C>::bytes(C);  // G, gamma, beta, dG, dbeta
  static constexpr int offRed = offVec + 5 * C * 4;     // partial maxima; [126]: extra dG of the last token; [127]: <dS_C, S0>
  static constexpr int kBytes = offRed + 128 * 4;
};

template <int D>
__global__ void __launch_bounds__(512, 1) gdn_bwd_fused_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v, const float* __restrict__ dO,
    const float* __restrict__ S0, const float* __restrict__ dSC, const float* __restrict__ Li,
    const float* __restrict__ Pg, const float* __restrict__ Gb, const float* __restrict__ beta,
    const uint8_t* __restrict__ sel, int L, int N, float scale, float* __restrict__ dq, float* __restrict__ dk,
    float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta) {
  using S = FusedSm<D>;
  constexpr int NTH = 512, NTD = D / 32, LD = H<D>::ld, LC = H<C>::ld;
  extern __shared__ __align__(16) uint8_t sm[];
  half* hS = (half*)(sm + S::offS);
  half* hT = (half*)(sm + S::offT);
  half* hQ = (half*)(sm + S::offQ);
  half* hK = (half*)(sm + S::offK);
  half* hV = (half*)(sm + S::offV);
  half* hO = (half*)(sm + S::offO);
  half* hU = (half*)(sm + S::offU);
  half* hD = (half*)(sm + S::offD);
  half* hL = (half*)(sm + S::offL);
  half* hLb = (half*)(sm + S::offLb);
  half* hP = (half*)(sm + S::offP);
  half* hA = (half*)(sm + S::offA);
  float* sG = (float*)(sm + S::offVec);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* sdG = sB + C;
  float* sdB = sdG + C;
  float* red = (float*)(sm + S::offRed);
  const long long chunk = blockIdx.x;
  const int c = (int)(chunk % N);
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)c * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool committed = sel[chunk] != 0 && c < N - 1;
  load_scalars(Gb, beta, row0, sG, sGam, sB);
  if (tid < C) sdG[tid] = sdB[tid] = 0.f;
  if (tid < 2) red[126 + tid] = 0.f;
  copy_h<D, NTH>(hV, (const half*)(v + row0 * D));  // v (bf16) staged where Vh will be formed
  // S0 and dS_C (a committed chunk's; zero otherwise), read in the same
  // order so that <dS_C, S0> is taken in fp32 on the way
  float ss, sd;
  {
    constexpr int V = D * D / 4 / NTH;
    const float* s0 = S0 + (size_t)chunk * D * D;
    const float* ds = dSC + (size_t)chunk * D * D;
    float4 a[V], b[V];
    float m[2] = {0.f, 0.f}, sc2[2], dot = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
      a[i] = *(const float4*)(s0 + (size_t)r * D + cc);
      m[0] = fmaxf(m[0], max4(a[i]));
    }
    if (committed) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
        b[i] = *(const float4*)(ds + (size_t)r * D + cc);
        m[1] = fmaxf(m[1], max4(b[i]));
        dot += a[i].x * b[i].x + a[i].y * b[i].y + a[i].z * b[i].z + a[i].w * b[i].w;
      }
    }
    block_scalesN<2, NTH>(m, red, sc2);
    ss = sc2[0];
    sd = sc2[1];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
      *(uint2*)(hS + r * LD + cc) = half4(a[i], ss);
      if (committed) *(uint2*)(hT + r * LD + cc) = half4(b[i], sd);
    }
    if (committed) {
      dot = warp_sum(dot);
      if (lane == 0) atomicAdd(red + 127, dot);
    }
  }
  // q, k, dO, Linv (plain and with its columns scaled by beta) and P: every
  // load in flight together, one reduction for the six scales
  float sq, sk, so, sl, slb, sp;
  {
    constexpr int VO = C * D / 4 / NTH, VC = C * C / 4 / NTH;
    BF16Tile<D, NTH> tq, tk;
    tq.load(q + row0 * D);
    tk.load(k + row0 * D);
    float4 o[VO], l[VC], pp[VC];
    float m[6] = {tq.m, tk.m, 0.f, 0.f, 0.f, 0.f}, s6[6];
    const float* lsrc = Li + (size_t)chunk * C * C;
    const float* psrc = Pg + (size_t)chunk * C * C;
#pragma unroll
    for (int i = 0; i < VO; ++i) {
      const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
      o[i] = *(const float4*)(dO + (row0 + r) * D + cc);
      m[2] = fmaxf(m[2], max4(o[i]));
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int x = tid + NTH * i, r = x / (C / 4), cc = 4 * (x % (C / 4));
      l[i] = *(const float4*)(lsrc + r * C + cc);
      pp[i] = *(const float4*)(psrc + r * C + cc);
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int x = tid + NTH * i, cc = 4 * (x % (C / 4));
      m[3] = fmaxf(m[3], max4(l[i]));
      const float4 lb = make_float4(l[i].x * sB[cc], l[i].y * sB[cc + 1], l[i].z * sB[cc + 2], l[i].w * sB[cc + 3]);
      m[4] = fmaxf(m[4], max4(lb));
      m[5] = fmaxf(m[5], max4(pp[i]));
    }
    block_scalesN<6, NTH>(m, red, s6);
    sq = s6[0], sk = s6[1], so = s6[2], sl = s6[3], slb = s6[4], sp = s6[5];
    tq.store(hQ, sq);
    tk.store(hK, sk);
#pragma unroll
    for (int i = 0; i < VO; ++i) {
      const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
      *(uint2*)(hO + r * LD + cc) = half4(o[i], so);
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int x = tid + NTH * i, r = x / (C / 4), cc = 4 * (x % (C / 4));
      const float4 lb = make_float4(l[i].x * sB[cc], l[i].y * sB[cc + 1], l[i].z * sB[cc + 2], l[i].w * sB[cc + 3]);
      *(uint2*)(hL + r * LC + cc) = half4(l[i], sl);
      *(uint2*)(hLb + r * LC + cc) = half4(lb, slb);
      *(uint2*)(hP + r * LC + cc) = half4(pp[i], sp);
    }
  }
  copy_wait();
  __syncthreads();
  const int m0 = 16 * (warp & 3), nD = (warp >> 2) * (D / 4), nC = (warp >> 2) * (C / 4);
  const float gC = sGam[C - 1];
  float acc[NTD][4], acc2[NTD][4];
  // Vh = V - diag(gamma) K S0^T
  zero(acc);
  hmm<NTD, D, false, true>(acc, m0, nD, hK, LD, hS, LD);
  {
    const float iks = 1.f / (sk * ss);
    const bf16* vs = (const bf16*)hV;
    each_mut(acc, m0, nD, [&](int i, int n, float val, int, int) {
      return __bfloat162float(vs[i * LD + n]) - sGam[i] * val * iks;
    });
  }
  const float svh = acc_h<NTD, D, NTH>(acc, m0, nD, hV, red);  // (every read of v precedes its barriers)
  __syncthreads();
  // U = Linv diag(beta) Vh
  zero(acc);
  hmm<NTD, C, false, true>(acc, m0, nD, hLb, LC, hV, LD);
  {
    const float iu = 1.f / (slb * svh);
    each_mut(acc, m0, nD, [&](int, int, float val, int, int) { return val * iu; });
  }
  const float su = acc_h<NTD, D, NTH>(acc, m0, nD, hU, red);
  __syncthreads();
  // dU = P^T dO + K~ dS_C^T
  zero(acc);
  zero(acc2);
  hmm<NTD, C, true, true>(acc, m0, nD, hP, LC, hO, LD);
  if (committed) hmm<NTD, D, false, true>(acc2, m0, nD, hK, LD, hT, LD);
  {
    const float ipo = 1.f / (sp * so), ikd = 1.f / (sk * sd);
    each_mut(acc, m0, nD, [&](int i, int, float val, int j, int e) {
      return val * ipo + gC / sGam[i] * acc2[j][e] * ikd;
    });
  }
  const float sdu = acc_h<NTD, D, NTH>(acc, m0, nD, hD, red);
  // dP = lower(dO U^T), P = R . Q~ K^T (the chunk factor, fp32): dP . R
  // replaces P; dG += row sums - column sums of dP . P
  float spm;
  {
    float ou[2][4];
    zero(ou);
    hmm<2, D, false, false>(ou, m0, nC, hO, LD, hU, LD);
    const float iou = 1.f / (so * su);
    const float* pg = Pg + (size_t)chunk * C * C;
    float rlo = 0.f, rhi = 0.f, col[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    each_mut(ou, m0, nC, [&](int i, int jj, float val, int j, int e) {
      float pm = 0.f;
      if (jj <= i) {
        const float r = __expf(sG[i] - sG[jj]);
        const float dP = val * iou;
        const float x = dP * pg[i * C + jj];
        if (e < 2) rlo += x; else rhi += x;
        col[j][e & 1] -= x;
        pm = dP * r;
      }
      return pm;
    });
    add_rows(rlo, rhi, m0, sdG);
    add_cols<2>(col, nC, sdG);
    spm = acc_h<2, C, NTH>(ou, m0, nC, hP, red);  // (every read of P precedes its barriers)
  }
  __syncthreads();
  // dq += scale diag(gamma) dO S0 + scale (dP . R) K (one accumulator: the
  // first product is brought to the second's scale before it is added);
  // dG_i += gamma_i (dO S0)_i . q~_i
  {
    zero(acc);
    hmm<NTD, D, false, false>(acc, m0, nD, hO, LD, hS, LD);
    const float ios = scale / (so * ss), f2 = scale / (spm * sk), if2 = (spm * sk) / scale, iq = 1.f / sq;
    float lo = 0.f, hi = 0.f;
    each_mut(acc, m0, nD, [&](int i, int n, float val, int, int e) {
      const float x = sGam[i] * val * ios;
      const float dd = x * __half2float(hQ[i * LD + n]) * iq;
      if (e < 2) lo += dd; else hi += dd;
      return x * if2;
    });
    add_rows(lo, hi, m0, sdG);
    hmm<NTD, C, false, true>(acc, m0, nD, hP, LC, hK, LD);
    each_mut(acc, m0, nD, [&](int, int, float val, int, int) { return val * f2; });
    acc_add_global<NTD, D>(acc, m0, nD, dq + row0 * D);
  }
  // Y = Linv^T dU (replaces dU); dv += diag(beta) Y; dbeta_i = Y_i . Vh_i
  float sy;
  {
    zero(acc);
    hmm<NTD, C, true, true>(acc, m0, nD, hL, LC, hD, LD);
    const float iy = 1.f / (sl * sdu), ivh = 1.f / svh;
    float lo = 0.f, hi = 0.f;
    each_mut(acc, m0, nD, [&](int i, int n, float val, int, int e) {
      const float y = val * iy;
      const float dd = y * __half2float(hV[i * LD + n]) * ivh;
      if (e < 2) lo += dd; else hi += dd;
      return y;
    });
    add_rows(lo, hi, m0, sdB);
    sy = acc_h<NTD, D, NTH>(acc, m0, nD, hD, red);  // (every read of dU precedes its barriers)
    each_mut(acc, m0, nD, [&](int i, int, float y, int, int) { return sB[i] * y; });
    acc_add_global<NTD, D>(acc, m0, nD, dv + row0 * D);
  }
  __syncthreads();
  // dL = -strict_lower(Y U^T), A = R . K K^T: dA = diag(beta) dL, A~ = dA . R,
  // dbeta_i += sum_j dL_ij A_ij, dG += row sums - column sums of dA . A
  float sa;
  {
    float yu[2][4], kk[2][4];
    zero(yu);
    zero(kk);
    hmm<2, D, false, false>(yu, m0, nC, hD, LD, hU, LD);
    hmm<2, D, false, false>(kk, m0, nC, hK, LD, hK, LD);
    const float iyu = 1.f / (sy * su), ikk = 1.f / (sk * sk);
    float rlo = 0.f, rhi = 0.f, blo = 0.f, bhi = 0.f, col[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    each_mut(yu, m0, nC, [&](int i, int jj, float val, int j, int e) {
      float at = 0.f;
      if (jj < i) {
        const float r = __expf(sG[i] - sG[jj]);
        const float A = r * kk[j][e] * ikk;
        const float dL = -val * iyu;
        const float dA = sB[i] * dL;
        const float x = dA * A;
        if (e < 2) rlo += x, blo += dL * A; else rhi += x, bhi += dL * A;
        col[j][e & 1] -= x;
        at = dA * r;
      }
      return at;
    });
    add_rows(rlo, rhi, m0, sdG);
    add_rows(blo, bhi, m0, sdB);
    add_cols<2>(col, nC, sdG);
    sa = acc_h<2, C, NTH>(yu, m0, nC, hA, red);
  }
  __syncthreads();
  // dk += diag(gamma_C / gamma) U dS_C - diag(gamma beta) Y S0 + (dP . R)^T Q~
  //       + (A~ + A~^T) K
  {
    float dkp[NTD][4];
    zero(dkp);
    const float ik = 1.f / sk;
    if (committed) {  // dG_j -= (U dS_C)_j . K~_j; the last token gains their sum
      hmm<NTD, D, false, false>(dkp, m0, nD, hU, LD, hT, LD);
      const float iud = 1.f / (su * sd);
      float lo = 0.f, hi = 0.f;
      each_mut(dkp, m0, nD, [&](int i, int n, float val, int, int e) {
        const float x = gC / sGam[i] * val * iud;
        const float dd = x * ik * __half2float(hK[i * LD + n]);
        if (e < 2) lo -= dd; else hi -= dd;
        return x;
      });
      const float tot = warp_sum(-(lo + hi));
      add_rows(lo, hi, m0, sdG);
      if (lane == 0) atomicAdd(red + 126, tot);
    }
    {  // dG_i -= gamma_i beta_i (Y S0)_i . k_i
      zero(acc);
      hmm<NTD, D, false, false>(acc, m0, nD, hD, LD, hS, LD);
      const float iys = 1.f / (sy * ss);
      float lo = 0.f, hi = 0.f;
      each(acc, m0, nD, [&](int i, int n, float val, int j, int e) {
        const float x = sGam[i] * sB[i] * val * iys;
        dkp[j][e] -= x;
        const float dd = x * ik * __half2float(hK[i * LD + n]);
        if (e < 2) lo -= dd; else hi -= dd;
      });
      add_rows(lo, hi, m0, sdG);
    }
    zero(acc);
    zero(acc2);
    hmm<NTD, C, true, true>(acc, m0, nD, hP, LC, hQ, LD);
    hmm<NTD, C, false, true>(acc2, m0, nD, hA, LC, hK, LD);
    hmm<NTD, C, true, true>(acc2, m0, nD, hA, LC, hK, LD);
    const float f1 = scale / (spm * sq), fa = 1.f / (sa * sk);
    each(acc, m0, nD, [&](int, int, float val, int j, int e) { dkp[j][e] += f1 * val + fa * acc2[j][e]; });
    acc_add_global<NTD, D>(dkp, m0, nD, dk + row0 * D);
  }
  __syncthreads();
  if (tid == 0) sdG[C - 1] += red[126] + gC * red[127];
  __syncthreads();
  if (warp == 0) {  // dg = reverse cumulative sum of dG over the chunk
    const float a0 = sdG[2 * lane], a1 = sdG[2 * lane + 1];
    float s = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, s, o);
      if (lane + o < 32) s += y;
    }
    // s = sum over lanes >= this one
    const float after = s - a0 - a1;
    dg[row0 + 2 * lane + 1] = a1 + after;
    dg[row0 + 2 * lane] = a0 + a1 + after;
  }
  if (tid < C) dbeta[row0 + tid] = sdB[tid];
}

// ------------------------------------------ the per-chunk products on tcgen05
// (d = 128).  The products of gdn_bwd_fused_kernel on the 5th-generation
// tensor cores: every C x D product is taken transposed (TMEM lane = feature
// dv or dk, column = token; M = 128, N = 64), the C x C ones as
// [Y; dO] U^T and [K; Q] K^T (rows of Y and K in lanes 0-63, of dO and Q in
// lanes 64-127, so that each lane quarter holds the rows its epilogue
// pairs).  Operand tiles are fp16 at their own power-of-two scales in
// 128-byte-swizzled lines; thread 0 issues each phase's MMAs, and warp w
// reads TMEM lanes 32 (w & 3) .. + 31, columns 16 (w >> 2) .. + 15.
namespace tcb {
constexpr int D = 128, NTH = 512;
constexpr int kBlk = 16384;     // distance between the 64-column blocks of a 128-column tile
constexpr int offS = 0;         // S0   [dk][dv]  (128 lines x 128 columns)
constexpr int offT = 32768;     // dS_C [dk][dv]
constexpr int offYO = 65536;    // [Y; dO] [128][dv]: Y lines 0-63, dO lines 64-127
constexpr int offKQ = 98304;    // [K; Q]  [128][dk]: K lines 0-63, Q lines 64-127
constexpr int offVh = 131072;   // Vh^T [dv][64]
constexpr int offU = 147456;    // U^T  [dv][64]
constexpr int offDU = 163840;   // dU^T [dv][64]
constexpr int offL = 180224;    // Linv [64][64]
constexpr int offLb = 188416;   // Linv diag(beta)
constexpr int offP = 196608;    // P, then dP . R
constexpr int offA = 204800;    // A~
constexpr int offVec = 212992;  // G, gamma, beta, dG, dbeta (fp32 [64] each)
constexpr int offRed = offVec + 5 * C * 4;  // 128 floats: partial maxima; [126] extra dG of the last token; [127] <dS_C, S0>
constexpr int offBar = offRed + 128 * 4;    // 6 mbarriers, one per phase
constexpr int offFlag = offBar + 6 * 8;     // a wait ran out (the rest of the CTA's waits are skipped)
constexpr int offTmem = offFlag + 8;
constexpr int kBytes = offTmem + 8 + 1024;  // + alignment slack of the dynamic base
static_assert(offVec == offA + 8192 && offA % 1024 == 0, "tiles");
// TMEM columns (64 fp32 each); the last phase reuses those read before it
constexpr uint32_t cVh = 0, cDqA = 64, cDub = 128, cKQ = 192, cU = 256, cDua = 320, cY = 384, cYO = 448;
constexpr uint32_t cDqB = 0, cDka = 256, cDkb = 320, cDkc = 384, cDkd = 128;
constexpr uint32_t ID_KK = tc::idesc_f16_f32(128, 64, false, false), ID_MK = tc::idesc_f16_f32(128, 64, true, false),
                   ID_KM = tc::idesc_f16_f32(128, 64, false, true), ID_MM = tc::idesc_f16_f32(128, 64, true, true);

// byte offset of element (r, c) of a swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 6) * kBlk + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}
// K-major operand at shared address t, lines r0 .., k = 16 kk .. + 15
__device__ __forceinline__ uint64_t kmaj(uint32_t t, int r0, int kk) {
  return tc::smem_desc_sw128(t + r0 * 128 + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
}
// MN-major operand at shared address t (lines = k), k = 16 kk .. + 15
__device__ __forceinline__ uint64_t mnmaj(uint32_t t, int kk) {
  return tc::smem_desc_sw128(t + kk * 2048, kBlk, 1024);
}
__device__ __forceinline__ void st4(uint8_t* tile, int r, int c, float4 v, float s) {
  *(uint2*)(tile + swz(r, c)) = half4(v, s);
}
__device__ __forceinline__ void st_bf8(uint8_t* tile, int r, int c, uint4 raw, float s) {
  const __nv_bfloat162* h2 = (const __nv_bfloat162*)&raw;
  uint4 o;
  uint32_t* o32 = (uint32_t*)&o;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 x = __bfloat1622float2(h2[u]);
    const __half2 hh = __floats2half2_rn(x.x * s, x.y * s);
    o32[u] = *(const uint32_t*)&hh;
  }
  *(uint4*)(tile + swz(r, c)) = o;
}
__device__ __forceinline__ float bf8_max(uint4 raw) {
  const __nv_bfloat162* h2 = (const __nv_bfloat162*)&raw;
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 x = __bfloat1622float2(h2[u]);
    m = fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y)));
  }
  return m;
}
// line r, columns c0 .. c0 + 15 (two 16-byte granules) of a swizzled tile
__device__ __forceinline__ void st_row16(uint8_t* tile, int r, int c0, const float (&v)[16], float s) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint4 o;
    uint32_t* o32 = (uint32_t*)&o;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2 hh = __floats2half2_rn(v[8 * g + 2 * u] * s, v[8 * g + 2 * u + 1] * s);
      o32[u] = *(const uint32_t*)&hh;
    }
    *(uint4*)(tile + swz(r, c0 + 8 * g)) = o;
  }
}
__device__ __forceinline__ void ld_row16(const uint8_t* tile, int r, int c0, float (&v)[16]) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const uint4 o = *(const uint4*)(tile + swz(r, c0 + 8 * g));
    const __half2* h2 = (const __half2*)&o;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = __half22float2(h2[u]);
      v[8 * g + 2 * u] = x.x;
      v[8 * g + 2 * u + 1] = x.y;
    }
  }
}
__device__ __forceinline__ float elem(const uint8_t* tile, int r, int c) {
  return __half2float(*(const half*)(tile + swz(r, c)));
}
// p[t] (token t0 + t) summed over the warp's 32 lanes and added into
// dst[t0 + t]: a halving exchange leaves lanes 2u and 2u + 1 with token u
__device__ __forceinline__ void add_tokens(const float (&p)[16], float* dst, int t0) {
  const int lane = threadIdx.x & 31;
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float w8[8], w4[4], w2[2];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w8[i] = (b4 ? p[i + 8] : p[i]) + __shfl_xor_sync(0xffffffffu, b4 ? p[i] : p[i + 8], 16);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w4[i] = (b3 ? w8[i + 4] : w8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? w8[i] : w8[i + 4], 8);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    w2[i] = (b2 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? w4[i] : w4[i + 2], 4);
  float w1 = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
  w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
  if (!(lane & 1)) atomicAdd(dst + t0 + ((lane >> 1) & 15), w1);
}
}  // namespace tcb

__global__ void __launch_bounds__(tcb::NTH, 1) gdn_bwd_tc_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v, const float* __restrict__ dO,
    const float* __restrict__ S0, const float* __restrict__ dSC, const float* __restrict__ Li,
    const float* __restrict__ Pg, const float* __restrict__ Gb, const float* __restrict__ beta,
    const uint8_t* __restrict__ sel, int L, int N, float scale, float* __restrict__ dq, float* __restrict__ dk,
    float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta, int* __restrict__ err,
    long long nchunks, int ahead) {
  using namespace tcb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = tc::smem_u32(sm);
  float* sG = (float*)(sm + offVec);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* sdG = sB + C;
  float* sdB = sdG + C;
  float* red = (float*)(sm + offRed);
  uint64_t* bars = (uint64_t*)(sm + offBar);
  volatile int* fail = (volatile int*)(sm + offFlag);
  uint32_t* tslot = (uint32_t*)(sm + offTmem);
  const long long chunk = blockIdx.x;
  const int c = (int)(chunk % N);
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)c * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int f = 32 * (warp & 3) + lane;  // this thread's TMEM lane
  const int t0 = 16 * (warp >> 2);       // and its first column
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const bool committed = sel[chunk] != 0 && c < N - 1;
  // the rows the epilogues read late (v, and dq, dk, dv before their
  // updates) start towards L2 while the operand tiles load
  if (tid == 64) prefetch_l2(v + row0 * D, C * D * 2);
  if (tid == 96) prefetch_l2(dv + row0 * D, C * D * 4);
  if (tid == 128) prefetch_l2(dq + row0 * D, C * D * 4);
  if (tid == 160) prefetch_l2(dk + row0 * D, C * D * 4);
  // and the second group of operand tiles, read after the states' reduction
  if (tid == 256) prefetch_l2(k + row0 * D, C * D * 2);
  if (tid == 288) prefetch_l2(q + row0 * D, C * D * 2);
  if (tid == 320) prefetch_l2(dO + row0 * D, C * D * 4);
  if (tid == 352) prefetch_l2(Li + (size_t)chunk * C * C, C * C * 4);
  if (tid == 384) prefetch_l2(Pg + (size_t)chunk * C * C, C * C * 4);
  // and the states of the chunk `ahead` CTAs later (about one SM count: the
  // CTA that starts when one of the running ones ends)
  if (tid == 192 && chunk + ahead < nchunks) prefetch_l2(S0 + (size_t)(chunk + ahead) * D * D, D * D * 4);
  if (tid == 224 && chunk + ahead < nchunks && sel[chunk + ahead] != 0 && (chunk + ahead) % N < N - 1)
    prefetch_l2(dSC + (size_t)(chunk + ahead) * D * D, D * D * 4);
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
    tc::fence_before();
  }
  if (tid == 32) {
    for (int i = 0; i < 6; ++i) tc::mbar_init(&bars[i], 1);
    tc::fence_barrier_init();
    *fail = 0;
  }
  load_scalars(Gb, beta, row0, sG, sGam, sB);
  if (tid < C) sdG[tid] = sdB[tid] = 0.f;
  if (tid < 2) red[126 + tid] = 0.f;
  // S0 and dS_C (a committed chunk's; zero otherwise), read in the same
  // order so that <dS_C, S0> is taken in fp32 on the way
  float ss, sd;
  {
    constexpr int V = D * D / 4 / NTH;
    const float* s0 = S0 + (size_t)chunk * D * D;
    const float* ds = dSC + (size_t)chunk * D * D;
    float4 a[V], b[V];
    float m[2] = {0.f, 0.f}, sc2[2], dot = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = tid + NTH * i;
      a[i] = *(const float4*)(s0 + (size_t)(x / (D / 4)) * D + 4 * (x % (D / 4)));
      m[0] = fmaxf(m[0], max4(a[i]));
    }
    if (committed) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int x = tid + NTH * i;
        b[i] = *(const float4*)(ds + (size_t)(x / (D / 4)) * D + 4 * (x % (D / 4)));
        m[1] = fmaxf(m[1], max4(b[i]));
        dot += a[i].x * b[i].x + a[i].y * b[i].y + a[i].z * b[i].z + a[i].w * b[i].w;
      }
    }
    block_scalesN<2, NTH>(m, red, sc2);
    ss = sc2[0];
    sd = sc2[1];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int x = tid + NTH * i, r = x / (D / 4), cc = 4 * (x % (D / 4));
      st4(sm + offS, r, cc, a[i], ss);
      if (committed) st4(sm + offT, r, cc, b[i], sd);
    }
    if (committed) {
      dot = warp_sum(dot);
      if (lane == 0) atomicAdd(red + 127, dot);
    }
  }
  // k, q, dO, Linv (plain and with its columns scaled by beta) and P: every
  // load in flight together, one reduction for the six scales
  float sq, sk, so, sl, slb, sp;
  {
    constexpr int VB = C * D / 8 / NTH, VO = C * D / 4 / NTH, VC = C * C / 4 / NTH;
    uint4 kr[VB], qr[VB];
    float4 o[VO], l[VC], pp[VC];
    float m[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, s6[6];
    const float* lsrc = Li + (size_t)chunk * C * C;
    const float* psrc = Pg + (size_t)chunk * C * C;
#pragma unroll
    for (int i = 0; i < VB; ++i) {
      const int x = tid + NTH * i, r = x / (D / 8), cc = 8 * (x % (D / 8));
      kr[i] = *(const uint4*)(k + (row0 + r) * D + cc);
      qr[i] = *(const uint4*)(q + (row0 + r) * D + cc);
    }
#pragma unroll
    for (int i = 0; i < VO; ++i) {
      const int x = tid + NTH * i;
      o[i] = *(const float4*)(dO + (row0 + x / (D / 4)) * D + 4 * (x % (D / 4)));
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int x = tid + NTH * i;
      l[i] = *(const float4*)(lsrc + (x / (C / 4)) * C + 4 * (x % (C / 4)));
      pp[i] = *(const float4*)(psrc + (x / (C / 4)) * C + 4 * (x % (C / 4)));
    }
#pragma unroll
    for (int i = 0; i < VB; ++i) m[0] = fmaxf(m[0], bf8_max(kr[i])), m[1] = fmaxf(m[1], bf8_max(qr[i]));
#pragma unroll
    for (int i = 0; i < VO; ++i) m[2] = fmaxf(m[2], max4(o[i]));
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int cc = 4 * ((tid + NTH * i) % (C / 4));
      m[3] = fmaxf(m[3], max4(l[i]));
      m[4] = fmaxf(m[4], max4(make_float4(l[i].x * sB[cc], l[i].y * sB[cc + 1], l[i].z * sB[cc + 2],
                                          l[i].w * sB[cc + 3])));
      m[5] = fmaxf(m[5], max4(pp[i]));
    }
    block_scalesN<6, NTH>(m, red, s6);
    sk = s6[0], sq = s6[1], so = s6[2], sl = s6[3], slb = s6[4], sp = s6[5];
#pragma unroll
    for (int i = 0; i < VB; ++i) {
      const int x = tid + NTH * i, r = x / (D / 8), cc = 8 * (x % (D / 8));
      st_bf8(sm + offKQ, r, cc, kr[i], sk);
      st_bf8(sm + offKQ, C + r, cc, qr[i], sq);
    }
#pragma unroll
    for (int i = 0; i < VO; ++i) {
      const int x = tid + NTH * i;
      st4(sm + offYO, C + x / (D / 4), 4 * (x % (D / 4)), o[i], so);
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const int x = tid + NTH * i, r = x / (C / 4), cc = 4 * (x % (C / 4));
      st4(sm + offL, r, cc, l[i], sl);
      st4(sm + offLb, r, cc,
          make_float4(l[i].x * sB[cc], l[i].y * sB[cc + 1], l[i].z * sB[cc + 2], l[i].w * sB[cc + 3]), slb);
      st4(sm + offP, r, cc, pp[i], sp);
    }
  }
  // V of this thread's feature f and tokens t0 .., for the Vh epilogue
  float vv[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) vv[t] = __bfloat162float(v[(row0 + t0 + t) * D + f]);
  tc::fence_proxy_async_smem();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = *tslot;
  const uint32_t sS = sb + offS, sT = sb + offT, sYO = sb + offYO, sKQ = sb + offKQ, sVh = sb + offVh,
                 sU = sb + offU, sDU = sb + offDU, sL = sb + offL, sLb = sb + offLb, sP = sb + offP, sA = sb + offA;
  // a phase's products, issued by one thread; every thread then waits for them
  auto issue = [&](int bar, auto body) {
    if (tid == 0 && !*fail) {
      tc::fence_after();
      body();
      tc::mma_commit(&bars[bar]);
    }
  };
  auto wait = [&](int bar) {
    if (!*fail && !tc::mbar_wait(&bars[bar], 0, err)) *fail = 1;
    tc::fence_after();
  };
  auto ld = [&](uint32_t col, float (&x)[16]) {
    tc::tmem_ld16(tm + col + t0 + lane_off, x);
    tc::tmem_ld_wait();
  };
  // the end of an epilogue: its tile writes visible to the MMAs, its TMEM
  // reads done before the next phase may overwrite their columns
  auto phase_end = [&]() {
    tc::fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
  };
  const float gC = sGam[C - 1];
  // products that need only the loaded tiles: Vh^T = (K S0^T)^T, (dO S0)^T,
  // (K dS_C^T)^T, [K; Q] K^T
  issue(0, [&] {
    for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cVh, mnmaj(sS, kk), kmaj(sKQ, 0, kk), ID_MK, kk > 0);
    for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cDqA, kmaj(sS, 0, kk), kmaj(sYO, C, kk), ID_KK, kk > 0);
    if (committed)
      for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cDub, mnmaj(sT, kk), kmaj(sKQ, 0, kk), ID_MK, kk > 0);
    for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cKQ, kmaj(sKQ, 0, kk), kmaj(sKQ, 0, kk), ID_KK, kk > 0);
  });
  wait(0);
  float svh;
  {  // Vh = V - diag(gamma) K S0^T; dG_i += gamma_i (dO S0)_i . q~_i
    float a[16], b[16], part[16];
    ld(cVh, a);
    ld(cDqA, b);
    const float iks = 1.f / (sk * ss), ios = scale / (so * ss), iq = 1.f / sq;
    float mx = 0.f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      a[t] = vv[t] - sGam[t0 + t] * a[t] * iks;
      mx = fmaxf(mx, fabsf(a[t]));
      part[t] = sGam[t0 + t] * b[t] * ios * elem(sm + offKQ, C + t0 + t, f) * iq;
    }
    add_tokens(part, sdG, t0);
    svh = block_scale<NTH>(mx, red);
    st_row16(sm + offVh, f, t0, a, svh);
  }
  phase_end();
  // U^T = (Linv diag(beta) Vh)^T
  issue(1, [&] {
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cU, kmaj(sVh, 0, kk), kmaj(sLb, 0, kk), ID_KK, kk > 0);
  });
  wait(1);
  float su;
  {
    float a[16];
    ld(cU, a);
    const float iu = 1.f / (slb * svh);
    float mx = 0.f;
#pragma unroll
    for (int t = 0; t < 16; ++t) a[t] *= iu, mx = fmaxf(mx, fabsf(a[t]));
    su = block_scale<NTH>(mx, red);
    st_row16(sm + offU, f, t0, a, su);
  }
  phase_end();
  // dU^T = (P^T dO + K~ dS_C^T)^T
  issue(2, [&] {
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cDua, mnmaj(sYO + C * 128, kk), mnmaj(sP, kk), ID_MM, kk > 0);
  });
  wait(2);
  float sdu;
  {
    float a[16], b[16];
    ld(cDua, a);
    if (committed) ld(cDub, b);
    const float ipo = 1.f / (sp * so), ikd = 1.f / (sk * sd);
    float mx = 0.f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      a[t] = a[t] * ipo + (committed ? gC / sGam[t0 + t] * b[t] * ikd : 0.f);
      mx = fmaxf(mx, fabsf(a[t]));
    }
    sdu = block_scale<NTH>(mx, red);
    st_row16(sm + offDU, f, t0, a, sdu);
  }
  phase_end();
  // Y^T = (Linv^T dU)^T; dv += diag(beta) Y; dbeta_j = Y_j . Vh_j
  issue(3, [&] {
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cY, kmaj(sDU, 0, kk), mnmaj(sL, kk), ID_KM, kk > 0);
  });
  float sy;
  {
    float old[16];  // dv before its update, read while the product runs
#pragma unroll
    for (int t = 0; t < 16; ++t) old[t] = dv[(row0 + t0 + t) * D + f];
    wait(3);
    float y[16], vh[16], part[16];
    ld(cY, y);
    ld_row16(sm + offVh, f, t0, vh);
    const float iy = 1.f / (sl * sdu), ivh = 1.f / svh;
    float mx = 0.f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      y[t] *= iy;
      mx = fmaxf(mx, fabsf(y[t]));
      part[t] = y[t] * vh[t] * ivh;
      dv[(row0 + t0 + t) * D + f] = old[t] + sB[t0 + t] * y[t];
    }
    add_tokens(part, sdB, t0);
    sy = block_scale<NTH>(mx, red);
#pragma unroll
    for (int t = 0; t < 16; ++t) *(half*)(sm + offYO + swz(t0 + t, f)) = __float2half_rn(y[t] * sy);
  }
  phase_end();
  // [Y; dO] U^T: lanes 0-63 Y U^T (with K K^T from the first phase), lanes
  // 64-127 dP = dO U^T (with Q K^T)
  issue(4, [&] {
    for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cYO, kmaj(sYO, 0, kk), mnmaj(sU, kk), ID_KM, kk > 0);
  });
  wait(4);
  float sa, spm;
  {
    float x1[16], x2[16], cs[16], o[16];
    ld(cYO, x1);
    ld(cKQ, x2);
    float rs = 0.f, bs = 0.f, mx = 0.f;
    if (f < C) {  // row j = f: dL = -strict_lower(Y U^T), A = R . K K^T, dA = diag(beta) dL, A~ = dA . R
      const int j = f;
      const float iyu = 1.f / (sy * su), ikk = 1.f / (sk * sk);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int jj = t0 + t;
        cs[t] = 0.f;
        o[t] = 0.f;
        if (jj < j) {
          const float r = __expf(sG[j] - sG[jj]);
          const float A = r * x2[t] * ikk;
          const float dL = -x1[t] * iyu;
          const float dA = sB[j] * dL;
          const float x = dA * A;
          rs += x;
          bs += dL * A;
          cs[t] = -x;
          o[t] = dA * r;
        }
        mx = fmaxf(mx, fabsf(o[t]));
      }
      atomicAdd(sdB + j, bs);
    } else {  // row i = f - 64: dP = lower(dO U^T), P = R . Q~ K^T: dP . R; dG from dP . P
      const int i = f - C;
      const float iou = 1.f / (so * su), iqk = scale / (sq * sk);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int jj = t0 + t;
        cs[t] = 0.f;
        o[t] = 0.f;
        if (jj <= i) {
          const float r = __expf(sG[i] - sG[jj]);
          const float dP = x1[t] * iou;
          const float x = dP * (r * x2[t] * iqk);
          rs += x;
          cs[t] = -x;
          o[t] = dP * r;
        }
        mx = fmaxf(mx, fabsf(o[t]));
      }
    }
    atomicAdd(sdG + (f & (C - 1)), rs);
    add_tokens(cs, sdG, t0);
    float m2[2] = {f < C ? mx : 0.f, f < C ? 0.f : mx}, s2[2];
    block_scalesN<2, NTH>(m2, red, s2);
    sa = s2[0];
    spm = s2[1];
    if (f < C)
      st_row16(sm + offA, f, t0, o, sa);
    else
      st_row16(sm + offP, f - C, t0, o, spm);  // P was last read by the dU products
  }
  phase_end();
  // dq^T: (dP . R) K;  dk^T: U dS_C, Y S0, (dP . R)^T Q~, (A~ + A~^T) K
  issue(5, [&] {
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cDqB, mnmaj(sKQ, kk), kmaj(sP, 0, kk), ID_MK, kk > 0);
    if (committed)
      for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cDka, kmaj(sT, 0, kk), mnmaj(sU, kk), ID_KM, kk > 0);
    for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cDkb, kmaj(sS, 0, kk), kmaj(sYO, 0, kk), ID_KK, kk > 0);
    for (int kk = 0; kk < 4; ++kk)
      tc::mma_bf16(tm + cDkc, mnmaj(sKQ + C * 128, kk), mnmaj(sP, kk), ID_MM, kk > 0);
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cDkd, mnmaj(sKQ, kk), kmaj(sA, 0, kk), ID_MK, kk > 0);
    for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tm + cDkd, mnmaj(sKQ, kk), mnmaj(sA, kk), ID_MM, 1);
  });
  // dq and dk before their updates, read while the products run
  float oldq[16], oldk[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) oldq[t] = dq[(row0 + t0 + t) * D + f], oldk[t] = dk[(row0 + t0 + t) * D + f];
  wait(5);
  {  // dq += scale diag(gamma) dO S0 + scale (dP . R) K
    float a[16], b[16];
    float (&old)[16] = oldq;
    ld(cDqA, a);
    ld(cDqB, b);
    const float ios = scale / (so * ss), f2 = scale / (spm * sk);
#pragma unroll
    for (int t = 0; t < 16; ++t) dq[(row0 + t0 + t) * D + f] = old[t] + sGam[t0 + t] * a[t] * ios + b[t] * f2;
  }
  {  // dk; dG_j -= (U dS_C)_j . K~_j and gamma_j beta_j (Y S0)_j . k_j; the
     // last token gains sum_j (U dS_C)_j . K~_j
    float acc[16], x[16], part[16];
    float (&old)[16] = oldk;
    const float ik = 1.f / sk;
    float kf[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) kf[t] = elem(sm + offKQ, t0 + t, f) * ik, part[t] = 0.f;
    float tot = 0.f;
    if (committed) {
      ld(cDka, x);
      const float iud = 1.f / (su * sd);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float xa = gC / sGam[t0 + t] * x[t] * iud;
        acc[t] = xa;
        part[t] -= xa * kf[t];
        tot += xa * kf[t];
      }
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[t] = 0.f;
    }
    ld(cDkb, x);
    const float iys = 1.f / (sy * ss);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const float xb = sGam[t0 + t] * sB[t0 + t] * x[t] * iys;
      acc[t] -= xb;
      part[t] -= xb * kf[t];
    }
    ld(cDkc, x);
    const float f1 = scale / (spm * sq);
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] += f1 * x[t];
    ld(cDkd, x);
    const float fa = 1.f / (sa * sk);
#pragma unroll
    for (int t = 0; t < 16; ++t) dk[(row0 + t0 + t) * D + f] = old[t] + acc[t] + fa * x[t];
    add_tokens(part, sdG, t0);
    tot = warp_sum(tot);
    if (lane == 0) atomicAdd(red + 126, tot);
  }
  tc::fence_before();
  __syncthreads();
  if (tid == 0) sdG[C - 1] += red[126] + gC * red[127];
  __syncthreads();
  if (warp == 0) {  // dg = reverse cumulative sum of dG over the chunk
    const float a0 = sdG[2 * lane], a1 = sdG[2 * lane + 1];
    float s = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, s, o);
      if (lane + o < 32) s += y;
    }
    const float after = s - a0 - a1;  // s: the sum over lanes >= this one
    dg[row0 + 2 * lane + 1] = a1 + after;
    dg[row0 + 2 * lane] = a0 + a1 + after;
    tc::fence_after();
    tc::tmem_dealloc(tm, 512);
  }
  if (tid < C) dbeta[row0 + tid] = sdB[tid];
}

template <int D>
cudaError_t set_attributes() {
  static const cudaError_t attr = [] {
    cudaError_t r = cudaFuncSetAttribute(gdn_bwd_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PrepSm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_scan_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ScanSm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_fused_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               FusedSm<D>::kBytes);
    if (r == cudaSuccess && D == 128)
      r = cudaFuncSetAttribute(gdn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tcb::kBytes);
    return r;
  }();
  return attr;
}

template <int D>
cudaError_t run_factors(const Problem& p, const void* q, const void* k, const float* g, const float* beta,
                        const GdnBwdScratch& w, cudaStream_t st) {
  cudaError_t e = set_attributes<D>();
  if (e != cudaSuccess) return e;
  gdn_bwd_prep_kernel<D><<<(unsigned)(p.BH * p.N), 256, PrepSm<D>::kBytes, st>>>(
      (const bf16*)q, (const bf16*)k, g, beta, p.L, p.N, p.scale, w.G, w.Li, w.P, (half*)w.W16, (half*)w.Qe16,
      (half*)w.Kt16, w.sc);
  return cudaGetLastError();
}

template <int D>
cudaError_t run_reverse_scan(const Problem& p, const uint8_t* sel, const float* dO, const GdnBwdScratch& w,
                             cudaStream_t st) {
  cudaError_t e = set_attributes<D>();
  if (e != cudaSuccess) return e;
  gdn_bwd_scan_kernel<D><<<(unsigned)(p.BH * (D / RB)), 256, ScanSm<D>::kBytes, st>>>(
      (const half*)w.Kt16, (const half*)w.W16, (const half*)w.Qe16, w.sc, dO, w.G, sel, p.L, p.N, w.dSC);
  return cudaGetLastError();
}

template <int D>
cudaError_t run_products(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const uint8_t* sel, const float* dO, const GdnBwdScratch& w, float* dq,
                         float* dk, float* dv, float* dg, float* dbeta, int* err, cudaStream_t st) {
  cudaError_t e = set_attributes<D>();
  if (e != cudaSuccess) return e;
  if constexpr (D == 128) {  // on tcgen05
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    gdn_bwd_tc_kernel<<<(unsigned)(p.BH * p.N), tcb::NTH, tcb::kBytes, st>>>(
        (const bf16*)q, (const bf16*)k, (const bf16*)v, dO, w.S0, w.dSC, w.Li, w.P, w.G, beta, sel, p.L, p.N,
        p.scale, dq, dk, dv, dg, dbeta, err, p.BH * p.N, sms);
    return cudaGetLastError();
  }
  gdn_bwd_fused_kernel<D><<<(unsigned)(p.BH * p.N), 512, FusedSm<D>::kBytes, st>>>(
      (const bf16*)q, (const bf16*)k, (const bf16*)v, dO, w.S0, w.dSC, w.Li, w.P, w.G, beta, sel, p.L, p.N, p.scale,
      dq, dk, dv, dg, dbeta);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_bwd_factors(const Problem& p, const void* q, const void* k, const float* g,
                                   const float* beta, const GdnBwdScratch& w, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run_factors<64>(p, q, k, g, beta, w, st) : run_factors<128>(p, q, k, g, beta, w, st);
}

cudaError_t launch_gdn_bwd_reverse_scan(const Problem& p, const uint8_t* sel, const float* dO,
                                        const GdnBwdScratch& w, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run_reverse_scan<64>(p, sel, dO, w, st) : run_reverse_scan<128>(p, sel, dO, w, st);
}

cudaError_t launch_gdn_bwd_products(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                                    const float* beta, const uint8_t* sel, const float* dO, const GdnBwdScratch& w,
                                    float* dq, float* dk, float* dv, float* dg, float* dbeta, int* err,
                                    cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run_products<64>(p, q, k, v, g, beta, sel, dO, w, dq, dk, dv, dg, dbeta, err, st)
                   : run_products<128>(p, q, k, v, g, beta, sel, dO, w, dq, dk, dv, dg, dbeta, err, st);
}

}  // namespace nats
