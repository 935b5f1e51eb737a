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
// Kernels (after the forward scan has written every chunk's S0):
//   gdn_bwd_prep_kernel  per chunk: G, Linv, P (fp32), W, Q_eff, K~ (bf16)
//   gdn_bwd_scan_kernel  per (b, h, 32 state rows): the reverse scan, writing
//                        dS_C of every committed chunk (fp32)
//   gdn_bwd_s0_kernel    per chunk: Vh, U, P^T dO; dq += diag(gamma) dO S0
//   gdn_bwd_ds_kernel    per chunk: dU, Y, dv; the U dS_C and dVh S0 terms
//   gdn_bwd_cc_kernel    per chunk: the C x C products, dq, dk, dbeta, dg
// Products run on warp-level tensor cores (mma.sync m16n8k8, tf32 operands,
// fp32 accumulation); the triangular inverse is a forward substitution on
// the CUDA cores.  Each CTA has 8 warps; a C x D output is split into 16-row
// strips (warp w & 3) and column halves (warp w >> 2).
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int C = kChunk;
constexpr int CS = C + 4;  // fp32 row stride of C x C tiles
using bf16 = __nv_bfloat16;

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                     uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc[j] (rows m0 .. m0 + 15, columns n0 + 8 j .. + 7) += sum_k A(i, k) B(k, n)
template <int NT, int K, class FA, class FB>
__device__ __forceinline__ void wmm(float (&acc)[NT][4], int m0, int n0, FA fa, FB fb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a0 = tf32(fa(m0 + g, k0 + t)), a1 = tf32(fa(m0 + g + 8, k0 + t));
    const uint32_t a2 = tf32(fa(m0 + g, k0 + t + 4)), a3 = tf32(fa(m0 + g + 8, k0 + t + 4));
#pragma unroll
    for (int j = 0; j < NT; ++j)
      mma8(acc[j], a0, a1, a2, a3, tf32(fb(k0 + t, n0 + 8 * j + g)), tf32(fb(k0 + t + 4, n0 + 8 * j + g)));
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}

// f(row, col, value, index into the tile) for every accumulator element
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
  static constexpr int NT = D / 16; // n8 tiles per warp of a C x D output
};

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
// every asynchronous copy this thread issued has landed (then a block
// barrier makes them visible to the other threads)
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// cooperative asynchronous copies global -> shared (256 threads, 16 bytes each)
template <int D>
__device__ __forceinline__ void load_bf(bf16* dst, const bf16* src) {  // C x D
  constexpr int V = C * D / 8;
#pragma unroll
  for (int x = threadIdx.x; x < V; x += 256) {
    const int r = x / (D / 8), c8 = x % (D / 8);
    cp16(dst + r * Tiles<D>::BS + 8 * c8, src + (size_t)r * D + 8 * c8);
  }
}
template <int ROWS, int COLS, int LD>
__device__ __forceinline__ void load_f(float* dst, const float* src) {  // ROWS x COLS, source row stride COLS
  constexpr int V = ROWS * COLS / 4;
#pragma unroll
  for (int x = threadIdx.x; x < V; x += 256) {
    const int r = x / (COLS / 4), c4 = x % (COLS / 4);
    cp16(dst + r * LD + 4 * c4, src + (size_t)r * COLS + 4 * c4);
  }
}

__device__ __forceinline__ float bf(const bf16* p) { return __bfloat162float(*p); }

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

// ------------------------------------------------------------------ prep
template <int D>
struct PrepSm {
  using T = Tiles<D>;
  static constexpr int offQ = 0;
  static constexpr int offK = offQ + C * T::BS * 2;
  static constexpr int offA = offK + C * T::BS * 2;
  static constexpr int offLi = offA + C * CS * 4;
  static constexpr int offP = offLi + C * CS * 4;
  static constexpr int offW = offP + C * CS * 4;
  static constexpr int offV = offW + C * T::FS * 4;  // G, gamma, beta
  static constexpr int kBytes = offV + 3 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_prep_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k,
                                                           const float* __restrict__ g,
                                                           const float* __restrict__ beta, int L, int N, float scale,
                                                           float* __restrict__ Gb, float* __restrict__ Li_out,
                                                           float* __restrict__ P_out, bf16* __restrict__ W16,
                                                           bf16* __restrict__ Qe16, bf16* __restrict__ Kt16) {
  using T = Tiles<D>;
  using S = PrepSm<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  bf16* sQ = (bf16*)(sm + S::offQ);
  bf16* sK = (bf16*)(sm + S::offK);
  float* sA = (float*)(sm + S::offA);
  float* sLi = (float*)(sm + S::offLi);
  float* sP = (float*)(sm + S::offP);
  float* sW = (float*)(sm + S::offW);
  float* sG = (float*)(sm + S::offV);
  float* sGam = sG + C;
  float* sB = sGam + C;
  const long long chunk = blockIdx.x;
  const long long bh = chunk / N;
  const int c = (int)(chunk % N);
  const size_t row0 = (size_t)bh * L + (size_t)c * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  load_bf<D>(sQ, q + row0 * D);
  load_bf<D>(sK, k + row0 * D);
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
  cp_wait_all();
  __syncthreads();
  // beta A (strictly lower) and P (lower, diagonal included)
  {
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
    float kk[4][4], qk[4][4];
    zero(kk);
    zero(qk);
    wmm<4, D>(kk, m0, n0, [&](int i, int x) { return bf(sK + i * T::BS + x); },
              [&](int x, int j) { return bf(sK + j * T::BS + x); });
    wmm<4, D>(qk, m0, n0, [&](int i, int x) { return bf(sQ + i * T::BS + x); },
              [&](int x, int j) { return bf(sK + j * T::BS + x); });
    each(kk, m0, n0, [&](int i, int j, float v, int, int) {
      sA[i * CS + j] = j < i ? sB[i] * __expf(sG[i] - sG[j]) * v : 0.f;
    });
    each(qk, m0, n0, [&](int i, int j, float v, int, int) {
      sP[i * CS + j] = j <= i ? scale * __expf(sG[i] - sG[j]) * v : 0.f;
    });
  }
  __syncthreads();
  // Linv = (I + beta A)^{-1} by forward substitution, one column per thread
  if (tid < C) {
    const int j = tid;
    float x[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
      float s = i == j ? 1.f : 0.f;
#pragma unroll
      for (int m4 = 0; m4 < i / 4; ++m4) {
        const float4 a = *(const float4*)(sA + i * CS + 4 * m4);
        s -= a.x * x[4 * m4] + a.y * x[4 * m4 + 1] + a.z * x[4 * m4 + 2] + a.w * x[4 * m4 + 3];
      }
#pragma unroll
      for (int m = (i / 4) * 4; m < i; ++m) s -= sA[i * CS + m] * x[m];
      x[i] = s;
    }
#pragma unroll
    for (int i = 0; i < C; ++i) sLi[i * CS + j] = x[i];
  }
  __syncthreads();
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
  // W = Linv diag(beta gamma) K
  {
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, C>(acc, m0, n0, [&](int i, int m) { return sLi[i * CS + m] * sB[m] * sGam[m]; },
                  [&](int m, int n) { return bf(sK + m * T::BS + n); });
    each(acc, m0, n0, [&](int i, int n, float v, int, int) {
      sW[i * T::FS + n] = v;
      W16[(row0 + i) * D + n] = __float2bfloat16_rn(v);
    });
  }
  __syncthreads();
  // Q_eff = diag(gamma) Q~ - P W, and K~ = diag(gamma_C / gamma) K
  {
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, C>(acc, m0, n0, [&](int i, int m) { return sP[i * CS + m]; },
                  [&](int m, int n) { return sW[m * T::FS + n]; });
    const float gC = sGam[C - 1];
    each(acc, m0, n0, [&](int i, int n, float v, int, int) {
      Qe16[(row0 + i) * D + n] = __float2bfloat16_rn(sGam[i] * scale * bf(sQ + i * T::BS + n) - v);
      Kt16[(row0 + i) * D + n] = __float2bfloat16_rn(gC / sGam[i] * bf(sK + i * T::BS + n));
    });
  }
  // Linv and P for the per-chunk gradient kernels
  for (int x = tid; x < C * C / 4; x += 256) {
    const int i = x / (C / 4), j4 = x % (C / 4);
    *(float4*)(Li_out + (size_t)chunk * C * C + i * C + 4 * j4) = *(const float4*)(sLi + i * CS + 4 * j4);
    *(float4*)(P_out + (size_t)chunk * C * C + i * C + 4 * j4) = *(const float4*)(sP + i * CS + 4 * j4);
  }
}

// ------------------------------------------------------------------ scan
constexpr int RB = 32;  // state-gradient rows per CTA

template <int D>
struct ScanSm {
  using T = Tiles<D>;
  static constexpr int kTile = C * T::BS * 2;
  static constexpr int kO = C * (RB + 4) * 4;
  static constexpr int kStage = 3 * kTile + kO;
  static constexpr int offS = 2 * kStage;          // fp32 [RB][FS]
  static constexpr int offX = offS + RB * T::FS * 4; // fp32 [RB][CS]
  static constexpr int kBytes = offX + RB * CS * 4;
};

template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_scan_kernel(const bf16* __restrict__ Kt16,
                                                           const bf16* __restrict__ W16,
                                                           const bf16* __restrict__ Qe16,
                                                           const float* __restrict__ dO, const float* __restrict__ Gb,
                                                           const uint8_t* __restrict__ sel, int L, int N,
                                                           float* __restrict__ dSC) {
  using T = Tiles<D>;
  using S = ScanSm<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sdS = (float*)(sm + S::offS);
  float* sX = (float*)(sm + S::offX);
  constexpr int splits = D / RB;
  const long long bh = blockIdx.x / splits;
  const int r0 = (blockIdx.x % splits) * RB;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int x = tid; x < RB * T::FS; x += 256) sdS[x] = 0.f;
  auto stage_ptr = [&](int s, int which) { return sm + s * S::kStage + which * S::kTile; };
  auto prefetch = [&](int c) {
    const int s = c & 1;
    const size_t row0 = (size_t)bh * L + (size_t)c * C;
    const bf16* srcs[3] = {Kt16, W16, Qe16};
#pragma unroll
    for (int w3 = 0; w3 < 3; ++w3) {
      bf16* dst = (bf16*)stage_ptr(s, w3);
      for (int x = tid; x < C * D / 8; x += 256) {
        const int r = x / (D / 8), c8 = x % (D / 8);
        cp16(dst + r * T::BS + 8 * c8, srcs[w3] + (row0 + r) * D + 8 * c8);
      }
    }
    float* dO_s = (float*)stage_ptr(s, 3);
    for (int x = tid; x < C * RB / 4; x += 256) {
      const int r = x / (RB / 4), c4 = x % (RB / 4);
      cp16(dO_s + r * (RB + 4) + 4 * c4, dO + (row0 + r) * D + r0 + 4 * c4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if (N > 0) prefetch(N - 1);
  for (int c = N - 1; c >= 0; --c) {
    if (c > 0) {
      prefetch(c - 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int s = c & 1;
    const bf16* sKt = (const bf16*)stage_ptr(s, 0);
    const bf16* sW = (const bf16*)stage_ptr(s, 1);
    const bf16* sQe = (const bf16*)stage_ptr(s, 2);
    const float* sO = (const float*)stage_ptr(s, 3);
    const bool lin = sel[bh * N + c] != 0;
    // dS_C of a committed chunk (the last chunk's is zero and is not read)
    if (lin && c < N - 1) {
      float* dst = dSC + (((size_t)bh * N + c) * D + r0) * D;
      for (int x = tid; x < RB * D / 4; x += 256) {
        const int i = x / (D / 4), c4 = x % (D / 4);
        *(float4*)(dst + (size_t)i * D + 4 * c4) = *(const float4*)(sdS + i * T::FS + 4 * c4);
      }
    }
    if (lin) {  // X = dS K~^T (RB x C)
      const int m0 = 16 * (warp & 1), n0 = 16 * (warp >> 1);
      float acc[2][4];
      zero(acc);
      wmm<2, D>(acc, m0, n0, [&](int i, int x) { return sdS[i * T::FS + x]; },
                [&](int x, int n) { return bf(sKt + n * T::BS + x); });
      each(acc, m0, n0, [&](int i, int n, float v, int, int) { sX[i * CS + n] = v; });
      __syncthreads();
    }
    {  // dS <- gamma_C dS - X W + dO^T Q_eff (committed), dS + dO^T Q_eff (rolled back)
      constexpr int NT = D / 32;
      const int m0 = 16 * (warp & 1), n0 = (warp >> 1) * (D / 4);
      float acc[NT][4];
      zero(acc);
      if (lin)
        wmm<NT, C>(acc, m0, n0, [&](int i, int m) { return -sX[i * CS + m]; },
                   [&](int m, int n) { return bf(sW + m * T::BS + n); });
      wmm<NT, C>(acc, m0, n0, [&](int i, int m) { return sO[m * (RB + 4) + i]; },
                 [&](int m, int n) { return bf(sQe + m * T::BS + n); });
      const float gC = lin ? __expf(Gb[(size_t)bh * L + (size_t)c * C + C - 1]) : 1.f;
      each(acc, m0, n0, [&](int i, int n, float v, int, int) { sdS[i * T::FS + n] = gC * sdS[i * T::FS + n] + v; });
    }
    __syncthreads();
  }
}

// -------------------------------------------------------- products with S0
template <int D>
struct S0Sm {
  using T = Tiles<D>;
  static constexpr int offS = 0;                          // fp32 [D][FS]
  static constexpr int offK = offS + D * T::FS * 4;       // bf16 [C][BS]
  static constexpr int offV = offK + C * T::BS * 2;
  static constexpr int offO = offV + C * T::BS * 2;       // fp32 [C][FS]
  static constexpr int offLi = offO + C * T::FS * 4;      // fp32 [C][CS]
  static constexpr int offP = offLi + C * CS * 4;
  static constexpr int offVh = offP + C * CS * 4;         // fp32 [C][FS]
  static constexpr int offVec = offVh + C * T::FS * 4;    // G, gamma, beta, dG
  static constexpr int kBytes = offVec + 4 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_s0_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v, const float* __restrict__ dO,
    const float* __restrict__ S0, const float* __restrict__ Li, const float* __restrict__ Pg,
    const float* __restrict__ Gb, const float* __restrict__ beta, int L, int N, float scale, float* __restrict__ Vh,
    float* __restrict__ Ug, float* __restrict__ PtdO, float* __restrict__ dq, float* __restrict__ dGs) {
  using T = Tiles<D>;
  using S = S0Sm<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sS = (float*)(sm + S::offS);
  bf16* sK = (bf16*)(sm + S::offK);
  bf16* sV = (bf16*)(sm + S::offV);
  float* sO = (float*)(sm + S::offO);
  float* sLi = (float*)(sm + S::offLi);
  float* sP = (float*)(sm + S::offP);
  float* sVh = (float*)(sm + S::offVh);
  float* sG = (float*)(sm + S::offVec);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* sdG = sB + C;
  const long long chunk = blockIdx.x;
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)(chunk % N) * C;
  const int tid = threadIdx.x, warp = tid >> 5;
  load_f<D, D, T::FS>(sS, S0 + (size_t)chunk * D * D);
  load_bf<D>(sK, k + row0 * D);
  load_bf<D>(sV, v + row0 * D);
  load_f<C, D, T::FS>(sO, dO + row0 * D);
  load_f<C, C, CS>(sLi, Li + (size_t)chunk * C * C);
  load_f<C, C, CS>(sP, Pg + (size_t)chunk * C * C);
  load_scalars(Gb, beta, row0, sG, sGam, sB);
  if (tid < C) sdG[tid] = 0.f;
  cp_wait_all();
  __syncthreads();
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
  {  // Vh = V - diag(gamma) K S0^T
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, D>(acc, m0, n0, [&](int i, int x) { return bf(sK + i * T::BS + x); },
                  [&](int x, int n) { return sS[n * T::FS + x]; });
    each(acc, m0, n0, [&](int i, int n, float val, int, int) {
      const float vh = bf(sV + i * T::BS + n) - sGam[i] * val;
      sVh[i * T::FS + n] = vh;
      Vh[(row0 + i) * D + n] = vh;
    });
  }
  {  // dO S0: dq += scale gamma_i (dO S0)_i; dG_i += gamma_i (dO S0)_i . q~_i
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, D>(acc, m0, n0, [&](int i, int a) { return sO[i * T::FS + a]; },
                  [&](int a, int n) { return sS[a * T::FS + n]; });
    float lo = 0.f, hi = 0.f;
    each(acc, m0, n0, [&](int i, int n, float val, int, int e) {
      const size_t o = (row0 + i) * D + n;
      dq[o] += scale * sGam[i] * val;
      const float d = scale * sGam[i] * val * __bfloat162float(q[o]);
      if (e < 2) lo += d; else hi += d;
    });
    add_rows(lo, hi, m0, sdG);
  }
  __syncthreads();
  {  // U = Linv diag(beta) Vh
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, C>(acc, m0, n0, [&](int i, int m) { return sLi[i * CS + m] * sB[m]; },
                  [&](int m, int n) { return sVh[m * T::FS + n]; });
    each(acc, m0, n0, [&](int i, int n, float val, int, int) { Ug[(row0 + i) * D + n] = val; });
  }
  {  // P^T dO
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, C>(acc, m0, n0, [&](int i, int m) { return sP[m * CS + i]; },
                  [&](int m, int n) { return sO[m * T::FS + n]; });
    each(acc, m0, n0, [&](int i, int n, float val, int, int) { PtdO[(row0 + i) * D + n] = val; });
  }
  __syncthreads();
  if (tid < C) dGs[row0 + tid] = sdG[tid];
}

// ----------------------------------------------------- products with dS_C
template <int D>
struct DsSm {
  using T = Tiles<D>;
  static constexpr int offS = 0;                          // fp32 [D][FS]: dS_C, then S0
  static constexpr int offK = offS + D * T::FS * 4;       // bf16 [C][BS]
  static constexpr int offU = offK + C * T::BS * 2;       // fp32 [C][FS]
  static constexpr int offLi = offU + C * T::FS * 4;      // fp32 [C][CS]
  static constexpr int offD = offLi + C * CS * 4;         // fp32 [C][FS]: dU, then Y
  static constexpr int offVec = offD + C * T::FS * 4;     // G, gamma, beta, dG, dbeta, reduction
  static constexpr int kBytes = offVec + 6 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_ds_kernel(
    const bf16* __restrict__ k, const float* __restrict__ S0, const float* __restrict__ dSC,
    const float* __restrict__ Ug, const float* __restrict__ Li, const float* __restrict__ PtdO,
    const float* __restrict__ Vh, const float* __restrict__ Gb, const float* __restrict__ beta,
    const uint8_t* __restrict__ sel, int L, int N, float* __restrict__ Yg, float* __restrict__ dv,
    float* __restrict__ dk, float* __restrict__ dGs, float* __restrict__ dbeta) {
  using T = Tiles<D>;
  using S = DsSm<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sS = (float*)(sm + S::offS);
  bf16* sK = (bf16*)(sm + S::offK);
  float* sU = (float*)(sm + S::offU);
  float* sLi = (float*)(sm + S::offLi);
  float* sD = (float*)(sm + S::offD);
  float* sG = (float*)(sm + S::offVec);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* sdG = sB + C;
  float* sdB = sdG + C;
  float* sRed = sdB + C;
  const long long chunk = blockIdx.x;
  const int c = (int)(chunk % N);
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)c * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool committed = sel[chunk] != 0 && c < N - 1;
  load_bf<D>(sK, k + row0 * D);
  load_f<C, D, T::FS>(sU, Ug + row0 * D);
  load_f<C, C, CS>(sLi, Li + (size_t)chunk * C * C);
  load_f<C, D, T::FS>(sD, PtdO + row0 * D);
  if (committed) load_f<D, D, T::FS>(sS, dSC + (size_t)chunk * D * D);
  load_scalars(Gb, beta, row0, sG, sGam, sB);
  if (tid < C) sdG[tid] = sdB[tid] = 0.f;
  if (tid == 0) sRed[0] = 0.f;
  cp_wait_all();
  __syncthreads();
  const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
  if (committed) {
    const float gC = sGam[C - 1];
    {  // dU += K~ dS_C^T
      float acc[T::NT][4];
      zero(acc);
      wmm<T::NT, D>(acc, m0, n0, [&](int i, int x) { return gC / sGam[i] * bf(sK + i * T::BS + x); },
                    [&](int x, int a) { return sS[a * T::FS + x]; });
      each(acc, m0, n0, [&](int i, int a, float val, int, int) { sD[i * T::FS + a] += val; });
    }
    {  // U dS_C: dk += diag(gamma_C / gamma) (U dS_C); dG_j -= (U dS_C)_j . K~_j; the last token gains their sum
      float acc[T::NT][4];
      zero(acc);
      wmm<T::NT, D>(acc, m0, n0, [&](int i, int a) { return sU[i * T::FS + a]; },
                    [&](int a, int n) { return sS[a * T::FS + n]; });
      float lo = 0.f, hi = 0.f;
      each(acc, m0, n0, [&](int i, int n, float val, int, int e) {
        const float f = gC / sGam[i];
        dk[(row0 + i) * D + n] += f * val;
        const float d = val * f * bf(sK + i * T::BS + n);
        if (e < 2) lo -= d; else hi -= d;
      });
      float tot = -(lo + hi);
      add_rows(lo, hi, m0, sdG);
      tot = warp_sum(tot);
      if (lane == 0) atomicAdd(sRed, tot);
    }
    {  // gamma_C <dS_C, S0> into the last token
      const float* s0 = S0 + (size_t)chunk * D * D;
      float acc = 0.f;
      for (int x = tid; x < D * D / 4; x += 256) {
        const int a = x / (D / 4), c4 = x % (D / 4);
        const float4 u = *(const float4*)(sS + a * T::FS + 4 * c4);
        const float4 w = *(const float4*)(s0 + (size_t)a * D + 4 * c4);
        acc += u.x * w.x + u.y * w.y + u.z * w.z + u.w * w.w;
      }
      acc = warp_sum(acc);
      if (lane == 0) atomicAdd(sRed, gC * acc);
    }
  }
  __syncthreads();
  if (tid == 0) sdG[C - 1] += sRed[0];
  // Y = Linv^T dU; dv += diag(beta) Y; dbeta_i = Y_i . Vh_i
  float accY[T::NT][4];
  zero(accY);
  wmm<T::NT, C>(accY, m0, n0, [&](int i, int m) { return sLi[m * CS + i]; },
                [&](int m, int n) { return sD[m * T::FS + n]; });
  __syncthreads();  // every read of dU is done
  {
    float lo = 0.f, hi = 0.f;
    each(accY, m0, n0, [&](int i, int n, float y, int, int e) {
      const size_t o = (row0 + i) * D + n;
      sD[i * T::FS + n] = y;
      Yg[o] = y;
      dv[o] += sB[i] * y;
      const float d = y * Vh[o];
      if (e < 2) lo += d; else hi += d;
    });
    add_rows(lo, hi, m0, sdB);
  }
  // S0 for the dVh S0 term (every read of dS_C ended at the barrier above)
  load_f<D, D, T::FS>(sS, S0 + (size_t)chunk * D * D);
  cp_wait_all();
  __syncthreads();
  {  // dk -= diag(gamma) dVh S0; dG_i -= gamma_i (dVh S0)_i . k_i
    float acc[T::NT][4];
    zero(acc);
    wmm<T::NT, D>(acc, m0, n0, [&](int i, int a) { return sB[i] * sD[i * T::FS + a]; },
                  [&](int a, int n) { return sS[a * T::FS + n]; });
    float lo = 0.f, hi = 0.f;
    each(acc, m0, n0, [&](int i, int n, float val, int, int e) {
      dk[(row0 + i) * D + n] -= sGam[i] * val;
      const float d = sGam[i] * val * bf(sK + i * T::BS + n);
      if (e < 2) lo -= d; else hi -= d;
    });
    add_rows(lo, hi, m0, sdG);
  }
  __syncthreads();
  if (tid < C) {
    dGs[row0 + tid] += sdG[tid];
    dbeta[row0 + tid] = sdB[tid];
  }
}

// ---------------------------------------------------- C x C products, dg
template <int D>
struct CcSm {
  using T = Tiles<D>;
  static constexpr int offQ = 0;                          // bf16 [C][BS]
  static constexpr int offK = offQ + C * T::BS * 2;
  static constexpr int offO = offK + C * T::BS * 2;       // fp32 [C][FS]
  static constexpr int offU = offO + C * T::FS * 4;
  static constexpr int offY = offU + C * T::FS * 4;
  static constexpr int offA = offY + C * T::FS * 4;       // fp32 [C][CS]: A~
  static constexpr int offP = offA + C * CS * 4;          // fp32 [C][CS]: dP . R
  static constexpr int offVec = offP + C * CS * 4;        // G, gamma, beta, dG, dbeta
  static constexpr int kBytes = offVec + 5 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(256) gdn_bwd_cc_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const float* __restrict__ dO,
    const float* __restrict__ Ug, const float* __restrict__ Yg, const float* __restrict__ Gb,
    const float* __restrict__ beta, int L, int N, float scale, float* __restrict__ dq, float* __restrict__ dk,
    const float* __restrict__ dGs, float* __restrict__ dbeta, float* __restrict__ dg) {
  using T = Tiles<D>;
  using S = CcSm<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  bf16* sQ = (bf16*)(sm + S::offQ);
  bf16* sK = (bf16*)(sm + S::offK);
  float* sO = (float*)(sm + S::offO);
  float* sU = (float*)(sm + S::offU);
  float* sY = (float*)(sm + S::offY);
  float* sA = (float*)(sm + S::offA);
  float* sP = (float*)(sm + S::offP);
  float* sG = (float*)(sm + S::offVec);
  float* sGam = sG + C;
  float* sB = sGam + C;
  float* sdG = sB + C;
  float* sdB = sdG + C;
  const long long chunk = blockIdx.x;
  const size_t row0 = (size_t)(chunk / N) * L + (size_t)(chunk % N) * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  load_bf<D>(sQ, q + row0 * D);
  load_bf<D>(sK, k + row0 * D);
  load_f<C, D, T::FS>(sO, dO + row0 * D);
  load_f<C, D, T::FS>(sU, Ug + row0 * D);
  load_f<C, D, T::FS>(sY, Yg + row0 * D);
  load_scalars(Gb, beta, row0, sG, sGam, sB);
  if (tid < C) sdG[tid] = sdB[tid] = 0.f;
  cp_wait_all();
  __syncthreads();
  {
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
    // dL = -strict_lower(Y U^T), A = R . K K^T: dA = diag(beta) dL, A~ = dA . R,
    // dbeta_i += sum_j dL_ij A_ij, dG += row sums - column sums of dA . A
    {
      float yu[4][4], kk[4][4];
      zero(yu);
      zero(kk);
      wmm<4, D>(yu, m0, n0, [&](int i, int a) { return sY[i * T::FS + a]; },
                [&](int a, int j) { return sU[j * T::FS + a]; });
      wmm<4, D>(kk, m0, n0, [&](int i, int x) { return bf(sK + i * T::BS + x); },
                [&](int x, int j) { return bf(sK + j * T::BS + x); });
      float rlo = 0.f, rhi = 0.f, blo = 0.f, bhi = 0.f, col[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) col[j][0] = col[j][1] = 0.f;
      each(yu, m0, n0, [&](int i, int jj, float val, int j, int e) {
        float at = 0.f;
        if (jj < i) {
          const float r = __expf(sG[i] - sG[jj]);
          const float A = r * kk[j][e];
          const float dL = -val;
          const float dA = sB[i] * dL;
          const float x = dA * A;
          if (e < 2) rlo += x, blo += dL * A; else rhi += x, bhi += dL * A;
          col[j][e & 1] -= x;
          at = dA * r;
        }
        sA[i * CS + jj] = at;
      });
      add_rows(rlo, rhi, m0, sdG);
      add_rows(blo, bhi, m0, sdB);
      add_cols<4>(col, n0, sdG);
    }
    // dP = lower(dO U^T), P = R . Q~ K^T: dPm = dP . R, dG += row sums - column sums of dP . P
    {
      float ou[4][4], qk[4][4];
      zero(ou);
      zero(qk);
      wmm<4, D>(ou, m0, n0, [&](int i, int a) { return sO[i * T::FS + a]; },
                [&](int a, int j) { return sU[j * T::FS + a]; });
      wmm<4, D>(qk, m0, n0, [&](int i, int x) { return bf(sQ + i * T::BS + x); },
                [&](int x, int j) { return bf(sK + j * T::BS + x); });
      float rlo = 0.f, rhi = 0.f, col[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) col[j][0] = col[j][1] = 0.f;
      each(ou, m0, n0, [&](int i, int jj, float val, int j, int e) {
        float pm = 0.f;
        if (jj <= i) {
          const float r = __expf(sG[i] - sG[jj]);
          const float P = r * scale * qk[j][e];
          const float x = val * P;
          if (e < 2) rlo += x; else rhi += x;
          col[j][e & 1] -= x;
          pm = val * r;
        }
        sP[i * CS + jj] = pm;
      });
      add_rows(rlo, rhi, m0, sdG);
      add_cols<4>(col, n0, sdG);
    }
  }
  __syncthreads();
  {
    const int m0 = 16 * (warp & 3), n0 = (warp >> 2) * (D / 2);
    {  // dq += scale (dP . R) K
      float acc[T::NT][4];
      zero(acc);
      wmm<T::NT, C>(acc, m0, n0, [&](int i, int j) { return sP[i * CS + j]; },
                    [&](int j, int n) { return bf(sK + j * T::BS + n); });
      each(acc, m0, n0, [&](int i, int n, float val, int, int) { dq[(row0 + i) * D + n] += scale * val; });
    }
    {  // dk += (dP . R)^T Q~ + (A~ + A~^T) K
      float acc[T::NT][4];
      zero(acc);
      wmm<T::NT, C>(acc, m0, n0, [&](int i, int j) { return sP[j * CS + i]; },
                    [&](int j, int n) { return scale * bf(sQ + j * T::BS + n); });
      wmm<T::NT, C>(acc, m0, n0, [&](int i, int j) { return sA[i * CS + j] + sA[j * CS + i]; },
                    [&](int j, int n) { return bf(sK + j * T::BS + n); });
      each(acc, m0, n0, [&](int i, int n, float val, int, int) { dk[(row0 + i) * D + n] += val; });
    }
  }
  __syncthreads();
  if (warp == 0) {  // dg = reverse cumulative sum of dG over the chunk
    const float a0 = sdG[2 * lane] + dGs[row0 + 2 * lane];
    const float a1 = sdG[2 * lane + 1] + dGs[row0 + 2 * lane + 1];
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
  if (tid < C) dbeta[row0 + tid] += sdB[tid];
}

template <int D>
cudaError_t run(const Problem& p, const void* q, const void* k, const void* v, const float* g, const float* beta,
                const uint8_t* sel, const float* dO, const GdnBwdScratch& w, float* dq, float* dk, float* dv,
                float* dg, float* dbeta, cudaStream_t st, int32_t* launches) {
  const long long chunks = p.BH * p.N;
  cudaError_t e;
  static const cudaError_t attr = [] {
    cudaError_t r = cudaFuncSetAttribute(gdn_bwd_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PrepSm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_scan_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ScanSm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_s0_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S0Sm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_ds_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DsSm<D>::kBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(gdn_bwd_cc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, CcSm<D>::kBytes);
    return r;
  }();
  if (attr != cudaSuccess) return attr;
  const bf16* qb = (const bf16*)q;
  const bf16* kb = (const bf16*)k;
  const bf16* vb = (const bf16*)v;
  gdn_bwd_prep_kernel<D><<<(unsigned)chunks, 256, PrepSm<D>::kBytes, st>>>(qb, kb, g, beta, p.L, p.N, p.scale, w.G,
                                                                          w.Li, w.P, w.W16, w.Qe16, w.Kt16);
  gdn_bwd_scan_kernel<D><<<(unsigned)(p.BH * (D / RB)), 256, ScanSm<D>::kBytes, st>>>(w.Kt16, w.W16, w.Qe16, dO,
                                                                                      w.G, sel, p.L, p.N, w.dSC);
  gdn_bwd_s0_kernel<D><<<(unsigned)chunks, 256, S0Sm<D>::kBytes, st>>>(qb, kb, vb, dO, w.S0, w.Li, w.P, w.G, beta,
                                                                      p.L, p.N, p.scale, w.Vh, w.U, w.PtdO, dq,
                                                                      w.dG);
  gdn_bwd_ds_kernel<D><<<(unsigned)chunks, 256, DsSm<D>::kBytes, st>>>(kb, w.S0, w.dSC, w.U, w.Li, w.PtdO, w.Vh,
                                                                      w.G, beta, sel, p.L, p.N, w.Y, dv, dk, w.dG,
                                                                      dbeta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (launches) *launches += 4;
  return cudaSuccess;
}

template <int D>
cudaError_t run_cc(const Problem& p, const void* q, const void* k, const float* beta, const float* dO,
                   const GdnBwdScratch& w, float* dq, float* dk, float* dg, float* dbeta, cudaStream_t st) {
  gdn_bwd_cc_kernel<D><<<(unsigned)(p.BH * p.N), 256, CcSm<D>::kBytes, st>>>(
      (const bf16*)q, (const bf16*)k, dO, w.U, w.Y, w.G, beta, p.L, p.N, p.scale, dq, dk, w.dG, dbeta, dg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_bwd_chunk(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const uint8_t* sel, const float* dO, const GdnBwdScratch& w,
                                 float* dq, float* dk, float* dv, float* dg, float* dbeta, cudaStream_t st,
                                 int32_t* launches) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run<64>(p, q, k, v, g, beta, sel, dO, w, dq, dk, dv, dg, dbeta, st, launches)
                   : run<128>(p, q, k, v, g, beta, sel, dO, w, dq, dk, dv, dg, dbeta, st, launches);
}

cudaError_t launch_gdn_bwd_cc(const Problem& p, const void* q, const void* k, const float* beta, const float* dO,
                              const GdnBwdScratch& w, float* dq, float* dk, float* dg, float* dbeta,
                              cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? run_cc<64>(p, q, k, beta, dO, w, dq, dk, dg, dbeta, st)
                   : run_cc<128>(p, q, k, beta, dO, w, dq, dk, dg, dbeta, st);
}

}  // namespace nats
