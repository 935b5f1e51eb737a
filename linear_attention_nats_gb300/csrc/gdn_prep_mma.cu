// gdn_prep_mma.cu - Gated DeltaNet phase 1 on warp-level tensor-core MMAs
// (bf16 inputs, d = 64; d = 128 uses the tcgen05 pipeline of gdn_prep_tc.cu):
// the per-chunk factors of the chunkwise WY/UT form, parallel over chunks.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3 (both states are pseudo-updated for every chunk);
// Gated DeltaNet S_t = a_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
// For one chunk (G = in-chunk cumulative sum of g):
//   A = strict_lower(beta_t e^{G_t - G_i} k_t . k_i),  T = (I + A)^{-1}
//   U = T diag(beta) V,  W = T diag(beta e^G) K,  P = lower_incl(scale e^{G_t - G_i} q_t . k_i)
// KK^T / QK^T and T.(beta V) / T.(beta e^G K) are warp-level bf16 MMAs
// (fp32 accumulate); the unit-lower-triangular inverse is fp32, blocked in
// 16 x 16 tiles.  Outputs (the operands of the chunk scan): W bf16
// [chunk][64][D]; U transposed, bf16 [chunk][D][64]; P bf16 [chunk][64][64];
// G fp32; and the merge gate of each token, w = sigmoid(q . W_g[h] + b_g[h])
// ("Kernmechanismen" item 4: weights generated from the query), fp32.
// Optionally it also scores the chunk ("Kernmechanismen" item 1: mean pool of
// [q ; k] over the chunk, one linear score per operation, the higher score
// wins, ties to softmax), from the Q and K it has staged anyway, so the
// layer forward needs no separate pass over Q and K for the selection.
#include "common.cuh"
#include "kernels.h"

namespace nats {
namespace {

constexpr int C = kChunk;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8 fp32) += A(16x8 tf32, row) * B(8x8 tf32, col)
__device__ __forceinline__ void mma1688_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// hardware barrier of `count` threads (whole warps) under barrier id `id`
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D>
struct PrepSmem {
  static constexpr int RS = D + 8;  // bf16 row stride (16-byte skew: conflict-free ldmatrix)
  static constexpr int TS = C + 8;  // bf16 row stride of T
  static constexpr int offK = 0;
  static constexpr int offQ = offK + C * RS * 2;
  static constexpr int offV = offQ + C * RS * 2;
  static constexpr int FS = C + 4;  // fp32 row stride (16-byte aligned rows)
  static constexpr int offA = offV + C * RS * 2;     // fp32 [C][FS]
  static constexpr int offT = offA + C * FS * 4;     // fp32 [C][FS]
  static constexpr int offTb = offT + C * FS * 4;    // bf16 [C][TS]
  static constexpr int offG = offTb + C * TS * 2;    // fp32 [C]
  static constexpr int offB = offG + C * 4;          // fp32 [C] beta
  static constexpr int offBg = offB + C * 4;         // fp32 [C] beta e^G
  static constexpr int offX = offBg + C * 4;         // fp32 [C][FS] scratch of the blocked inverse
  static constexpr int offRed = offX + C * FS * 4;   // fp32 [2][4] per-warp partial chunk scores, [2] bias
  static constexpr int kBytes = offRed + 64;
};

// One CTA (8 warps) per (b, h, chunk).  Warp w = (wr, wh), wr = w % 4 owns
// rows 16 wr .. 16 wr + 15 of the 64-row products; wh = w / 4 picks the
// column half of K K^T / Q K^T, and U (wh = 0) or W (wh = 1) in the last
// product, so the two run side by side.
template <int D>
__global__ void __launch_bounds__(256, 2) gdn_prep_mma_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ g, const float* __restrict__ beta, int L,
    int N, float scale, float* __restrict__ Gout, __nv_bfloat16* __restrict__ Wout,
    __nv_bfloat16* __restrict__ Uout, __nv_bfloat16* __restrict__ Pout, const float* __restrict__ w_g, const float* __restrict__ b_g, int H,
    float* __restrict__ gate_out, const float* __restrict__ w_s, const float* __restrict__ b_s,
    uint8_t* __restrict__ sel_out, float* __restrict__ T_out) {
  using S = PrepSmem<D>;
  constexpr int RS = S::RS, TS = S::TS, FS = S::FS;
  constexpr int NT = 256;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* Ks = (__nv_bfloat16*)(smem + S::offK);
  __nv_bfloat16* Qs = (__nv_bfloat16*)(smem + S::offQ);
  __nv_bfloat16* Vs = (__nv_bfloat16*)(smem + S::offV);
  float* As = (float*)(smem + S::offA);
  float* Ts = (float*)(smem + S::offT);
  __nv_bfloat16* Tb = (__nv_bfloat16*)(smem + S::offTb);
  float* Gs = (float*)(smem + S::offG);
  float* Bs = (float*)(smem + S::offB);
  float* Bg = (float*)(smem + S::offBg);
  float* Xs = (float*)(smem + S::offX);
  float* red = (float*)(smem + S::offRed);
  constexpr int UTS = C + 8;  // bf16 line stride of the staged U^T
  __nv_bfloat16* UTs = (__nv_bfloat16*)(smem + S::offA);  // reuses A and T once T is in Tb
  static_assert(D * UTS * 2 <= 2 * C * S::FS * 4, "U^T staging must fit the A / T scratch");
  __nv_bfloat16* Wst = (__nv_bfloat16*)(smem + S::offX);  // W staged in the inverse scratch
  static_assert(C * RS * 2 <= C * S::FS * 4, "W staging must fit the inverse scratch");

  const long long blk = blockIdx.x;
  const int c = (int)(blk % N);
  const long long bh = blk / N;
  const int h = (int)(bh % H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wr = warp & 3, wh = warp >> 2;
  const int gq = lane >> 2, cq = lane & 3;  // fragment row / column-pair
  const size_t tok0 = (size_t)bh * L + (size_t)c * C;

  // ---- stage K, Q, V (16-byte async copies) and the gates
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  for (int e = tid; e < C * VPR; e += NT) {
    const int t = e / VPR, x = e % VPR;
    cp_async16(Ks + t * RS + x * 8, k + (tok0 + t) * D + x * 8);
    cp_async16(Qs + t * RS + x * 8, q + (tok0 + t) * D + x * 8);
    cp_async16(Vs + t * RS + x * 8, v + (tok0 + t) * D + x * 8);
  }
  if (warp == 0) {
    const float g0 = g[tok0 + 2 * lane], g1 = g[tok0 + 2 * lane + 1];
    float x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const float excl = x - (g0 + g1);
    Gs[2 * lane] = excl + g0;
    Gs[2 * lane + 1] = excl + g0 + g1;
    Gout[tok0 + 2 * lane] = excl + g0;
    Gout[tok0 + 2 * lane + 1] = excl + g0 + g1;
  } else if (warp == 1) {
    Bs[2 * lane] = beta[tok0 + 2 * lane];
    Bs[2 * lane + 1] = beta[tok0 + 2 * lane + 1];
    if (lane < 2) red[8 + lane] = (sel_out && b_s) ? b_s[2 * h + lane] : 0.f;  // score bias, for the end
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- KK^T and QK^T for rows 16 wr .. 16 wr + 15, columns 32 wh .. 32 wh + 31
  const int m0 = 16 * wr;
  {
    float kk[4][4], qk[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int x = 0; x < 4; ++x) kk[j][x] = qk[j][x] = 0.f;
    const int arow = m0 + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int acol = 8 * (lane >> 4);
    const int brow = (lane & 7) + 8 * (lane >> 4);
    const int bcol = 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t ka[4], qa[4];
      ldsm_x4(smem_addr(Ks + arow * RS + 16 * ks + acol), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(smem_addr(Qs + arow * RS + 16 * ks + acol), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
      for (int jq = 0; jq < 2; ++jq) {  // key rows 16 jp .. 16 jp + 15 = two n-tiles
        const int jp = 2 * wh + jq;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_addr(Ks + (16 * jp + brow) * RS + 16 * ks + bcol), b0, b1, b2, b3);
        mma16816(kk[2 * jq], ka[0], ka[1], ka[2], ka[3], b0, b1);
        mma16816(kk[2 * jq + 1], ka[0], ka[1], ka[2], ka[3], b2, b3);
        mma16816(qk[2 * jq], qa[0], qa[1], qa[2], qa[3], b0, b1);
        mma16816(qk[2 * jq + 1], qa[0], qa[1], qa[2], qa[3], b2, b3);
      }
    }
    // decay, masks; A -> shared fp32, P -> global bf16
    __nv_bfloat16* P = Pout + (size_t)blk * C * C;
#pragma unroll
    for (int jl = 0; jl < 4; ++jl) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int t = m0 + gq + 8 * hh;
        const int i0 = 8 * (4 * wh + jl) + 2 * cq;
        float av[2], pv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = i0 + u;
          const float dec = __expf(Gs[t] - Gs[i]);
          av[u] = (i < t) ? Bs[t] * dec * kk[jl][2 * hh + u] : 0.f;
          pv[u] = (i <= t) ? scale * dec * qk[jl][2 * hh + u] : 0.f;
        }
        As[t * FS + i0] = av[0];
        As[t * FS + i0 + 1] = av[1];
        *(uint32_t*)(P + t * C + i0) = pack2(pv[0], pv[1]);
      }
    }
  }
  __syncthreads();
  // ---- two warp groups side by side: both depend only on the products
  // above, and each synchronises on its own named barrier (every thread of a
  // group reaches every barrier of its group)
  if (warp >= 4) {
    // warps 4-7: merge gate, the column sums of Q and K for the chunk score,
    // then V rows *= beta and K rows *= beta e^G
    const int t4 = tid - 128;
    {
      // merge gate: two threads per token, D/2 features each
      const int t = t4 >> 1, hh = t4 & 1;
      const float* wg = w_g + (size_t)h * D + hh * (D / 2);
      const __nv_bfloat16* qr = Qs + t * RS + hh * (D / 2);
      float z = 0.f;
#pragma unroll
      for (int x8 = 0; x8 < D / 16; ++x8) {
        const uint4 qv = *(const uint4*)(qr + 8 * x8);
        const __nv_bfloat162* q2 = (const __nv_bfloat162*)&qv;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(q2[i]);
          z = fmaf(f.x, wg[8 * x8 + 2 * i], fmaf(f.y, wg[8 * x8 + 2 * i + 1], z));
        }
      }
      z += __shfl_xor_sync(0xffffffffu, z, 1);
      if (hh == 0) gate_out[tok0 + t] = 1.f / (1.f + __expf(-(z + (b_g ? b_g[h] : 0.f))));
    }
    {
      // column sums of Q and K for the chunk score; a thread keeps one
      // 8-column group x = t4 % VPR over its rows
      float cs[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) cs[x] = 0.f;
      for (int e = t4; e < C * VPR; e += 128) {
        const int t = e / VPR, x = e % VPR;
        const uint4 inq = *(const uint4*)(Qs + t * RS + x * 8);
        const uint4 ink = *(const uint4*)(Ks + t * RS + x * 8);
        const __nv_bfloat162* hq = (const __nv_bfloat162*)&inq;
        const __nv_bfloat162* hk = (const __nv_bfloat162*)&ink;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 vq = __bfloat1622float2(hq[i]);
          const float2 vk = __bfloat1622float2(hk[i]);
          cs[2 * i] += vq.x;
          cs[2 * i + 1] += vq.y;
          cs[8 + 2 * i] += vk.x;
          cs[8 + 2 * i + 1] += vk.y;
        }
      }
      if (sel_out) {
        // chunk score, linear in the column sums: combine the threads of the
        // warp that share x, dot each group with the score weights, reduce
        // over the warp; the four warps' partials are added after the join
#pragma unroll
        for (int o = VPR; o < 32; o <<= 1)
#pragma unroll
          for (int x = 0; x < 16; ++x) cs[x] += __shfl_xor_sync(0xffffffffu, cs[x], o);
        float s0 = 0.f, s1 = 0.f;
        if (lane < VPR) {
          const float* W = w_s + (size_t)h * 4 * D + 8 * lane;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            s0 = fmaf(W[cc], cs[cc], fmaf(W[D + cc], cs[8 + cc], s0));
            s1 = fmaf(W[2 * D + cc], cs[cc], fmaf(W[3 * D + cc], cs[8 + cc], s1));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (lane == 0) {
          red[warp - 4] = s0;
          red[warp] = s1;  // 4 + (warp - 4)
        }
      }
    }
    if (t4 < C) Bg[t4] = Bs[t4] * __expf(Gs[t4]);
    named_barrier(2, 128);
    // V rows *= beta, K rows *= beta e^G (in place, 8 columns per step)
    for (int e = t4; e < C * VPR; e += 128) {
      const int t = e / VPR, x8 = (e % VPR) * 8;
      const float fb = Bs[t], fg = Bg[t];
      uint4 vv = *(uint4*)(Vs + t * RS + x8);
      uint4 kv = *(uint4*)(Ks + t * RS + x8);
      __nv_bfloat162* v2 = (__nv_bfloat162*)&vv;
      __nv_bfloat162* k2 = (__nv_bfloat162*)&kv;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 a2 = __bfloat1622float2(v2[x]);
        const float2 c2 = __bfloat1622float2(k2[x]);
        v2[x] = __floats2bfloat162_rn(a2.x * fb, a2.y * fb);
        k2[x] = __floats2bfloat162_rn(c2.x * fg, c2.y * fg);
      }
      *(uint4*)(Vs + t * RS + x8) = vv;
      *(uint4*)(Ks + t * RS + x8) = kv;
    }
  } else {
    // warps 0-3: T = (I + A)^{-1}, unit lower triangular, blocked in 16 x 16 tiles:
    //   T_bb = (I + A_bb)^{-1}                          (forward substitution, fp32)
    //   T_ij = -T_ii sum_{j <= k < i} A_ik T_kj  (i > j, by distance i - j)
    if (tid < C) {
      // diagonal tile b, column jj: a 16-long dependency chain in registers
      const int b = tid >> 4, jj = tid & 15, j = 16 * b + jj;
      float x[16];
#pragma unroll
      for (int tt = 0; tt < 16; ++tt) {
        const int t = 16 * b + tt;
        float acc = (tt == jj) ? 1.f : 0.f;
#pragma unroll
        for (int ii = 0; ii < tt; ++ii)
          if (ii >= jj) acc = fmaf(-As[t * FS + 16 * b + ii], x[ii], acc);
        x[tt] = (tt >= jj) ? acc : 0.f;
      }
#pragma unroll
      for (int tt = 0; tt < 16; ++tt) Ts[(16 * b + tt) * FS + j] = x[tt];
    }
    named_barrier(1, 128);
    // off-diagonal tiles on tf32 MMAs (fp32 accumulate; T is rounded to bf16
    // for the U / W products right after, far coarser than the tf32
    // operands), blocked in two levels so that the chain is four products:
    //   halves a = rows 0-31, b = rows 32-63:  T = [[T_a, 0], [T_ba, T_b]]
    //   level 1: T_10 = -T_11 (A_10 T_00), T_32 = -T_33 (A_32 T_22)
    //   level 2: Y = A_ba T_a, then T_ba = -T_b Y (four 16 x 16 tiles each)
    // acc (16 x 16, two n-tiles) += M1[r0.., c0 .. c0+klen) * M2[c0'.., n0 ..]
    auto tile_mma = [&](float (&acc)[2][4], const float* M1, int r0, int c0, const float* M2, int k0, int n0,
                        int klen) {
      for (int kk = 0; kk < klen; kk += 8) {
        const float* ar = M1 + (r0 + gq) * FS + c0 + kk + cq;
        const uint32_t a0 = tf32(ar[0]), a1 = tf32(ar[8 * FS]), a2 = tf32(ar[4]), a3 = tf32(ar[8 * FS + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float* br = M2 + (k0 + kk + cq) * FS + n0 + 8 * nt + gq;
          mma1688_tf32(acc[nt], a0, a1, a2, a3, tf32(br[0]), tf32(br[4 * FS]));
        }
      }
    };
    auto tile_store = [&](float* M, int r0, int n0, const float (&acc)[2][4], float sgn) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float* dr = M + (r0 + gq) * FS + n0 + 8 * nt + 2 * cq;
        dr[0] = sgn * acc[nt][0];
        dr[1] = sgn * acc[nt][1];
        dr[8 * FS] = sgn * acc[nt][2];
        dr[8 * FS + 1] = sgn * acc[nt][3];
      }
    };
    if (warp < 2) {
      // level 1: tile (i, j) = (2w + 1, 2w)
      const int i = 2 * warp + 1, j = 2 * warp;
      float x[2][4] = {};
      tile_mma(x, As, 16 * i, 16 * j, Ts, 16 * j, 16 * j, 16);  // A_ij T_jj
      tile_store(Xs, 16 * i, 16 * j, x, 1.f);
      __syncwarp();
      float y[2][4] = {};
      tile_mma(y, Ts, 16 * i, 16 * i, Xs, 16 * i, 16 * j, 16);  // T_ii X_ij
      tile_store(Ts, 16 * i, 16 * j, y, -1.f);
    }
    named_barrier(1, 128);
    // level 2, warp w owns tile (i, j) = (2 + w / 2, w % 2) of the lower-left block
    const int li = 2 + (warp >> 1), lj = warp & 1;
    {
      // Y_ij = sum_{k = j..1} A_ik T_kj   (T_a is lower triangular)
      float yv[2][4] = {};
      tile_mma(yv, As, 16 * li, 16 * lj, Ts, 16 * lj, 16 * lj, 16 * (2 - lj));
      tile_store(Xs, 16 * li, 16 * lj, yv, 1.f);
    }
    named_barrier(1, 128);
    {
      // T_ij = -sum_{k = 2..i} T_ik Y_kj   (T_b is lower triangular)
      float tv[2][4] = {};
      tile_mma(tv, Ts, 16 * li, 32, Xs, 32, 16 * lj, 16 * (li - 1));
      tile_store(Ts, 16 * li, 16 * lj, tv, -1.f);
    }
    named_barrier(1, 128);
    // T -> bf16 (zero above the diagonal), 8 columns per step
    for (int e = tid; e < C * C / 8; e += 128) {
      const int t = e >> 3, j0 = (e & 7) * 8;
      const float4 a0 = *(const float4*)(Ts + t * FS + j0);
      const float4 a1 = *(const float4*)(Ts + t * FS + j0 + 4);
      const float v8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      uint4 o;
      uint32_t* o32 = (uint32_t*)&o;
#pragma unroll
      for (int x = 0; x < 4; ++x)
        o32[x] = pack2(j0 + 2 * x <= t ? v8[2 * x] : 0.f, j0 + 2 * x + 1 <= t ? v8[2 * x + 1] : 0.f);
      *(uint4*)(Tb + t * TS + j0) = o;
      if (T_out) {  // T in fp32 for the backward pass
        float* dst = T_out + (size_t)blk * C * C + t * C + j0;
#pragma unroll
        for (int x = 0; x < 8; ++x) dst[x] = j0 + x <= t ? v8[x] : 0.f;
      }
    }
  }
  __syncthreads();
  // ---- U = T (beta V) on warps wh = 0, W = T (beta e^G K) on warps wh = 1:
  // rows 16 wr .., k-steps up to the diagonal
  {
    const int arow = m0 + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int acol = 8 * (lane >> 4);
    const int trow = (lane & 7) + 8 * ((lane >> 3) & 1);  // k row within the 16-row step
    const int tcol = 8 * (lane >> 4);                     // n column offset
    const __nv_bfloat16* Bsrc = wh == 0 ? Vs : Ks;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[n][x] = 0.f;
    for (int ks = 0; ks <= wr; ++ks) {
      uint32_t a[4];
      ldsm_x4(smem_addr(Tb + arow * TS + 16 * ks + acol), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_addr(Bsrc + (16 * ks + trow) * RS + 16 * np + tcol), b0, b1, b2, b3);
        mma16816(acc[2 * np], a[0], a[1], a[2], a[3], b0, b1);
        mma16816(acc[2 * np + 1], a[0], a[1], a[2], a[3], b2, b3);
      }
    }
    if (wh == 0) {
      // U^T staged in the (now dead) A / T scratch: line e, column t
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int e = 8 * n + 2 * cq;
        UTs[e * UTS + m0 + gq] = __float2bfloat16_rn(acc[n][0]);
        UTs[(e + 1) * UTS + m0 + gq] = __float2bfloat16_rn(acc[n][1]);
        UTs[e * UTS + m0 + gq + 8] = __float2bfloat16_rn(acc[n][2]);
        UTs[(e + 1) * UTS + m0 + gq + 8] = __float2bfloat16_rn(acc[n][3]);
      }
    } else {
      // W staged in the (now dead) inverse scratch
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int col = 8 * n + 2 * cq;
        *(uint32_t*)(Wst + (m0 + gq) * RS + col) = pack2(acc[n][0], acc[n][1]);
        *(uint32_t*)(Wst + (m0 + gq + 8) * RS + col) = pack2(acc[n][2], acc[n][3]);
      }
    }
  }
  __syncthreads();
  {
    __nv_bfloat16* Ug = Uout + (size_t)blk * C * D;  // [D][64]
    for (int e8 = tid; e8 < D * 8; e8 += NT) {
      const int e = e8 >> 3, x = e8 & 7;
      *(uint4*)(Ug + e * C + x * 8) = *(const uint4*)(UTs + e * UTS + x * 8);
    }
    __nv_bfloat16* Wg = Wout + (size_t)blk * C * D;  // [64][D]
    for (int e = tid; e < C * VPR; e += NT) {
      const int t = e / VPR, x = e % VPR;
      *(uint4*)(Wg + t * D + x * 8) = *(const uint4*)(Wst + t * RS + x * 8);
    }
  }
  if (sel_out && tid == 0) {
    // chunk score = (1/C) w_s . (column sums of [Q ; K]) + b_s; ties to softmax
    // (done last: no warp waits for it)
    const float a = ((red[0] + red[1]) + (red[2] + red[3])) * (1.0f / C) + red[8];
    const float bb = ((red[4] + red[5]) + (red[6] + red[7])) * (1.0f / C) + red[9];
    sel_out[blk] = (a >= bb) ? 0 : 1;
  }
}

}  // namespace

cudaError_t launch_gdn_prep_mma(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* w_g, const float* b_g, float* G, void* W16,
                                void* U16, void* P16, float* gate, const float* w_s, const float* b_s,
                                uint8_t* sel_out, float* T_out, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(p.BH * p.N), 256, smem, st>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, g, beta, p.L, p.N, p.scale,
        G, (__nv_bfloat16*)W16, (__nv_bfloat16*)U16, (__nv_bfloat16*)P16, w_g, b_g, p.H, gate, w_s, b_s,
        sel_out, T_out);
    return cudaGetLastError();
  };
  // d = 128 takes the tcgen05 pipeline (gdn_prep_tc.cu)
  if (p.d != 64) return cudaErrorInvalidValue;
  return run(gdn_prep_mma_kernel<64>, PrepSmem<64>::kBytes);
}

}  // namespace nats
