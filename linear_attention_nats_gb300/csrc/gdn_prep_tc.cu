// gdn_prep_tc.cu - Gated DeltaNet phase 1 on the 5th-generation tensor cores
// (bf16, d = 128): the per-chunk factors of the chunkwise WY/UT form, as a
// persistent, warp-specialised pipeline over the chunks.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3 (both states are pseudo-updated for every chunk);
// Gated DeltaNet S_t = a_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
// For one chunk (G = in-chunk cumulative sum of g):
//   A = strict_lower(beta_t e^{G_t - G_i} k_t . k_i),  T = (I + A)^{-1}
//   U = T diag(beta) V,  W = T diag(beta e^G) K,  P = lower_incl(scale e^{G_t - G_i} q_t . k_i)
// plus G, the merge gate
// w = sigmoid(q . W_g[h] + b_g[h]) ("Kernmechanismen" item 4) and, when asked,
// the chunk's selection ("Kernmechanismen" item 1: mean pool of [q ; k], one
// linear score per operation, the higher wins, ties to softmax).  The outputs
// and their layouts are those of the warp-MMA kernel in gdn_prep_mma.cu (the
// chunk scan forms the decayed Q~ and K~ itself, from Q, K and G).
//
// One CTA per SM walks the chunks blockIdx.x, + gridDim.x, ...; chunk i uses
// slot j = i % 2 of every double buffer (input stage, TMEM accumulators, the
// bf16 T tile).  Roles (448 threads):
//   warp 0       TMA of K, Q, V (the K and Q tiles of a 64-column half side by
//                side, so [K; Q] is one 128-line MMA operand) and the chunk's
//                scalars G, beta, beta e^G, G log2(e)
//   warp 1       TMEM owner and MMA issuer:
//                  [K; Q] K^T            (M = 128, N = 64, K = d) -> KK^T | QK^T
//                  U^T = (beta V)^T T^T  and  W^T = (beta e^G K)^T T^T
//                                        (M = d, N = 64, K = 64, A read
//                                         feature-major from the same tiles)
//   warps 2-5    gate and the score's column sums; then, once the first
//                product has read K, beta e^G K in place
//   warps 6-9    A (fp32, shared) and P (bf16, TMA store) from KK^T / QK^T;
//                then T = (I + A)^{-1} blocked in 16 x 16 tiles, as bf16
//   warps 10-13  U^T and W^T from TMEM through swizzled tiles to TMA stores;
//                beta V in place, one chunk ahead
// The first product of chunk i + 1 is issued before the second of chunk i, so
// the inverse warps never wait for it.  Every wait is bounded
// (tc::kWaitLimitNs); a warp group agrees on giving up through a barrier
// reduction, so no named barrier is left with missing threads.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {

bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D);

namespace {

constexpr int C = kChunk;
constexpr int D = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int FS = C + 4;  // fp32 row stride of A, T and the inverse scratch

struct PrepTcSmem {
  // input stage: [K_h0 | Q_h0 | K_h1 | Q_h1 | V_h0 | V_h1] (8 KiB boxes of 64
  // lines x 64 columns, 128-byte swizzle), then four fp32 [C] scalar rows
  static constexpr int kKQ = 4 * 8192;
  static constexpr int kV = 2 * 8192;
  static constexpr int kScal = 4 * C * 4;
  static constexpr int kStage = 51200;  // kKQ + kV + kScal rounded up to 1 KiB
  static_assert(kKQ + kV + kScal <= kStage, "stage");
  static constexpr int kStages = 2;
  static constexpr int offA = kStages * kStage;      // 2 x fp32 [C][FS] (A of chunks i % 2)
  static constexpr int offT = offA + 2 * C * FS * 4; // fp32 [C][FS]
  static constexpr int offX = offT + C * FS * 4;     // fp32 [C][FS] scratch of the blocked inverse
  static constexpr int offTb = offX + C * FS * 4;    // 2 x bf16 [C][C] swizzled (MMA operand)
  static constexpr int offP = offTb + 2 * 8192;      // bf16 [C][C] swizzled (TMA store)
  static constexpr int offW = offP + 8192;           // bf16 U^T [D][C], then W [C][D], as two 64-line boxes (TMA stores)
  static constexpr int offRed = offW + 16384;        // fp32 [2][8] per-warp partial chunk scores
  static constexpr int offBar = offRed + 64;
  static constexpr int kNumBars = 21;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;  // + alignment slack of the dynamic smem base
  static_assert(offTb % 1024 == 0 && offP % 1024 == 0 && offW % 1024 == 0, "1 KiB tiles");
};

// slot j = i % 2 of each pair
enum {
  B_FULL = 0, B_EMPTY = 2, B_KQF = 4, B_KQE = 6, B_ELF = 8, B_TBF = 10, B_UWF = 12, B_UWE = 14,
  B_AF = 16,  // A of the chunk written (epilogue warps -> inverse warps)
  B_AE = 18,  // A of the chunk read for the last time (inverse warps -> epilogue warps)
  B_DONE = 20
};

// TMEM columns
constexpr uint32_t kColKQ = 0;    // 2 x 64: lanes 0-63 KK^T rows, lanes 64-127 QK^T rows
constexpr uint32_t kColUW = 128;  // 2 x 128: U^T (64 columns) then W^T (64 columns), lane = feature

// warp roles
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpEl = 2, kWarpInv = 6, kWarpUw = 10, kWarpEpi = 14, kThreads = 576;
// named barriers (0 is __syncthreads)
constexpr int kBarEl = 1, kBarInv = 2, kBarUw = 3, kBarEpi = 4;

using tc::group_all;
using tc::named_barrier;

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

// two bf16 (low half first) as a packed fp32 pair (exact)
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
  return tc::f2_pack(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// byte offset of the 16-byte granule g (columns 8g .. 8g + 7) of line t in a
// 128-byte-swizzled box
__device__ __forceinline__ uint32_t sw_gran(int t, int g) { return (uint32_t)(t * 128 + ((g ^ (t & 7)) << 4)); }

__global__ void __launch_bounds__(kThreads, 1)
    gdn_prep_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_p,
                       const float* __restrict__ g, const float* __restrict__ beta, int L, int N, int H,
                       long long nchunks, float scale, float* __restrict__ Gout, const float* __restrict__ w_g, const float* __restrict__ b_g, float* __restrict__ gate_out,
                       const float* __restrict__ w_s, const float* __restrict__ b_s, uint8_t* __restrict__ sel_out,
                       int* __restrict__ err, float* __restrict__ T_out) {
  using S = PrepTcSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int j = 0; j < 2; ++j) {
      tc::mbar_init(&bars[B_FULL + j], 2);  // expect_tx arrival + scalars arrival
      tc::mbar_init(&bars[B_EMPTY + j], 1);
      tc::mbar_init(&bars[B_KQF + j], 1);
      tc::mbar_init(&bars[B_KQE + j], 4);
      tc::mbar_init(&bars[B_ELF + j], 8);  // K (warps 2-5) and V (warps 10-13) scaled
      tc::mbar_init(&bars[B_TBF + j], 4);
      tc::mbar_init(&bars[B_UWF + j], 1);
      tc::mbar_init(&bars[B_UWE + j], 4);
      tc::mbar_init(&bars[B_AF + j], 4);
      tc::mbar_init(&bars[B_AE + j], 4);
    }
    tc::mbar_init(&bars[B_DONE], 1);
    tc::fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long stride = gridDim.x;
  // number of chunks this CTA processes
  const int nmine = blockIdx.x < nchunks ? (int)((nchunks - 1 - blockIdx.x) / stride + 1) : 0;
  auto stage = [&](int j) { return smem + j * S::kStage; };
  // (b h, chunk, head) of the chunks this CTA walks, advanced by gridDim.x
  // chunks per step with adds only (no per-step integer division)
  struct Pos {
    int blk, bh, c, h;
  };
  const int adv_bh = (int)gridDim.x / N, adv_c = (int)gridDim.x - adv_bh * N, adv_h = adv_bh % H;
  auto first_pos = [&]() {
    Pos p;
    p.blk = (int)blockIdx.x;
    p.bh = p.blk / N;
    p.c = p.blk - p.bh * N;
    p.h = p.bh % H;
    return p;
  };
  auto next_pos = [&](Pos& p) {
    p.blk += (int)gridDim.x;
    p.c += adv_c;
    p.bh += adv_bh;
    p.h += adv_h;
    if (p.c >= N) {
      p.c -= N;
      ++p.bh;
      ++p.h;
    }
    if (p.h >= H) p.h -= H;
  };
  // G, beta, beta e^G, G log2(e)
  auto scal = [&](int j) { return (float*)(smem + j * S::kStage + S::kKQ + S::kV); };

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_v);
    }
    bool ok = true;
    Pos pos = first_pos();
    for (int i = 0; i < nmine; ++i, next_pos(pos)) {
      const int j = i & 1, k = i >> 1;
      const long long tok0 = (long long)pos.bh * L + (long long)pos.c * C;
      // g and beta of the chunk (two tokens per lane), read before the wait
      const float g0 = g[tok0 + 2 * lane], g1 = g[tok0 + 2 * lane + 1];
      const float b0 = beta[tok0 + 2 * lane], b1 = beta[tok0 + 2 * lane + 1];
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_EMPTY + j], (k & 1) ^ 1, err)))) break;
      uint8_t* st = stage(j);
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(&bars[B_FULL + j], S::kKQ + S::kV);
        for (int h = 0; h < 2; ++h) {
          tc::tma_load_2d(st + h * 16384, &tm_k, 64 * h, (int)tok0, &bars[B_FULL + j]);
          tc::tma_load_2d(st + h * 16384 + 8192, &tm_q, 64 * h, (int)tok0, &bars[B_FULL + j]);
          tc::tma_load_2d(st + S::kKQ + h * 8192, &tm_v, 64 * h, (int)tok0, &bars[B_FULL + j]);
        }
      }
      // G = in-chunk inclusive cumsum of g
      float x = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float G0 = x - g1, G1 = x;
      float* sc = scal(j);
      sc[2 * lane] = G0;
      sc[2 * lane + 1] = G1;
      sc[C + 2 * lane] = b0;
      sc[C + 2 * lane + 1] = b1;
      sc[2 * C + 2 * lane] = b0 * __expf(G0);
      sc[2 * C + 2 * lane + 1] = b1 * __expf(G1);
      sc[3 * C + 2 * lane] = G0 * kLog2e;
      sc[3 * C + 2 * lane + 1] = G1 * kLog2e;
      *(float2*)(Gout + tok0 + 2 * lane) = make_float2(G0, G1);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_FULL + j]);
    }
    // drain: the stages' loads have landed and their last readers are done
    if (lane == 0) {
      for (int i = nmine - 2 < 0 ? 0 : nmine - 2; i < nmine; ++i) {
        const int j = i & 1, k = i >> 1;
        tc::mbar_wait(&bars[B_FULL + j], k & 1, nullptr);
        if (ok) tc::mbar_wait(&bars[B_EMPTY + j], k & 1, err);
      }
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_kq = tc::idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id_uw = tc::idesc_bf16_f32(128, 64, true, false);
      const uint32_t s0 = tc::smem_u32(smem);
      const uint64_t kq0 = tc::smem_desc_sw128(s0, 16, 1024);                // [K; Q] and K, feature-major lines
      const uint64_t va0 = tc::smem_desc_sw128(s0 + S::kKQ, 8192, 1024);     // (beta V)^T: halves 8 KiB apart
      const uint64_t ka0 = tc::smem_desc_sw128(s0, 16384, 1024);             // (beta e^G K)^T: halves 16 KiB apart
      const uint64_t tb0 = tc::smem_desc_sw128(s0 + S::offTb, 16, 1024);     // T, lines t, columns j
      bool ok = true;
      auto issue_kq = [&](int i) -> bool {
        const int j = i & 1, k = i >> 1;
        if (!tc::mbar_wait(&bars[B_FULL + j], k & 1, err)) return false;
        if (i >= 2 && !tc::mbar_wait(&bars[B_KQE + j], (k - 1) & 1, err)) return false;
        tc::fence_after();
        const uint32_t sb = j * S::kStage;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = sb + (kk >> 2) * 16384 + (kk & 3) * 32;
          tc::mma_bf16(tmem + kColKQ + j * 64, tc::desc_add(kq0, off), tc::desc_add(kq0, off), id_kq, kk > 0);
        }
        tc::mma_commit(&bars[B_KQF + j]);
        return true;
      };
      auto issue_uw = [&](int i) -> bool {
        const int j = i & 1, k = i >> 1;
        if (!tc::mbar_wait(&bars[B_ELF + j], k & 1, err)) return false;
        if (!tc::mbar_wait(&bars[B_TBF + j], k & 1, err)) return false;
        if (i >= 2 && !tc::mbar_wait(&bars[B_UWE + j], (k - 1) & 1, err)) return false;
        tc::fence_after();
        const uint32_t sb = j * S::kStage;
        const uint32_t tu = tmem + kColUW + j * 128;
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          tc::mma_bf16(tu, tc::desc_add(va0, sb + kk * 2048), tc::desc_add(tb0, j * 8192 + kk * 32), id_uw, kk > 0);
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          tc::mma_bf16(tu + 64, tc::desc_add(ka0, sb + kk * 2048), tc::desc_add(tb0, j * 8192 + kk * 32), id_uw,
                       kk > 0);
        tc::mma_commit(&bars[B_UWF + j]);
        tc::mma_commit(&bars[B_EMPTY + j]);
        return true;
      };
      if (nmine > 0) ok = issue_kq(0);
      for (int i = 0; i < nmine && ok; ++i) {
        if (i + 1 < nmine && !(ok = issue_kq(i + 1))) break;
        ok = issue_uw(i);
      }
      // every product has completed before TMEM is released
      tc::mma_commit(&bars[B_DONE]);
      tc::mbar_wait(&bars[B_DONE], 0, err);
    }
  } else if (warp >= kWarpEl && warp < kWarpInv) {
    // ----------------- gate, the score's column sums, beta e^G K in place
    const int el = threadIdx.x - 32 * kWarpEl, ew = warp - kWarpEl;
    const int x = el & 15, hx = x >> 3, gg = x & 7, t0 = el >> 4;  // granule column, rows t0 + 8m
    float* red = (float*)(smem + S::offRed);
    // per-head weights are read ahead of their use (global latency): W_g[h]
    // (this thread's 8 features) and b_g[h] one chunk ahead, the score
    // weights at the top of the chunk that uses them at its end
    float wg[8], bg = 0.f;
    auto load_gate_w = [&](int h) {
      const float4* pg = (const float4*)(w_g + (size_t)h * D + 8 * x);
      const float4 a = pg[0], b = pg[1];
      wg[0] = a.x, wg[1] = a.y, wg[2] = a.z, wg[3] = a.w;
      wg[4] = b.x, wg[5] = b.y, wg[6] = b.z, wg[7] = b.w;
      bg = b_g ? b_g[h] : 0.f;
    };
    Pos pos = first_pos();
    if (nmine > 0) load_gate_w(pos.h);
    bool ok = true;
    for (int i = 0; i < nmine; ++i) {
      const int j = i & 1, k = i >> 1;
      const int blk = pos.blk, h = pos.h;
      const long long tok0 = (long long)pos.bh * L + (long long)pos.c * C;
      next_pos(pos);  // pos: the next chunk
      float sq0[8], sq1[8], bs0 = 0.f, bs1 = 0.f;  // score rows, Q parts, of this head
      if (sel_out) {
        const float4* W = (const float4*)(w_s + (size_t)h * 4 * D + 8 * x);
        const float4 a0 = W[0], a1 = W[1], c0 = W[D / 2], c1 = W[D / 2 + 1];  // rows 0 and 1
        sq0[0] = a0.x, sq0[1] = a0.y, sq0[2] = a0.z, sq0[3] = a0.w, sq0[4] = a1.x, sq0[5] = a1.y, sq0[6] = a1.z, sq0[7] = a1.w;
        sq1[0] = c0.x, sq1[1] = c0.y, sq1[2] = c0.z, sq1[3] = c0.w, sq1[4] = c1.x, sq1[5] = c1.y, sq1[6] = c1.z, sq1[7] = c1.w;
        if (b_s) bs0 = b_s[2 * h], bs1 = b_s[2 * h + 1];
      }
      ok = tc::mbar_wait(&bars[B_FULL + j], k & 1, err);
      uint8_t* st = stage(j);
      const float* sc = scal(j);
      float csq[8], csk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) csq[u] = csk[u] = 0.f;
      // Q: the merge gate's partial dot products (this thread's 8 features of
      // its 8 tokens, then summed over the 16 lanes of a token) and the
      // column sums of Q
      {
        const uint8_t* qb = st + hx * 16384 + 8192;
        const uint64_t w2[4] = {tc::f2_pack(wg[0], wg[1]), tc::f2_pack(wg[2], wg[3]), tc::f2_pack(wg[4], wg[5]),
                                tc::f2_pack(wg[6], wg[7])};
        uint64_t cs2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) cs2[u] = tc::f2_pack(0.f, 0.f);
        float z[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 in = *(const uint4*)(qb + sw_gran(t0 + 8 * m, gg));
          const uint32_t* h2 = (const uint32_t*)&in;
          uint64_t acc = tc::f2_pack(0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint64_t f2 = bf16x2_to_f2(h2[u]);
            acc = tc::f2_fma(f2, w2[u], acc);
            cs2[u] = tc::f2_add(cs2[u], f2);
          }
          float a0, a1;
          tc::f2_unpack(acc, a0, a1);
          z[m] = a0 + a1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) tc::f2_unpack(cs2[u], csq[2 * u], csq[2 * u + 1]);
        // sum over the 16 lanes of a token group, halving the rows kept per
        // lane at each step (8 shuffles): lane x ends with row
        // m = 4 x3 + 2 x2 + x1 (x = 8 x3 + 4 x2 + 2 x1 + x0), twice
        float z4[4], z2[2];
        const bool b3 = x & 8, b2 = x & 4, b1 = x & 2;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          z4[u] = (b3 ? z[4 + u] : z[u]) + __shfl_xor_sync(0xffffffffu, b3 ? z[u] : z[4 + u], 8);
#pragma unroll
        for (int u = 0; u < 2; ++u)
          z2[u] = (b2 ? z4[2 + u] : z4[u]) + __shfl_xor_sync(0xffffffffu, b2 ? z4[u] : z4[2 + u], 4);
        float z1 = (b1 ? z2[1] : z2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? z2[0] : z2[1], 2);
        z1 += __shfl_xor_sync(0xffffffffu, z1, 1);
        if ((x & 1) == 0) {
          const int m = 4 * (x >> 3) + 2 * ((x >> 2) & 1) + ((x >> 1) & 1);
          gate_out[tok0 + t0 + 8 * m] = 1.f / (1.f + __expf(-(z1 + bg)));
        }
      }
      if (i + 1 < nmine) load_gate_w(pos.h);
      // score rows' K parts of this head (used after the K pass)
      float sk0[8], sk1[8];
      if (sel_out) {
        const float4* W = (const float4*)(w_s + (size_t)h * 4 * D + D + 8 * x);
        const float4 a0 = W[0], a1 = W[1], c0 = W[D / 2], c1 = W[D / 2 + 1];
        sk0[0] = a0.x, sk0[1] = a0.y, sk0[2] = a0.z, sk0[3] = a0.w, sk0[4] = a1.x, sk0[5] = a1.y, sk0[6] = a1.z, sk0[7] = a1.w;
        sk1[0] = c0.x, sk1[1] = c0.y, sk1[2] = c0.z, sk1[3] = c0.w, sk1[4] = c1.x, sk1[5] = c1.y, sk1[6] = c1.z, sk1[7] = c1.w;
      }
      // the first product has read K: beta e^G K in place and the column sums of K
      ok = tc::mbar_wait(&bars[B_KQF + j], k & 1, err) && ok;
      {
        uint8_t* kb = st + hx * 16384;
        uint64_t cs2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) cs2[u] = tc::f2_pack(0.f, 0.f);
#pragma unroll 2
        for (int m = 0; m < 8; ++m) {
          const int t = t0 + 8 * m;
          uint4* p = (uint4*)(kb + sw_gran(t, gg));
          const uint4 in = *p;
          const uint32_t* h2 = (const uint32_t*)&in;
          const float fb = sc[2 * C + t];
          const uint64_t fb2 = tc::f2_pack(fb, fb);
          uint4 w;
          uint32_t* w32 = (uint32_t*)&w;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint64_t f2 = bf16x2_to_f2(h2[u]);
            float a0, a1;
            tc::f2_unpack(tc::f2_mul(f2, fb2), a0, a1);
            w32[u] = tc::pack_bf16x2(a0, a1);
            cs2[u] = tc::f2_add(cs2[u], f2);
          }
          *p = w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) tc::f2_unpack(cs2[u], csk[2 * u], csk[2 * u + 1]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_ELF + j]);
      // chunk score, linear in the column sums: per-thread partial dot
      // products, reduced over the warp, then over the four warps
      if (sel_out) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          s0 = fmaf(sq0[u], csq[u], fmaf(sk0[u], csk[u], s0));
          s1 = fmaf(sq1[u], csq[u], fmaf(sk1[u], csk[u], s1));
        }
        s0 = warp_sum(s0);
        s1 = warp_sum(s1);
        if (lane == 0) {
          red[8 * j + ew] = s0;
          red[8 * j + 4 + ew] = s1;
        }
      }
      if (!(ok = group_all(kBarEl, 128, ok))) break;
      if (sel_out && el == 0) {
        const float a = ((red[8 * j] + red[8 * j + 1]) + (red[8 * j + 2] + red[8 * j + 3])) * (1.0f / C) + bs0;
        const float bb = ((red[8 * j + 4] + red[8 * j + 5]) + (red[8 * j + 6] + red[8 * j + 7])) * (1.0f / C) + bs1;
        sel_out[blk] = (a >= bb) ? 0 : 1;
      }
    }
  } else if (warp >= kWarpInv && warp < kWarpUw) {
    // --------------------------------------------- T = (I + A)^{-1} as bf16
    const int gi = threadIdx.x - 32 * kWarpInv, gw = warp - kWarpInv;
    const int gq = lane >> 2, cq = lane & 3;  // mma fragment row / column pair
    float* Ts = (float*)(smem + S::offT);
    float* Xs = (float*)(smem + S::offX);
    auto tile_mma = [&](float (&acc)[2][4], const float* M1, int r0, int c0, const float* M2, int k0, int n0,
                        int klen) {
      for (int kq = 0; kq < klen; kq += 8) {
        const float* ar = M1 + (r0 + gq) * FS + c0 + kq + cq;
        const uint32_t a0 = tf32(ar[0]), a1 = tf32(ar[8 * FS]), a2 = tf32(ar[4]), a3 = tf32(ar[8 * FS + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float* br = M2 + (k0 + kq + cq) * FS + n0 + 8 * nt + gq;
          mma1688_tf32(acc[nt], a0, a1, a2, a3, tf32(br[0]), tf32(br[4 * FS]));
        }
      }
    };
    // fp32 tile to M; a final tile of T also goes to the bf16 operand tile tb
    auto tile_store = [&](float* M, int r0, int n0, const float (&acc)[2][4], float sgn, uint8_t* tb) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int r = r0 + gq, cc = n0 + 8 * nt + 2 * cq;
        const float v0 = sgn * acc[nt][0], v1 = sgn * acc[nt][1], v2 = sgn * acc[nt][2], v3 = sgn * acc[nt][3];
        float* dr = M + r * FS + cc;
        dr[0] = v0;
        dr[1] = v1;
        dr[8 * FS] = v2;
        dr[8 * FS + 1] = v3;
        if (tb) {
          *(uint32_t*)(tb + sw_gran(r, cc >> 3) + (cc & 7) * 2) = tc::pack_bf16x2(v0, v1);
          *(uint32_t*)(tb + sw_gran(r + 8, cc >> 3) + (cc & 7) * 2) = tc::pack_bf16x2(v2, v3);
        }
      }
    };
    // the blocks above the diagonal of both T tiles stay zero
    for (int e = gi; e < 2 * 8192 / 16; e += 128) ((uint4*)(smem + S::offTb))[e] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    bool ok = true;
    for (int i = 0; i < nmine; ++i) {
      const int j = i & 1, k = i >> 1;
      ok = tc::mbar_wait(&bars[B_AF + j], k & 1, err);
      // T tile j is free once chunk i - 2's U / W products are done
      if (i >= 2) ok = tc::mbar_wait(&bars[B_UWF + j], (k - 1) & 1, err) && ok;
      // also: every thread has finished the previous chunk's T
      if (!(ok = group_all(kBarInv, 128, ok))) break;
      float* As = (float*)(smem + S::offA) + j * C * FS;
      uint8_t* Tb = smem + S::offTb + j * 8192;  // T as bf16, swizzled lines t of 64 columns
      // T = (I + A)^{-1}, unit lower triangular, blocked in 16 x 16 tiles.
      // Diagonal tiles by forward substitution (fp32), one column per thread:
      if (gi < C) {
        const int b = gi >> 4, jj = gi & 15, jc = 16 * b + jj;
        float xv[16];
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          const int t = 16 * b + tt;
          float acc = (tt == jj) ? 1.f : 0.f;
#pragma unroll
          for (int ii = 0; ii < tt; ++ii)  // xv[ii] = 0 for ii < jj: no branch needed
            acc = fmaf(-As[t * FS + 16 * b + ii], xv[ii], acc);
          xv[tt] = (tt >= jj) ? acc : 0.f;
        }
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          const int t = 16 * b + tt;
          Ts[t * FS + jc] = xv[tt];
          *(__nv_bfloat16*)(Tb + sw_gran(t, jc >> 3) + (jc & 7) * 2) = __float2bfloat16_rn(xv[tt]);
        }
      }
      if (!(ok = group_all(kBarInv, 128, ok))) break;
      // off-diagonal tiles on tf32 MMAs (fp32 accumulate; T is rounded to
      // bf16 right after, far coarser than the tf32 operands), two levels:
      //   halves a = rows 0-31, b = rows 32-63:  T = [[T_a, 0], [T_ba, T_b]]
      //   level 1: T_10 = -T_11 (A_10 T_00), T_32 = -T_33 (A_32 T_22)
      //   level 2: Y = A_ba T_a, then T_ba = -T_b Y (four 16 x 16 tiles each)
      if (gw < 2) {
        const int ti = 2 * gw + 1, tj = 2 * gw;
        float xa[2][4] = {};
        tile_mma(xa, As, 16 * ti, 16 * tj, Ts, 16 * tj, 16 * tj, 16);  // A_ij T_jj
        tile_store(Xs, 16 * ti, 16 * tj, xa, 1.f, nullptr);
        __syncwarp();
        float ya[2][4] = {};
        tile_mma(ya, Ts, 16 * ti, 16 * ti, Xs, 16 * ti, 16 * tj, 16);  // T_ii X_ij
        tile_store(Ts, 16 * ti, 16 * tj, ya, -1.f, Tb);
      }
      named_barrier(kBarInv, 128);
      const int li = 2 + (gw >> 1), lj = gw & 1;
      {
        float yv[2][4] = {};
        tile_mma(yv, As, 16 * li, 16 * lj, Ts, 16 * lj, 16 * lj, 16 * (2 - lj));  // Y_ij = sum_k A_ik T_kj
        tile_store(Xs, 16 * li, 16 * lj, yv, 1.f, nullptr);
      }
      named_barrier(kBarInv, 128);
      if (lane == 0) tc::mbar_arrive(&bars[B_AE + j]);  // A of this chunk is no longer read
      {
        float tv[2][4] = {};
        tile_mma(tv, Ts, 16 * li, 32, Xs, 32, 16 * lj, 16 * (li - 1));  // T_ij = -sum_k T_ik Y_kj
        tile_store(Ts, 16 * li, 16 * lj, tv, -1.f, Tb);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_TBF + j]);
      if (T_out) {  // T in fp32 for the backward pass (zero above the diagonal blocks)
        named_barrier(kBarInv, 128);
        float* dst = T_out + (size_t)(blockIdx.x + i * stride) * C * C;
        for (int e4 = gi; e4 < C * C / 4; e4 += 128) {
          const int t = e4 / (C / 4), c4 = 4 * (e4 % (C / 4));
          const float4 x = c4 < 16 * (t / 16 + 1) ? *(const float4*)(Ts + t * FS + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
          *(float4*)(dst + t * C + c4) = x;
        }
      }
    }
  } else if (warp >= kWarpEpi) {
    // ----------------------------- A (fp32, shared) and P (bf16) from TMEM
    const int r = 32 * (warp & 3) + lane;  // TMEM lane: KK^T row r (< 64) or QK^T row r - 64
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    uint8_t* Pst = smem + S::offP;
    const bool p_issuer = (warp == kWarpEpi) && lane == 0;  // TMEM lane 64: a P row writer
    bool ok = true;
    for (int i = 0; i < nmine; ++i) {
      const int j = i & 1, k = i >> 1;
      const long long blk = blockIdx.x + i * stride;
      float* As = (float*)(smem + S::offA) + j * C * FS;
      ok = tc::mbar_wait(&bars[B_FULL + j], k & 1, err);
      ok = tc::mbar_wait(&bars[B_KQF + j], k & 1, err) && ok;
      // A buffer j: chunk i - 2's inverse has read it; P tile: the previous store has read it
      if (i >= 2) ok = tc::mbar_wait(&bars[B_AE + j], (k - 1) & 1, err) && ok;
      if (p_issuer) tc::bulk_wait_read_all();
      if (!(ok = group_all(kBarEpi, 128, ok))) break;
      tc::fence_after();
      // A row t (lanes < 64): beta_t e^{G_t - G_i} k_t . k_i for i < t, fp32;
      // P row t (lanes >= 64): scale e^{G_t - G_i} q_t . k_i for i <= t, bf16.
      // One 8-column block per step (a compact loop: the roles of this kernel
      // run different code side by side), the next block's TMEM load in flight.
      {
        const float* sc = scal(j);
        const bool arow = r < C;  // warp-uniform
        const int t = arow ? r : r - C;
        const int lim = arow ? t : t + 1;  // columns i < lim are kept
        const float mult = arow ? sc[C + t] : scale;
        const uint64_t gt2 = tc::f2_pack(sc[3 * C + t], sc[3 * C + t]), m2 = tc::f2_pack(mult, mult);
        const uint32_t ta = tmem + kColKQ + j * 64 + lane_off;
        uint32_t cur[8], nxt[8];
        tc::tmem_ld8u(ta, cur);
        tc::tmem_ld_wait();
#pragma unroll 1
        for (int q8 = 0; q8 < 8; ++q8) {
          if (q8 < 7) tc::tmem_ld8u(ta + 8 * q8 + 8, nxt);
          const float4 g0 = *(const float4*)(sc + 3 * C + 8 * q8), g1 = *(const float4*)(sc + 3 * C + 8 * q8 + 4);
          const uint64_t gi[4] = {tc::f2_pack(g0.x, g0.y), tc::f2_pack(g0.z, g0.w), tc::f2_pack(g1.x, g1.y),
                                  tc::f2_pack(g1.z, g1.w)};
          float o[8];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float d0, d1;
            tc::f2_unpack(tc::f2_sub(gt2, gi[u]), d0, d1);  // (G_t - G_i) log2 e
            const uint64_t e2 = tc::f2_mul(m2, tc::f2_pack(tc::fast_exp2(d0), tc::fast_exp2(d1)));
            tc::f2_unpack(tc::f2_mul(e2, tc::f2_pack(__uint_as_float(cur[2 * u]), __uint_as_float(cur[2 * u + 1]))),
                          o[2 * u], o[2 * u + 1]);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) o[u] = (8 * q8 + u < lim) ? o[u] : 0.f;
          if (arow) {
            *(float4*)(As + t * FS + 8 * q8) = make_float4(o[0], o[1], o[2], o[3]);
            *(float4*)(As + t * FS + 8 * q8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
          } else {
            *(uint4*)(Pst + sw_gran(t, q8)) = make_uint4(tc::pack_bf16x2(o[0], o[1]), tc::pack_bf16x2(o[2], o[3]),
                                                         tc::pack_bf16x2(o[4], o[5]), tc::pack_bf16x2(o[6], o[7]));
          }
          tc::tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u) cur[u] = nxt[u];
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars[B_KQE + j]);
        if (!arow) tc::fence_proxy_async_smem();
      }
      if (!(ok = group_all(kBarEpi, 128, ok))) break;
      if (lane == 0) tc::mbar_arrive(&bars[B_AF + j]);
      if (p_issuer) {
        tc::tma_store_2d(&tm_p, Pst, 0, (int)(blk * C));
        tc::bulk_commit();
      }
    }
    if (p_issuer) tc::bulk_wait_all();
  } else {
    // ------------------------------------------- U^T and W^T to global memory
    const int gu = threadIdx.x - 32 * kWarpUw;
    const int e = 32 * (warp & 3) + lane;  // TMEM lane = feature
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    uint8_t* Wst = smem + S::offW;
    const bool issuer = gu == 0;
    // beta V in place for chunk i (the second product's A operand); these
    // warps run it one chunk ahead of their own U / W work
    const int x = gu & 15, hx = x >> 3, gg = x & 7, t0 = gu >> 4;
    auto scale_v = [&](int i) -> bool {
      const int j = i & 1, k = i >> 1;
      const bool w_ok = tc::mbar_wait(&bars[B_FULL + j], k & 1, err);
      uint8_t* vb = stage(j) + S::kKQ + hx * 8192;
      const float* sc = scal(j);
#pragma unroll 2
      for (int m = 0; m < 8; ++m) {
        const int t = t0 + 8 * m;
        uint4* p = (uint4*)(vb + sw_gran(t, gg));
        const uint4 in = *p;
        const uint32_t* h2 = (const uint32_t*)&in;
        const float fb = sc[C + t];
        const uint64_t fb2 = tc::f2_pack(fb, fb);
        uint4 w;
        uint32_t* w32 = (uint32_t*)&w;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float a0, a1;
          tc::f2_unpack(tc::f2_mul(bf16x2_to_f2(h2[u]), fb2), a0, a1);
          w32[u] = tc::pack_bf16x2(a0, a1);
        }
        *p = w;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_ELF + j]);
      return w_ok;
    };
    bool ok = nmine > 0 ? group_all(kBarUw, 128, scale_v(0)) : true;
    for (int i = 0; i < nmine && ok; ++i) {
      const int j = i & 1, k = i >> 1;
      const long long blk = blockIdx.x + i * stride;
      ok = tc::mbar_wait(&bars[B_UWF + j], k & 1, err);
      // the previous chunk's W store has read the staging tile
      if (issuer) tc::bulk_wait_read_all();
      if (!(ok = group_all(kBarUw, 128, ok))) break;
      tc::fence_after();
      // U^T through the staging tile (line e of [D][64], 8 tokens per step),
      // then W (column e: elements (t, e) of box e / 64) through the same tile
      const uint32_t ta = tmem + kColUW + j * 128 + lane_off;
#pragma unroll 1
      for (int q8 = 0; q8 < 8; ++q8) {
        uint32_t ur[8];
        tc::tmem_ld8u(ta + 8 * q8, ur);
        tc::tmem_ld_wait();
        *(uint4*)(Wst + sw_gran(e, q8)) =
            make_uint4(tc::pack_bf16x2(__uint_as_float(ur[0]), __uint_as_float(ur[1])),
                       tc::pack_bf16x2(__uint_as_float(ur[2]), __uint_as_float(ur[3])),
                       tc::pack_bf16x2(__uint_as_float(ur[4]), __uint_as_float(ur[5])),
                       tc::pack_bf16x2(__uint_as_float(ur[6]), __uint_as_float(ur[7])));
      }
      tc::fence_proxy_async_smem();
      named_barrier(kBarUw, 128);
      if (issuer) {
        tc::tma_store_2d(&tm_u, Wst, 0, (int)(blk * D));
        tc::tma_store_2d(&tm_u, Wst + 8192, 0, (int)(blk * D + 64));
        tc::bulk_commit();
        tc::bulk_wait_read_all();
      }
      named_barrier(kBarUw, 128);
      {
        uint8_t* wb = Wst + (e >> 6) * 8192 + (e & 7) * 2;
        const int ge = (e & 63) >> 3;
#pragma unroll 1
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t wr[8];
          tc::tmem_ld8u(ta + 64 + 8 * q8, wr);
          tc::tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *(__nv_bfloat16*)(wb + sw_gran(8 * q8 + u, ge)) = __float2bfloat16_rn(__uint_as_float(wr[u]));
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_UWE + j]);
      tc::fence_proxy_async_smem();
      named_barrier(kBarUw, 128);
      if (issuer) {
        tc::tma_store_2d(&tm_w, Wst, 0, (int)(blk * C));
        tc::tma_store_2d(&tm_w, Wst + 8192, 64, (int)(blk * C));
        tc::bulk_commit();
      }
      if (i + 1 < nmine && !(ok = group_all(kBarUw, 128, scale_v(i + 1)))) break;
    }
    if (issuer) tc::bulk_wait_all();
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_gdn_prep_tc(const Problem& p, const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* w_g, const float* b_g, float* G, void* W16,
                               void* U16, void* P16, float* gate, const float* w_s, const float* b_s,
                               uint8_t* sel_out, int* err, float* T_out, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  if (p.d != D) return cudaErrorInvalidValue;
  CUtensorMap mk, mq, mv, mw, mu, mp;
  const long long rows = p.BH * p.L;  // = BH * N * 64
  if (!make_tile_map(&mk, k, rows, D) || !make_tile_map(&mq, q, rows, D) || !make_tile_map(&mv, v, rows, D) ||
      !make_tile_map(&mw, W16, rows, D) || !make_tile_map(&mu, U16, p.BH * (long long)p.N * D, 64) ||
      !make_tile_map(&mp, P16, rows, 64))
    return cudaErrorInvalidValue;
  const int smem = PrepTcSmem::kBytes;
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long nchunks = p.BH * p.N;
  const unsigned grid = (unsigned)(nchunks < sms ? nchunks : sms);
  gdn_prep_tc_kernel<<<grid, kThreads, smem, st>>>(mk, mq, mv, mw, mu, mp, g, beta, p.L, p.N, p.H, nchunks,
                                                   p.scale, G, w_g, b_g, gate, w_s, b_s, sel_out, err, T_out);
  return cudaGetLastError();
}

}  // namespace nats
