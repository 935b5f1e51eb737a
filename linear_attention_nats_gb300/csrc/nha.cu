// nha.cu - the Native Hybrid Attention (NHA) layer forward on the
// 5th-generation tensor cores: a slot memory updated by a gated linear RNN
// and a sliding window of recent tokens, joined into one key / value set
// under one softmax.
//
// "Native Hybrid Attention for Efficient Sequence Modeling", section
// "2. Methodologie", "Kernprincipes".  The slot update is the reading taken
// for "inspired by Gated Slot Attention": m slots K~, V~ (m x d); a token j
// writes K~ <- diag(alpha_j) K~ + (1 - alpha_j) k_j^T (V~ likewise with v_j)
// when it leaves the window; the query at t attends with one softmax over
// [the slots after the writes of j <= t - w ; the window keys t - w < j <= t].
//
// Chunkwise form (C = 64 tokens, d = 128, m = 64).  Within the chunk c' of
// the write stream, with lambda = log alpha and A_tau = sum_{i <= tau}
// lambda_i (per slot), a reference A_r = A_31, and the chunk-start slots
// S0, V0:
//   K~ after write tau = e^{A_tau} S0 + sum_{i <= tau} (1 - alpha_i) e^{A_tau - A_i} k_i
// so for a query row tau of the chunk that reads it (scale s):
//   z_slot = s E' (.) (Q S0''^T + lower(Q K^T) G')            (64 x m)
//   o_slot = (p (.) E') V0'' + lower((p (.) E') G'^T) V       (64 x d)
// with E'[tau, s] = e^{A_tau - A_r}, G'[i, s] = (1 - alpha_i) e^{A_r - A_i},
// S0'' = diag(e^{A_r}) S0 and V0'' likewise; every product is a dense
// matrix product on the tensor cores, and the factors stay within
// e^{|A_63 - A_0| / 2} of one (the reference sits mid-chunk).  Between
// chunks S0 <- e^{A_63} (.) S0 + Gamma^T K, Gamma[i, s] = (1 - alpha_i)
// e^{A_63 - A_i} <= 1.
//
// Three kernels.
//   nha_gate_kernel: chunk-parallel; from the log-gates of each chunk it
//     writes G' (bf16 [C][m]), E' (fp32 [C][m]), Gamma (bf16 [C][m]) and the
//     per-slot e^{A_r}, e^{A_63}.
//   nha_state_kernel: two CTAs per (b, h), one per memory (K~, V~), walk the
//     chunks in order with the slot memory in registers (thread = feature);
//     the tensor cores form each chunk's write X^T Gamma ahead of them; per
//     chunk they store S0''^T, V0''^T (bf16 [d][m]).
//   nha_attn_kernel: persistent CTAs over tiles of 128 query rows (two
//     chunks of one head).  The first key block (the two write chunks) runs
//     the slot terms and that block's window keys in one online softmax;
//     the remaining window blocks are plain flash-attention blocks.
// Supported: bf16, d = 128, m = 64, w = 0, a multiple of 128, or >= L.
// Every wait is bounded (tc::kWaitLimitNs); on expiry a kernel records an
// error, drains what it issued and exits.
#include <cmath>

#include "../../include/nats.h"
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {

bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D);

namespace {

constexpr int C = kChunk;  // 64
constexpr int D = 128;     // head size
constexpr int MS = 64;     // slots
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ uint32_t sw128(int line, int col_bf16) {
  // byte offset of bf16 element (line, col) in a [lines x 64] 128-byte-swizzled tile
  return (uint32_t)(line * 128 + ((((col_bf16 >> 3) ^ (line & 7))) << 4) + (col_bf16 & 7) * 2);
}

// ============================================================ gate factors
// Chunk-parallel: one CTA per chunk of the write stream turns its log-gates
// into the factors the scan and the attention read.  Thread (part, s) forms
// the running sum of slot s over tokens 16 part .. 16 part + 15, the four
// parts' totals give each its offset, and every thread then writes four
// (token, slot-quad) groups of E', G' and Gamma.
__global__ void __launch_bounds__(256) nha_gate_kernel(const float* __restrict__ log_alpha,
                                                       __nv_bfloat16* __restrict__ gh_out,
                                                       float* __restrict__ ep_out,
                                                       __nv_bfloat16* __restrict__ gam_out,
                                                       float* __restrict__ er_out) {
  __shared__ __align__(16) float lam[C * MS];
  __shared__ __align__(16) float A[C * MS];
  __shared__ float tot[4][MS];
  const size_t chunk = blockIdx.x;
  const int tid = threadIdx.x;
  const size_t base = chunk * C * MS;
  {
    const float4* src = (const float4*)(log_alpha + base);
#pragma unroll
    for (int j = 0; j < 4; ++j) ((float4*)lam)[tid + 256 * j] = src[tid + 256 * j];
  }
  __syncthreads();
  const int sl = tid & 63, part = tid >> 6;
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int i = 16 * part + j;
    acc += lam[i * MS + sl];
    A[i * MS + sl] = acc;
  }
  tot[part][sl] = acc;
  __syncthreads();
  float off = 0.f;
  for (int p2 = 0; p2 < part; ++p2) off += tot[p2][sl];
#pragma unroll
  for (int j = 0; j < 16; ++j) A[(16 * part + j) * MS + sl] += off;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e4 = tid + 256 * j;  // group of four slots
    const int i = e4 >> 4, s0 = (e4 & 15) * 4;
    float ep[4], gh[4], gm[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int sx = s0 + x;
      const float Ai = A[i * MS + sx], Ar = A[31 * MS + sx], A63 = A[63 * MS + sx];
      const float om = -expm1f(lam[i * MS + sx]);  // 1 - alpha_i, without cancellation
      ep[x] = __expf(Ai - Ar);
      gh[x] = om * __expf(Ar - Ai);
      gm[x] = om * __expf(A63 - Ai);
      if (i == 0) {
        er_out[chunk * 2 * MS + sx] = __expf(Ar);
        er_out[chunk * 2 * MS + MS + sx] = __expf(A63);
      }
    }
    *(float4*)(ep_out + base + 4 * e4) = make_float4(ep[0], ep[1], ep[2], ep[3]);
    *(uint2*)(gh_out + base + 4 * e4) = make_uint2(tc::pack_bf16x2(gh[0], gh[1]), tc::pack_bf16x2(gh[2], gh[3]));
    *(uint2*)(gam_out + base + 4 * e4) = make_uint2(tc::pack_bf16x2(gm[0], gm[1]), tc::pack_bf16x2(gm[2], gm[3]));
  }
}

// ============================================================ state scan
// One CTA per (b, h, memory): memory 0 is the key slots K~, 1 the value
// slots V~ (independent recurrences of the same gates).  The slot memory of
// the CTA, transposed (feature r x 64 slots), lives in the registers of
// state thread r.  Per chunk the tensor cores form the chunk's write
// X^T Gamma (M = 128 features, N = 64 slots, K = 64 tokens) into one of two
// TMEM buffers with no dependence on the state, so they run ahead of the
// state threads, whose chain per chunk is: store the chunk-start memory
// scaled by e^{A_r} (bf16), then S <- e^{A_63} S + X^T Gamma.
struct StSmem {
  static constexpr int kX = C * D * 2;                  // 16 KiB token tile (two 8 KiB feature halves)
  static constexpr int kG = C * MS * 2;                 // 8 KiB Gamma (TMA, 128-byte swizzle)
  static constexpr int kE = 2 * MS * 4;                 // e^{A_r}, e^{A_63}
  static constexpr int kStage = kX + kG + 1024;         // 1 KiB aligned
  static constexpr int kStages = 4;
  static constexpr int offBar = kStages * kStage;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
  static_assert(kX + kG + kE <= kStage, "stage");
};
enum { B_FULL = 0, B_EMPTY = StSmem::kStages, B_DFULL = 2 * StSmem::kStages, B_DEMPTY = B_DFULL + 2,
       B_DONE = B_DEMPTY + 2 };

__global__ void __launch_bounds__(192, 1)
    nha_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_gam, const float* __restrict__ er, int L, int N,
                     __nv_bfloat16* __restrict__ st_out, __nv_bfloat16* __restrict__ ut_out, int* __restrict__ err) {
  using S = StSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = blockIdx.x >> 1;
  const int mem = blockIdx.x & 1;  // 0: key slots, 1: value slots
  const CUtensorMap* tm_x = mem ? &tm_v : &tm_k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      tc::mbar_init(&bars[B_FULL + s], 1);
      tc::mbar_init(&bars[B_EMPTY + s], 1 + 4);  // the MMA's commit + the four state warps (they read E)
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars[B_DFULL + b], 1);
      tc::mbar_init(&bars[B_DEMPTY + b], 4);
    }
    tc::mbar_init(&bars[B_DONE], 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;  // columns 64 b .. 64 b + 63: the write of chunks c = b (mod 2)

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tensormap(tm_x);
      tc::prefetch_tensormap(&tm_gam);
      bool ok = true;
      for (int c = 0; c < N && ok; ++c) {
        const int s = c % S::kStages;
        if (!(ok = tc::mbar_wait(&bars[B_EMPTY + s], ((c / S::kStages) & 1) ^ 1, err))) break;
        uint8_t* st = smem + s * S::kStage;
        const int row = (int)(bh * L + (long long)c * C);
        const long long ch = bh * N + c;
        tc::mbar_arrive_expect_tx(&bars[B_FULL + s], S::kX + S::kG + S::kE);
        tc::tma_load_2d(st, tm_x, 0, row, &bars[B_FULL + s]);
        tc::tma_load_2d(st + 8192, tm_x, 64, row, &bars[B_FULL + s]);
        tc::tma_load_2d(st + S::kX, &tm_gam, 0, (int)(ch * C), &bars[B_FULL + s]);
        tc::bulk_load_1d(st + S::kX + S::kG, er + ch * 2 * MS, S::kE, &bars[B_FULL + s]);
      }
      // every copy issued has landed before the CTA may exit
      for (int s = 0; s < S::kStages; ++s) {
        const int uses = N > s ? (N - 1 - s) / S::kStages + 1 : 0;
        if (uses > 0) tc::mbar_wait(&bars[B_FULL + s], (uses - 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // D[feature, slot] = sum_i X[i, feature] Gamma[i, slot]: A = X^T read
      // feature-major from the token tile, B = Gamma slot-major
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, MS, true, true);
      const uint32_t s0 = tc::smem_u32(smem);
      bool ok = true;
      for (int c = 0; c < N && ok; ++c) {
        const int s = c % S::kStages, b = c & 1;
        if (!(ok = tc::mbar_wait(&bars[B_FULL + s], (c / S::kStages) & 1, err))) break;
        if (c >= 2 && !(ok = tc::mbar_wait(&bars[B_DEMPTY + b], ((c - 2) >> 1) & 1, err))) break;
        tc::fence_after();
        const uint32_t xb = s0 + s * S::kStage;
        const uint64_t xd = tc::smem_desc_sw128(xb, 8192, 1024);
        const uint64_t gd = tc::smem_desc_sw128(xb + S::kX, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          tc::mma_bf16(tmem + MS * b, tc::desc_add(xd, kk * 2048), tc::desc_add(gd, kk * 2048), idesc, kk > 0);
        tc::mma_commit(&bars[B_DFULL + b]);
        tc::mma_commit(&bars[B_EMPTY + s]);
      }
      tc::mma_commit(&bars[B_DONE]);
      tc::mbar_wait(&bars[B_DONE], 0, nullptr);
    }
  } else {
    // ---- state warps 2..5: thread r owns feature r (TMEM lane r)
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    __nv_bfloat16* outp = mem ? ut_out : st_out;
    float sm[MS];
#pragma unroll
    for (int x = 0; x < MS; ++x) sm[x] = 0.f;
    bool ok = true;
    for (int c = 0; c < N && ok; ++c) {
      const int s = c % S::kStages, b = c & 1;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_FULL + s], (c / S::kStages) & 1, err)))) break;
      const float* ef = (const float*)(smem + s * S::kStage + S::kX + S::kG);  // e^{A_r} [MS], e^{A_63} [MS]
      // the chunk-start memory, scaled by e^{A_r}: row r of [D][MS]
      {
        uint4* dst = (uint4*)(outp + ((size_t)(bh * N + c) * D + r) * MS);
#pragma unroll
        for (int x8 = 0; x8 < MS / 8; ++x8) {
          uint4 pk;
          pk.x = tc::pack_bf16x2(sm[8 * x8] * ef[8 * x8], sm[8 * x8 + 1] * ef[8 * x8 + 1]);
          pk.y = tc::pack_bf16x2(sm[8 * x8 + 2] * ef[8 * x8 + 2], sm[8 * x8 + 3] * ef[8 * x8 + 3]);
          pk.z = tc::pack_bf16x2(sm[8 * x8 + 4] * ef[8 * x8 + 4], sm[8 * x8 + 5] * ef[8 * x8 + 5]);
          pk.w = tc::pack_bf16x2(sm[8 * x8 + 6] * ef[8 * x8 + 6], sm[8 * x8 + 7] * ef[8 * x8 + 7]);
          dst[x8] = pk;
        }
      }
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_DFULL + b], (c >> 1) & 1, err)))) break;
      tc::fence_after();
      float w[MS];
      tc::tmem_ld32(tmem + lane_off + MS * b, *reinterpret_cast<float(*)[32]>(&w[0]));
      tc::tmem_ld32(tmem + lane_off + MS * b + 32, *reinterpret_cast<float(*)[32]>(&w[32]));
      tc::tmem_ld_wait();
#pragma unroll
      for (int x = 0; x < MS; ++x) sm[x] = fmaf(sm[x], ef[MS + x], w[x]);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&bars[B_DEMPTY + b]);
        tc::mbar_arrive(&bars[B_EMPTY + s]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
}

// ========================================================= attention
struct AtSmem {
  static constexpr int kBlk = 128 * D * 2;  // 32 KiB: 128 lines x 128 features (two 16 KiB halves)
  static constexpr int KS = 2, VS = 2;
  static constexpr int offQ = 0;
  static constexpr int offSU = offQ + kBlk;     // S0''^T then V0''^T of the two write chunks
  static constexpr int offGH = offSU + kBlk;    // G' of the two write chunks: 128 lines x 64 slots
  static constexpr int offK = offGH + 128 * MS * 2;
  static constexpr int offV = offK + KS * kBlk;
  static constexpr int offBar = offV + VS * kBlk;
  static constexpr int kNumBars = 40;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;
};
enum {
  T_QF = 0, T_QE, T_SUF, T_SUE, T_UF, T_UE, T_GF, T_GE, T_KF, T_KE = T_KF + 2, T_VF = T_KE + 2, T_VE = T_VF + 2,
  T_S0 = T_VE + 2,  // slot block: X and the block's scores ready
  T_P1, T_Z, T_A2, T_R, T_A3,
  T_SF, T_PF = T_SF + 2, T_PVB = T_PF + 2,  // regular blocks, per S buffer
  T_PV = T_PVB + 2,  // every P V product (one phase each)
  T_OF,      // the tile's products are complete
  T_OFREE,   // the epilogue has read O
  T_DONE
};
constexpr uint32_t kTZ = 0, kTS = 128, kTR = 256, kTO = 384;
enum { mNone = 0, mFull = 1, mLower = 2, mUpper = 3 };

struct NhaTile {
  long long bh;
  int c0, w0, nb, j0, Wt;
  bool has_c1, slots;
};

__device__ __forceinline__ NhaTile nha_tile(long long i, int T, int N, int Wq, bool full) {
  NhaTile t;
  t.bh = i / T;
  const int p = (int)(i % T);
  t.c0 = 2 * p;
  t.has_c1 = t.c0 + 1 < N;
  t.Wt = full ? t.c0 + 2 : min(Wq, t.c0 + 2);
  t.w0 = t.c0 - t.Wt;                 // first write chunk (>= -2, even)
  t.slots = t.w0 >= 0;                // both halves read slots (not in full mode: w0 = -2 there)
  t.nb = t.Wt / 2 + 1;                // key blocks (pairs of chunks w0 + 2j, w0 + 2j + 1)
  t.j0 = t.w0 < 0 ? 1 : 0;            // block 0 holds no chunk when w0 = -2
  return t;
}

// window mask of key chunk u (chunk w0 + u) for query half h (chunk w0 + Wt + h)
__device__ __forceinline__ int win_mode(const NhaTile& t, int u, int h, int N) {
  const int ca = t.w0 + u;
  if (ca < 0 || ca >= N || u < h || u > t.Wt + h) return mNone;
  const bool lo = u == h, hi = u == t.Wt + h;
  if (lo && hi) return mNone;  // w = 0: the window is empty
  if (lo) return mUpper;       // keys of the first window chunk after the query's position
  if (hi) return mLower;       // the query's own chunk, causally
  return mFull;
}

__device__ __forceinline__ void apply_mode(float (&v)[32], int mode, int key0, int tau) {
  if (mode == mNone) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = -INFINITY;
  } else if (mode == mLower) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = (key0 + x <= tau) ? v[x] : -INFINITY;
  } else if (mode == mUpper) {
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] = (key0 + x > tau) ? v[x] : -INFINITY;
  }
}

// A bounded wait that, when it gives up, also records where: err[1] = the
// first expired wait's code (role * 100 + barrier), err[2] its CTA, err[3]
// the phase parity it waited for.
__device__ __forceinline__ bool wait_at(uint64_t* bars, int bar, int parity, int role, int* err) {
  if (tc::mbar_wait(&bars[bar], (uint32_t)parity, err)) return true;
  if (atomicCAS(err + 1, 0, role * 100 + bar + 1) == 0) {
    err[2] = (int)blockIdx.x;
    err[3] = parity;
  }
  return false;
}

__global__ void __launch_bounds__(256, 1)
    nha_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_st,
                    const __grid_constant__ CUtensorMap tm_ut, const __grid_constant__ CUtensorMap tm_gh,
                    const float* __restrict__ ep, int L, int N, int T, long long BH, int Wq, int full, float sl2,
                    __nv_bfloat16* __restrict__ out, int* __restrict__ err) {
  using S = AtSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n_tiles = BH * T;

  if (threadIdx.x == 0) {
    for (int b = 0; b < T_DONE + 1; ++b) {
      // arrivals of the softmax warps (4 warps, lane 0 each); the rest: one
      // arrival (a TMA transaction count or an MMA commit)
      const bool sm = b == T_P1 || b == T_A2 || b == T_A3 || b == T_PF || b == T_PF + 1 || b == T_OFREE;
      tc::mbar_init(&bars[b], sm ? 4 : 1);
    }
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tensormap(&tm_q);
      tc::prefetch_tensormap(&tm_k);
      tc::prefetch_tensormap(&tm_v);
      tc::prefetch_tensormap(&tm_st);
      tc::prefetch_tensormap(&tm_ut);
      tc::prefetch_tensormap(&tm_gh);
      int tn = 0, sn = 0, gk = 0;
      bool ok = true;
      auto clampc = [&](int c) { return c < 0 ? 0 : (c >= N ? N - 1 : c); };
      for (long long ti = blockIdx.x; ti < n_tiles && ok; ti += gridDim.x, ++tn) {
        const NhaTile t = nha_tile(ti, T, N, Wq, full != 0);
        const long long row0 = t.bh * (long long)L;
        if (!(ok = wait_at(bars, T_QE, (tn & 1) ^ 1, 1, err))) break;
        tc::mbar_arrive_expect_tx(&bars[T_QF], S::kBlk);
        for (int hh = 0; hh < 2; ++hh)
          for (int rc = 0; rc < 2; ++rc)
            tc::tma_load_2d(smem + S::offQ + hh * 16384 + rc * 8192, &tm_q, 64 * hh,
                            (int)(row0 + 64LL * (t.c0 + rc)), &bars[T_QF]);
        auto load_kv = [&](int j) -> bool {
          const int ks = gk % S::KS, par = ((gk / S::KS) & 1) ^ 1;
          if (!wait_at(bars, T_KE + ks, par, 1, err)) return false;
          tc::mbar_arrive_expect_tx(&bars[T_KF + ks], S::kBlk);
          for (int u2 = 0; u2 < 2; ++u2)
            for (int hh = 0; hh < 2; ++hh)
              tc::tma_load_2d(smem + S::offK + ks * S::kBlk + hh * 16384 + u2 * 8192, &tm_k, 64 * hh,
                              (int)(row0 + 64LL * clampc(t.w0 + 2 * j + u2)), &bars[T_KF + ks]);
          if (!wait_at(bars, T_VE + ks, par, 1, err)) return false;
          tc::mbar_arrive_expect_tx(&bars[T_VF + ks], S::kBlk);
          for (int u2 = 0; u2 < 2; ++u2)
            for (int hh = 0; hh < 2; ++hh)
              tc::tma_load_2d(smem + S::offV + ks * S::kBlk + hh * 16384 + u2 * 8192, &tm_v, 64 * hh,
                              (int)(row0 + 64LL * clampc(t.w0 + 2 * j + u2)), &bars[T_VF + ks]);
          ++gk;
          return true;
        };
        if (t.slots) {
          // S0''^T of the two write chunks, then their G'
          if (!(ok = wait_at(bars, T_UE, (sn & 1) ^ 1, 1, err))) break;
          tc::mbar_arrive_expect_tx(&bars[T_SUF], S::kBlk);
          for (int u2 = 0; u2 < 2; ++u2)
            for (int rr = 0; rr < 2; ++rr)
              tc::tma_load_2d(smem + S::offSU + u2 * 16384 + rr * 8192, &tm_st, 0,
                              (int)((t.bh * N + t.w0 + u2) * D + 64 * rr), &bars[T_SUF]);
          if (!(ok = wait_at(bars, T_GE, (sn & 1) ^ 1, 1, err))) break;
          tc::mbar_arrive_expect_tx(&bars[T_GF], 128 * MS * 2);
          for (int u2 = 0; u2 < 2; ++u2)
            tc::tma_load_2d(smem + S::offGH + u2 * 8192, &tm_gh, 0, (int)((t.bh * N + t.w0 + u2) * C), &bars[T_GF]);
          if (!(ok = load_kv(0))) break;
          // V0''^T replaces S0''^T once the first product has read it
          if (!(ok = wait_at(bars, T_SUE, sn & 1, 1, err))) break;
          tc::mbar_arrive_expect_tx(&bars[T_UF], S::kBlk);
          for (int u2 = 0; u2 < 2; ++u2)
            for (int rr = 0; rr < 2; ++rr)
              tc::tma_load_2d(smem + S::offSU + u2 * 16384 + rr * 8192, &tm_ut, 0,
                              (int)((t.bh * N + t.w0 + u2) * D + 64 * rr), &bars[T_UF]);
          ++sn;
        }
        for (int j = t.slots ? 1 : t.j0; j < t.nb && ok; ++j) ok = load_kv(j);
      }
      // drain
      for (int s = 0; s < S::KS; ++s) {
        const int uses = gk > s ? (gk - 1 - s) / S::KS + 1 : 0;
        if (uses > 0) {
          tc::mbar_wait(&bars[T_KF + s], (uses - 1) & 1, nullptr);
          tc::mbar_wait(&bars[T_VF + s], (uses - 1) & 1, nullptr);
          if (ok) {
            tc::mbar_wait(&bars[T_KE + s], (uses - 1) & 1, err);
            tc::mbar_wait(&bars[T_VE + s], (uses - 1) & 1, err);
          }
        }
      }
      if (tn > 0) tc::mbar_wait(&bars[T_QF], (tn - 1) & 1, nullptr);
      if (sn > 0) {
        tc::mbar_wait(&bars[T_UF], (sn - 1) & 1, nullptr);
        tc::mbar_wait(&bars[T_GF], (sn - 1) & 1, nullptr);
        if (ok) tc::mbar_wait(&bars[T_UE], (sn - 1) & 1, err);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_k = tc::idesc_bf16_f32(128, 128, false, false);   // B K-major, N = 128
      constexpr uint32_t id_n = tc::idesc_bf16_f32(128, 128, false, true);    // B N-major, N = 128
      constexpr uint32_t id_n64 = tc::idesc_bf16_f32(128, 64, false, true);   // B N-major, N = 64
      const uint32_t s0 = tc::smem_u32(smem);
      const uint64_t qd = tc::smem_desc_sw128(s0 + S::offQ, 16, 1024);
      const uint64_t sud_n = tc::smem_desc_sw128(s0 + S::offSU, 16384, 1024);  // S0''^T: K = features, N = slots
      const uint64_t sud_k = tc::smem_desc_sw128(s0 + S::offSU, 16, 1024);     // V0''^T: N = features, K = slots
      const uint64_t ghd_n = tc::smem_desc_sw128(s0 + S::offGH, 8192, 1024);   // G': K = keys, N = slots
      const uint64_t ghd_k = tc::smem_desc_sw128(s0 + S::offGH, 16, 1024);     // G'^T: N = keys, K = slots
      const uint64_t kd0 = tc::smem_desc_sw128(s0 + S::offK, 16, 1024);
      const uint64_t vd0 = tc::smem_desc_sw128(s0 + S::offV, 16384, 1024);
      int tn = 0, sn = 0, gk = 0, npv = 0;
      int ub[2] = {0, 0};  // uses of the regular S buffers
      bool ok = true;
      for (long long ti = blockIdx.x; ti < n_tiles && ok; ti += gridDim.x, ++tn) {
        const NhaTile t = nha_tile(ti, T, N, Wq, full != 0);
        if (tn > 0 && !(ok = wait_at(bars, T_OFREE, (tn - 1) & 1, 2, err))) break;
        if (!(ok = wait_at(bars, T_QF, tn & 1, 2, err))) break;
        bool first_pv = true;
        auto pv = [&](uint32_t a_tmem, int vs) {
          const uint64_t vd = tc::desc_add(vd0, vs * S::kBlk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16_ts(tmem + kTO, a_tmem + kk * 8, tc::desc_add(vd, kk * 2048), id_n,
                            (!first_pv) || (kk > 0));
          first_pv = false;
        };
        auto qk = [&](uint32_t d_tmem, int ks) {
          const uint64_t kd = tc::desc_add(kd0, ks * S::kBlk);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            tc::mma_bf16(d_tmem, tc::desc_add(qd, off), tc::desc_add(kd, off), id_k, kk > 0);
          }
        };
        // scores of regular block r (key block j0r + r, global key block g0r + r)
        // into its S buffer, issued one block ahead of that block's P V so
        // that the tensor pipe computes S_{r+1} while the softmax warps turn
        // S_r into P_r
        const int j0r = t.slots ? 1 : t.j0, nreg = t.nb - j0r;
        int g0r = gk + (t.slots ? 1 : 0);
        auto issue_s = [&](int r) -> bool {
          const int g = g0r + r, ks = g % S::KS, b = r & 1;
          // the buffer's previous P has been read by its product
          if (ub[b] > 0 && !wait_at(bars, T_PVB + b, (ub[b] - 1) & 1, 2, err)) return false;
          if (!wait_at(bars, T_KF + ks, (g / S::KS) & 1, 2, err)) return false;
          tc::fence_after();
          qk(tmem + (b ? kTR : kTZ), ks);
          tc::mma_commit(&bars[T_SF + b]);
          tc::mma_commit(&bars[T_KE + ks]);
          return true;
        };
        int next_s = 0;  // regular blocks whose scores are issued
        if (t.slots) {
          const int ks = gk % S::KS;
          if (!(ok = wait_at(bars, T_SUF, sn & 1, 2, err))) break;
          if (!(ok = wait_at(bars, T_KF + ks, (gk / S::KS) & 1, 2, err))) break;
          tc::fence_after();
          // X = Q S0''^T (both write chunks side by side, N = 128)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma_bf16(tmem + kTZ, tc::desc_add(qd, (kk >> 2) * 16384 + (kk & 3) * 32),
                         tc::desc_add(sud_n, kk * 2048), id_n, kk > 0);
          tc::mma_commit(&bars[T_SUE]);
          qk(tmem + kTS, ks);  // the first key block's scores
          tc::mma_commit(&bars[T_S0]);
          // Z += lower(Q K^T) G' into each half's slot columns
          if (!(ok = wait_at(bars, T_P1, sn & 1, 2, err))) break;
          if (!(ok = wait_at(bars, T_GF, sn & 1, 2, err))) break;
          tc::fence_after();
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc::mma_bf16_ts(tmem + kTZ + 64 * half, tmem + kTR + kk * 8, tc::desc_add(ghd_n, kk * 2048), id_n64,
                              1);
          tc::mma_commit(&bars[T_Z]);
          // O = P~ V0'' and R = P~ G'^T (P~ block-diagonal over the two halves' slots)
          if (!(ok = wait_at(bars, T_A2, sn & 1, 2, err))) break;
          if (!(ok = wait_at(bars, T_UF, sn & 1, 2, err))) break;
          tc::fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16_ts(tmem + kTO, tmem + kTZ + kk * 8,
                            tc::desc_add(sud_k, (kk >> 2) * 16384 + (kk & 3) * 32), id_k, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_bf16_ts(tmem + kTR, tmem + kTZ + kk * 8, tc::desc_add(ghd_k, (kk & 3) * 32), id_k, kk > 0);
          first_pv = false;
          tc::mma_commit(&bars[T_R]);
          tc::mma_commit(&bars[T_UE]);
          tc::mma_commit(&bars[T_GE]);
          // Z's columns are free once the two products above have read P~
          // (issue order): the next block's scores go there now
          if (nreg > 0) {
            if (!(ok = issue_s(0))) break;
            next_s = 1;
          }
          // O += (lower(R) + P_window) V of the first key block
          if (!(ok = wait_at(bars, T_A3, sn & 1, 2, err))) break;
          if (!(ok = wait_at(bars, T_VF + ks, (gk / S::KS) & 1, 2, err))) break;
          tc::fence_after();
          pv(tmem + kTS, ks);
          tc::mma_commit(&bars[T_PV]);
          ++npv;
          tc::mma_commit(&bars[T_KE + ks]);
          tc::mma_commit(&bars[T_VE + ks]);
          ++gk;
          ++sn;
        }
        for (int r = 0; r < nreg && ok; ++r, ++gk) {
          const int ks = gk % S::KS, b = r & 1;
          if (next_s == r) {
            if (!(ok = issue_s(r))) break;
            ++next_s;
          }
          if (r + 1 < nreg) {
            if (!(ok = issue_s(r + 1))) break;
            ++next_s;
          }
          if (!(ok = wait_at(bars, T_PF + b, ub[b] & 1, 2, err))) break;
          if (!(ok = wait_at(bars, T_VF + ks, (gk / S::KS) & 1, 2, err))) break;
          tc::fence_after();
          pv(tmem + (b ? kTR : kTZ), ks);
          tc::mma_commit(&bars[T_PVB + b]);
          tc::mma_commit(&bars[T_PV]);
          tc::mma_commit(&bars[T_VE + ks]);
          ++npv;
          ++ub[b];
        }
        if (!ok) break;
        tc::mma_commit(&bars[T_OF]);
        tc::mma_commit(&bars[T_QE]);
      }
      (void)npv;
      tc::mma_commit(&bars[T_DONE]);
      tc::mbar_wait(&bars[T_DONE], 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x - 128;
    const int h = r >> 6, tau = r & 63;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tZ = tmem + kTZ + lane_off, tS = tmem + kTS + lane_off, tR = tmem + kTR + lane_off,
                   tO = tmem + kTO + lane_off;
    int tn = 0, sn = 0, npv = 0;
    int ub[2] = {0, 0};
    bool ok = true;
    auto wait_all = [&](int bar, int par) -> bool {
      return __all_sync(0xffffffffu, wait_at(bars, bar, par, 3, err));
    };
    auto arrive = [&](int bar) {
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[bar]);
    };
    for (long long ti = blockIdx.x; ti < n_tiles && ok; ti += gridDim.x, ++tn) {
      const NhaTile t = nha_tile(ti, T, N, Wq, full != 0);
      float m_used = -INFINITY, l = 0.f;
      bool have_pv = false;
      if (t.slots) {
        // E' of this row's write chunk (w0 + h), read ahead of its use
        float e[MS];
        {
          // (a missing second chunk reads its partner's row; those rows are not stored)
          const int wc = min(t.w0 + h, N - 1);
          const float4* src = (const float4*)(ep + (((size_t)t.bh * N + wc) * C + tau) * MS);
#pragma unroll
          for (int x = 0; x < MS / 4; ++x) {
            const float4 f = src[x];
            e[4 * x] = f.x, e[4 * x + 1] = f.y, e[4 * x + 2] = f.z, e[4 * x + 3] = f.w;
          }
        }
        // ---- P1 = lower(Q K^T) over the row's own write chunk, bf16 into R's columns
        if (!(ok = wait_all(T_S0, sn & 1))) break;
        tc::fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float v[32];
          tc::tmem_ld32(tS + 32 * ch, v);
          tc::tmem_ld_wait();
          const bool own = (ch >> 1) == h;
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int i0 = (ch & 1) * 32 + 2 * x;
            pk[x] = tc::pack_bf16x2(own && i0 <= tau ? v[2 * x] : 0.f, own && i0 + 1 <= tau ? v[2 * x + 1] : 0.f);
          }
          tc::tmem_st16u(tR + 16 * ch, pk);
        }
        tc::tmem_st_wait();
        arrive(T_P1);
        // ---- slot logits, the first block's window logits, one row max
        if (!(ok = wait_all(T_Z, sn & 1))) break;
        tc::fence_after();
        float zs[MS];
        tc::tmem_ld32_at<0>(tZ + 64 * h, zs);
        tc::tmem_ld32_at<32>(tZ + 64 * h + 32, zs);
        tc::tmem_ld_wait();
        float mx = -INFINITY;
#pragma unroll
        for (int x = 0; x < MS; ++x) {
          zs[x] *= sl2 * e[x];
          mx = fmaxf(mx, zs[x]);
        }
        // the window logits of the first block: their max now, their
        // probabilities below (read twice from TMEM, 32 columns at a time)
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float wv[32];
          tc::tmem_ld32(tS + 32 * ch, wv);
          tc::tmem_ld_wait();
          apply_mode(wv, win_mode(t, ch >> 1, h, N), (ch & 1) * 32, tau);
#pragma unroll
          for (int x = 0; x < 32; ++x) mx = fmaxf(mx, wv[x] * sl2);
        }
        m_used = mx;  // finite: every slot logit is
        float sum = 0.f;
        // P~ = p_slot e' (bf16) into Z's columns, the other half's slots zero
        {
          uint32_t pk[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const float p0 = tc::fast_exp2(zs[2 * x] - mx), p1 = tc::fast_exp2(zs[2 * x + 1] - mx);
            sum += p0 + p1;
            pk[x] = tc::pack_bf16x2(p0 * e[2 * x], p1 * e[2 * x + 1]);
          }
          uint32_t zero[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) zero[x] = 0u;
          if (h == 0) {
            tc::tmem_st32u(tZ, pk);
            tc::tmem_st32u(tZ + 32, zero);
          } else {
            tc::tmem_st32u(tZ, zero);
            tc::tmem_st32u(tZ + 32, pk);
          }
        }
        // window probabilities of the first block (fp32) over its scores
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float p[32];
          tc::tmem_ld32(tS + 32 * ch, p);
          tc::tmem_ld_wait();
          apply_mode(p, win_mode(t, ch >> 1, h, N), (ch & 1) * 32, tau);
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            p[x] = tc::fast_exp2(p[x] * sl2 - mx);
            sum += p[x];
          }
          tc::tmem_st32(tS + 32 * ch, p);
        }
        tc::tmem_st_wait();
        l = sum;
        arrive(T_A2);
        // ---- A3 = lower(R) over the own write chunk + the window probabilities
        if (!(ok = wait_all(T_R, sn & 1))) break;
        tc::fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float rv[32], pw[32];
          tc::tmem_ld32(tR + 32 * ch, rv);
          tc::tmem_ld32(tS + 32 * ch, pw);
          tc::tmem_ld_wait();
          const bool own = (ch >> 1) == h;
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int i0 = (ch & 1) * 32 + 2 * x;
            const float a0 = pw[2 * x] + (own && i0 <= tau ? rv[2 * x] : 0.f);
            const float a1 = pw[2 * x + 1] + (own && i0 + 1 <= tau ? rv[2 * x + 1] : 0.f);
            pk[x] = tc::pack_bf16x2(a0, a1);
          }
          tc::tmem_st16u(tS + 16 * ch, pk);  // bf16 columns 16 ch .. : read already
        }
        tc::tmem_st_wait();
        arrive(T_A3);
        ++npv;
        have_pv = true;
        ++sn;
      }
      // ---- plain window blocks
      int rb = 0;
      for (int j = t.slots ? 1 : t.j0; j < t.nb && ok; ++j, ++rb) {
        const int b = rb & 1;
        const uint32_t tb = b ? tR : tZ;
        if (!(ok = wait_all(T_SF + b, ub[b] & 1))) break;
        tc::fence_after();
        float v[128];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(tb + 32 * ch, *reinterpret_cast<float(*)[32]>(&v[32 * ch]));
        tc::tmem_ld_wait();
        float mx = -INFINITY;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          apply_mode(*reinterpret_cast<float(*)[32]>(&v[32 * ch]), win_mode(t, 2 * j + (ch >> 1), h, N),
                     (ch & 1) * 32, tau);
#pragma unroll
          for (int x = 0; x < 32; ++x) mx = fmaxf(mx, v[32 * ch + x]);
        }
        const float m_cand = mx * sl2;
        float alpha = 1.f;
        bool need = false;
        if (!have_pv) {
          if (m_cand > -INFINITY) m_used = m_cand;
        } else if (m_cand > m_used + kRescaleLog2) {
          need = true;
          alpha = tc::fast_exp2(m_used - m_cand);
          m_used = m_cand;
        }
        const float mu = m_used > -INFINITY ? m_used : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float e0 = tc::fast_exp2(v[32 * ch + 2 * x] * sl2 - mu);
            const float e1 = tc::fast_exp2(v[32 * ch + 2 * x + 1] * sl2 - mu);
            sum += e0 + e1;
            pk[x] = tc::pack_bf16x2(e0, e1);
          }
          tc::tmem_st16u(tb + 16 * ch, pk);
        }
        tc::tmem_st_wait();
        if (__any_sync(0xffffffffu, need)) {
          // O holds every product so far before it is rescaled in place
          if (!(ok = wait_all(T_PV, (npv - 1) & 1))) break;
          tc::fence_after();
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float o[32];
            tc::tmem_ld32(tO + 32 * ch, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            tc::tmem_st32(tO + 32 * ch, o);
          }
          tc::tmem_st_wait();
        }
        l = l * alpha + sum;
        arrive(T_PF + b);
        ++ub[b];
        ++npv;
        have_pv = true;
      }
      if (!ok) break;
      // ---- epilogue: out = O / l
      if (!(ok = wait_all(T_OF, tn & 1))) break;
      tc::fence_after();
      {
        const float inv = 1.f / l;
        float o[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tc::tmem_ld32(tO + 32 * ch, *reinterpret_cast<float(*)[32]>(&o[32 * ch]));
        tc::tmem_ld_wait();
        arrive(T_OFREE);
        if (h == 0 || t.has_c1) {
          __nv_bfloat16* dst = out + ((size_t)t.bh * L + (size_t)(t.c0 + h) * C + tau) * D;
#pragma unroll
          for (int c8 = 0; c8 < D / 8; ++c8) {
            uint4 pk;
            pk.x = tc::pack_bf16x2(o[8 * c8] * inv, o[8 * c8 + 1] * inv);
            pk.y = tc::pack_bf16x2(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv);
            pk.z = tc::pack_bf16x2(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv);
            pk.w = tc::pack_bf16x2(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv);
            ((uint4*)dst)[c8] = pk;
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t nha_workspace_bytes(long long BH, int L) {
  const size_t chunks = (size_t)BH * (L / C);
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(chunks * D * MS * 2) * 2 + al(chunks * C * MS * 2) * 2 + al(chunks * C * MS * 4) +
         al(chunks * 2 * MS * 4) + 256;
}

cudaError_t launch_nha_fwd(long long BH, int L, int window, float scale, const void* q, const void* k, const void* v,
                           const float* log_alpha, void* out, void* ws, cudaStream_t st, void* const* ev_start,
                           void* const* ev_stop, int* launches) {
  auto mark = [&](void* const* ev, int i) -> cudaError_t {
    return (ev && ev[i]) ? cudaEventRecord((cudaEvent_t)ev[i], st) : cudaSuccess;
  };
  const int N = L / C;
  if (BH == 0 || N == 0) return cudaSuccess;
  const size_t chunks = (size_t)BH * N;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  char* p = (char*)ws;
  __nv_bfloat16* st_buf = (__nv_bfloat16*)p;
  p += al(chunks * D * MS * 2);
  __nv_bfloat16* ut_buf = (__nv_bfloat16*)p;
  p += al(chunks * D * MS * 2);
  __nv_bfloat16* gh_buf = (__nv_bfloat16*)p;
  p += al(chunks * C * MS * 2);
  __nv_bfloat16* gam_buf = (__nv_bfloat16*)p;
  p += al(chunks * C * MS * 2);
  float* ep_buf = (float*)p;
  p += al(chunks * C * MS * 4);
  float* er_buf = (float*)p;
  p += al(chunks * 2 * MS * 4);
  int* err = (int*)p;
  cudaError_t e = cudaMemsetAsync(err, 0, 16, st);
  if (e != cudaSuccess) return e;
  const long long rows = BH * (long long)L;
  const bool full = window >= L;
  CUtensorMap mk, mv;
  if (!make_tile_map(&mk, k, rows, D) || !make_tile_map(&mv, v, rows, D)) return cudaErrorInvalidValue;
  if (!full) {
    CUtensorMap mgam;
    if (!make_tile_map(&mgam, gam_buf, (long long)chunks * C, MS)) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(nha_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, StSmem::kBytes);
    if (e != cudaSuccess) return e;
    if ((e = mark(ev_start, 0)) != cudaSuccess) return e;
    nha_gate_kernel<<<(unsigned)chunks, 256, 0, st>>>(log_alpha, gh_buf, ep_buf, gam_buf, er_buf);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nha_state_kernel<<<(unsigned)(2 * BH), 192, StSmem::kBytes, st>>>(mk, mv, mgam, er_buf, L, N, st_buf, ut_buf,
                                                                       err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = mark(ev_stop, 0)) != cudaSuccess) return e;
    if (launches) *launches += 2;
  }
  CUtensorMap mq, mst, mut, mgh;
  if (!make_tile_map(&mq, q, rows, D) || !make_tile_map(&mst, st_buf, (long long)chunks * D, MS) ||
      !make_tile_map(&mut, ut_buf, (long long)chunks * D, MS) ||
      !make_tile_map(&mgh, gh_buf, (long long)chunks * C, MS))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(nha_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AtSmem::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int T = (N + 1) / 2;
  const long long tiles = BH * T;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  if ((e = mark(ev_start, 1)) != cudaSuccess) return e;
  nha_attn_kernel<<<grid, 256, AtSmem::kBytes, st>>>(mq, mk, mv, mst, mut, mgh, ep_buf, L, N, T, BH,
                                                     full ? 0 : window / C, full ? 1 : 0, scale * kLog2e,
                                                     (__nv_bfloat16*)out, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = mark(ev_stop, 1)) != cudaSuccess) return e;
  if (launches) ++*launches;
  return cudaSuccess;
}

int* nha_err_flag(void* ws, long long BH, int L) {
  return (int*)((char*)ws + nha_workspace_bytes(BH, L) - 256);
}

// ------------------------------------------------------------------ C ABI
namespace {

nats_status check_nha_dims(const nats_nha_dims* d) {
  if (!d) return NATS_ERR_NULL;
  if (d->dtype != NATS_BF16) return NATS_ERR_DTYPE;
  if (d->B < 0 || d->H < 0 || d->L < 0 || d->window < 0 || d->L % kChunk != 0) return NATS_ERR_SHAPE;
  if (d->d != D || d->slots != MS) return NATS_ERR_UNSUPPORTED;
  if (d->window % 128 != 0 && d->window < d->L) return NATS_ERR_UNSUPPORTED;
  if (!std::isfinite(d->scale) || d->scale < 0.f) return NATS_ERR_VALUE;
  const long long BH = (long long)d->B * d->H;
  if (BH * (long long)d->L > (1LL << 31) - 1 - 128 || BH * (d->L / kChunk) * (long long)D > (1LL << 31) - 1)
    return NATS_ERR_UNSUPPORTED;
  return NATS_OK;
}

}  // namespace
}  // namespace nats

using namespace nats;

extern "C" {

size_t nats_nha_workspace_size(const nats_nha_dims* dims) {
  if (check_nha_dims(dims) != NATS_OK) return 0;
  return nha_workspace_bytes((long long)dims->B * dims->H, dims->L);
}

nats_status nats_nha_fwd_profiled(const nats_nha_dims* dims, const void* q, const void* k, const void* v,
                                  const float* log_alpha, void* out, void* workspace, size_t workspace_bytes,
                                  nats_stream_t stream, nats_profile* prof) {
  const nats_status s = check_nha_dims(dims);
  if (s != NATS_OK) return s;
  const long long BH = (long long)dims->B * dims->H;
  if (BH == 0 || dims->L == 0) return NATS_OK;
  if (!q || !k || !v || !log_alpha || !out || !workspace) return NATS_ERR_NULL;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)log_alpha | (uintptr_t)out | (uintptr_t)workspace) &
      15)
    return NATS_ERR_ALIGN;
  if (workspace_bytes < nha_workspace_bytes(BH, dims->L)) return NATS_ERR_WORKSPACE;
  const float scale = dims->scale > 0.f ? dims->scale : 1.0f / std::sqrt((float)D);
  if (prof) {
    prof->launches = 0;
    for (int i = 0; i < NATS_NUM_STAGES; ++i) prof->stage_launches[i] = 0;
  }
  const cudaError_t e = launch_nha_fwd(BH, dims->L, dims->window, scale, q, k, v, log_alpha, out, workspace,
                                       (cudaStream_t)stream, prof ? prof->start : nullptr,
                                       prof ? prof->stop : nullptr, prof ? &prof->launches : nullptr);
  if (prof) {
    prof->stage_launches[0] = dims->window < dims->L ? 2 : 0;
    prof->stage_launches[1] = 1;
  }
  return e == cudaSuccess ? NATS_OK : NATS_ERR_CUDA;
}

nats_status nats_nha_fwd(const nats_nha_dims* dims, const void* q, const void* k, const void* v,
                         const float* log_alpha, void* out, void* workspace, size_t workspace_bytes,
                         nats_stream_t stream) {
  return nats_nha_fwd_profiled(dims, q, k, v, log_alpha, out, workspace, workspace_bytes, stream, nullptr);
}

nats_status nats_nha_workspace_check(const nats_nha_dims* dims, const void* workspace, nats_stream_t stream) {
  const nats_status s = check_nha_dims(dims);
  if (s != NATS_OK) return s;
  const long long BH = (long long)dims->B * dims->H;
  if (BH == 0 || dims->L == 0) return NATS_OK;
  if (!workspace) return NATS_ERR_NULL;
  int flag = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&flag, nha_err_flag((void*)workspace, BH, dims->L), sizeof(int), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return NATS_ERR_CUDA;
  return flag ? NATS_ERR_INTERNAL : NATS_OK;
}

}  // extern "C"
