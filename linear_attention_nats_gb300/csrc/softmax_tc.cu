// softmax_tc.cu - softmax branch on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA), bf16 inputs.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 3: the softmax state is the set of keys and values
// of the chunks that chose softmax; inside a chunk both correlations are
// computed, so every query of chunk c attends to the retained chunks before
// c plus its own chunk causally (diagonal included).
//
// Tiling.  A CTA owns one 128-row query tile = the two chunks c0 = 2p and
// c1 = 2p + 1 of one (b, h).  Its key/value blocks are 128 keys = two 64-token
// chunk slots: first the softmax chunks before c0 (sel_idx[0 .. nprev[c0]),
// in pairs), then the diagonal block (c0, c1).  Rows of c1 also see c0 when c0
// chose softmax; both diagonal slots are causal for their own rows.  Slots
// without a chunk are loaded with c0 (finite data) and masked.
//
// Roles (256 threads):
//   warp 0     TMA producer: Q tile once, then K/V blocks into two stages
//   warp 1     TMEM owner + MMA issuer: S_j = Q K_j^T (TMEM), O += P_j V_j (TMEM)
//   warps 4-7  softmax: thread r owns query row r (its TMEM lane); online
//              softmax in the exp2 domain, P_j written to shared memory as the
//              bf16 A operand of the next MMA.  The running max used for the
//              exponent is raised (and O, l rescaled in place) only when a
//              row's max grows by more than 2^8, so P stays <= 256 and the
//              rescale (which waits for the previous P V product) is rare.
// TMEM: two S buffers (2 x 128 columns) + the O accumulator (D columns).
// Every wait is bounded (tc::kWaitLimitNs); on expiry the kernel records an
// error, drains what it issued and exits.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

enum { kFull = 0, kCausal = 1, kNone = 2 };

template <int D>
struct SoftmaxSmem {
  static constexpr int kHalf = 128 * 128;           // bytes of one 128-row x 64-col bf16 block
  static constexpr int kQ = 128 * D * 2;
  static constexpr int kKV = 128 * D * 2;
  static constexpr int kP = 128 * 128 * 2;
  static constexpr int offQ = 0;
  static constexpr int offK = offQ + kQ;           // 2 stages
  static constexpr int offV = offK + 2 * kKV;      // 2 stages
  static constexpr int offP = offV + 2 * kKV;      // 2 buffers
  static constexpr int offBar = offP + 2 * kP;
  static constexpr int kNumBars = 12;
  static constexpr int offTmem = offBar + kNumBars * 8;
  static constexpr int kBytes = offTmem + 16 + 1024;  // + alignment slack
};

// barrier slots
enum { B_Q = 0, B_KVF = 1, B_KVE = 3, B_SF = 5, B_PF = 7, B_OF = 9, B_DONE = 11 };

constexpr float kRescaleLog2 = 8.f;  // lazy-rescale threshold (log2 units)

template <int D>
__global__ void __launch_bounds__(256, 1)
    softmax_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ nprev,
                      const int32_t* __restrict__ sel_idx, const uint8_t* __restrict__ sel, int L, int N,
                      int T, long long BH, float sl2, float* __restrict__ o_s, int* __restrict__ err) {
  using S = SoftmaxSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* Qs = smem + S::offQ;
  uint64_t* bars = (uint64_t*)(smem + S::offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + S::offTmem);

  const long long bid = blockIdx.x;
  const int p = T - 1 - (int)(bid / BH);  // heaviest tiles first
  const long long bh = bid % BH;
  const int c0 = 2 * p, c1 = 2 * p + 1;
  const bool has_c1 = c1 < N;
  const int n0 = nprev[bh * N + c0];
  const int nbp = (n0 + 1) >> 1;  // prefix blocks
  const int nb = nbp + 1;         // + diagonal block
  const bool c0_soft = sel[bh * N + c0] == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row0 = bh * (long long)L;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[B_KVF + s], 1);
      tc::mbar_init(&bars[B_KVE + s], 1);
      tc::mbar_init(&bars[B_SF + s], 1);
      tc::mbar_init(&bars[B_PF + s], 128);
      tc::mbar_init(&bars[B_OF + s], 1);
    }
    tc::mbar_init(&bars[B_DONE], 1);
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
      tc::mbar_arrive_expect_tx(&bars[B_Q], S::kQ);
      for (int h = 0; h < D / 64; ++h)
        for (int rc = 0; rc < 2; ++rc)
          tc::tma_load_2d(Qs + h * S::kHalf + rc * (S::kHalf / 2), &tm_q, 64 * h,
                          (int)(row0 + 128LL * p + 64 * rc), &bars[B_Q]);
      int issued[2] = {0, 0};
      bool ok = true;
      for (int j = 0; j < nb && ok; ++j) {
        const int s = j & 1;
        if (!tc::mbar_wait(&bars[B_KVE + s], ((j >> 1) & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        int ch[2];
        if (j < nbp) {
          ch[0] = sel_idx[bh * N + 2 * j];
          ch[1] = (2 * j + 1 < n0) ? sel_idx[bh * N + 2 * j + 1] : c0;
        } else {
          ch[0] = c0;
          ch[1] = has_c1 ? c1 : c0;
        }
        uint8_t* Ks = smem + S::offK + s * S::kKV;
        uint8_t* Vs = smem + S::offV + s * S::kKV;
        tc::mbar_arrive_expect_tx(&bars[B_KVF + s], 2 * S::kKV);
        for (int slot = 0; slot < 2; ++slot) {
          const int y = (int)(row0 + 64LL * ch[slot]);
          for (int h = 0; h < D / 64; ++h) {
            tc::tma_load_2d(Ks + h * S::kHalf + slot * (S::kHalf / 2), &tm_k, 64 * h, y, &bars[B_KVF + s]);
            tc::tma_load_2d(Vs + h * S::kHalf + slot * (S::kHalf / 2), &tm_v, 64 * h, y, &bars[B_KVF + s]);
          }
        }
        issued[s]++;
      }
      if (ok) {
        // the last commits on the "empty" barriers must land before exit
        for (int s = 0; s < 2; ++s)
          if (issued[s] > 0) tc::mbar_wait(&bars[B_KVE + s], (issued[s] - 1) & 1, err);
      } else {
        // drain loads still in flight
        tc::mbar_wait(&bars[B_Q], 0, nullptr);
        for (int s = 0; s < 2; ++s)
          if (issued[s] > 0) tc::mbar_wait(&bars[B_KVF + s], (issued[s] - 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, D, false, true);
      const uint32_t q_base = tc::smem_u32(Qs);
      bool ok = tc::mbar_wait(&bars[B_Q], 0, err);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!tc::mbar_wait(&bars[B_KVF + s], (j >> 1) & 1, err)) return false;
        tc::fence_after();
        const uint32_t k_base = tc::smem_u32(smem + S::offK + s * S::kKV);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * S::kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + s * 128, tc::smem_desc_sw128(q_base + off, 16, 1024),
                       tc::smem_desc_sw128(k_base + off, 16, 1024), idesc_qk, kk > 0);
        }
        tc::mma_commit(&bars[B_SF + s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nb && ok; ++j) {
        if (j + 1 < nb && !(ok = issue_s(j + 1))) break;
        const int b = j & 1;
        if (!(ok = tc::mbar_wait(&bars[B_PF + b], (j >> 1) & 1, err))) break;
        tc::fence_after();
        const uint32_t p_base = tc::smem_u32(smem + S::offP + b * S::kP);
        const uint32_t v_base = tc::smem_u32(smem + S::offV + b * S::kKV);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          tc::mma_bf16(tmem + 256,
                       tc::smem_desc_sw128(p_base + (kk >> 2) * S::kHalf + (kk & 3) * 32, 16, 1024),
                       tc::smem_desc_sw128(v_base + kk * 2048, S::kHalf, 1024), idesc_pv, (j > 0) || (kk > 0));
        }
        tc::mma_commit(&bars[B_OF + b]);
        tc::mma_commit(&bars[B_KVE + b]);
      }
      tc::mma_commit(&bars[B_DONE]);
      tc::mbar_wait(&bars[B_DONE], 0, err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x - 128;
    const int half = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t o_addr = tmem + 256 + lane_off;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int b = j & 1;
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_SF + b], (j >> 1) & 1, err)))) break;
      tc::fence_after();
      int mode[2];
      if (j < nbp) {
        mode[0] = kFull;
        mode[1] = (2 * j + 1 < n0) ? kFull : kNone;
      } else if (half == 0) {
        mode[0] = kCausal;
        mode[1] = kNone;
      } else {
        mode[0] = has_c1 ? (c0_soft ? kFull : kNone) : kFull;
        mode[1] = has_c1 ? kCausal : kNone;
      }
      const uint32_t s_addr = tmem + b * 128 + lane_off;
      float mx = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float v[32];
        tc::tmem_ld32(s_addr + ch * 32, v);
        tc::tmem_ld_wait();
        const int md = mode[ch >> 1];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = (ch & 1) * 32 + i;
          const bool keep = (md == kFull) || (md == kCausal && key <= rr);
          mx = keep ? fmaxf(mx, v[i]) : mx;
        }
      }
      const float m_cand = mx * sl2;  // every row sees >= 1 key of every block
      // P[b] is free once P_{j-2} V_{j-2} is done
      if (j >= 2 && !(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OF + b], ((j - 2) >> 1) & 1, err))))
        break;
      if (j == 0) {
        m_used = m_cand;
      } else {
        const bool need = m_cand > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold every product so far before it is rescaled in place
          const int jp = j - 1;
          if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OF + (jp & 1)], (jp >> 1) & 1, err)))) break;
          tc::fence_after();
          const float alpha = need ? tc::fast_exp2(m_used - m_cand) : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float v[32];
            tc::tmem_ld32(o_addr + ch * 32, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tc::tmem_st32(o_addr + ch * 32, v);
          }
          tc::tmem_st_wait();
          if (need) {
            l *= alpha;
            m_used = m_cand;
          }
        }
      }
      float sum = 0.f;
      uint8_t* Pb = smem + S::offP + b * S::kP;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float v[32];
        tc::tmem_ld32(s_addr + ch * 32, v);
        tc::tmem_ld_wait();
        const int md = mode[ch >> 1];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = (ch & 1) * 32 + i;
          const bool keep = (md == kFull) || (md == kCausal && key <= rr);
          v[i] = keep ? tc::fast_exp2(fmaf(v[i], sl2, -m_used)) : 0.f;
          sum += v[i];
        }
        uint8_t* row = Pb + (ch >> 1) * S::kHalf + r * 128;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const int g = (ch & 1) * 4 + g4;
          uint4 pk;
          pk.x = tc::pack_bf16x2(v[g4 * 8 + 0], v[g4 * 8 + 1]);
          pk.y = tc::pack_bf16x2(v[g4 * 8 + 2], v[g4 * 8 + 3]);
          pk.z = tc::pack_bf16x2(v[g4 * 8 + 4], v[g4 * 8 + 5]);
          pk.w = tc::pack_bf16x2(v[g4 * 8 + 6], v[g4 * 8 + 7]);
          *(uint4*)(row + ((g ^ (r & 7)) << 4)) = pk;
        }
      }
      l += sum;
      tc::fence_proxy_async_smem();
      tc::fence_before();
      tc::mbar_arrive(&bars[B_PF + b]);
    }
    if (ok) {
      const int jl = nb - 1;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OF + (jl & 1)], (jl >> 1) & 1, err));
    }
    if (ok) {
      tc::fence_after();
      const float inv = 1.f / l;
      const bool valid = (half == 0 || has_c1);
      float* dst = o_s + (size_t)(row0 + 128LL * p + r) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float v[32];
        tc::tmem_ld32(o_addr + ch * 32, v);
        tc::tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            ((float4*)(dst + ch * 32))[i] =
                make_float4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  });
  return fn;
}

}  // namespace

// [rows, D] bf16 row-major matrix viewed as 64 x 64 boxes, 128-byte swizzle.
bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_tc_t(const Problem& p, const void* q, const void* k, const void* v,
                               const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel, float* o_s,
                               int* err, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  const long long rows = p.BH * p.L;
  if (!make_tile_map(&mq, q, rows, D) || !make_tile_map(&mk, k, rows, D) || !make_tile_map(&mv, v, rows, D))
    return cudaErrorInvalidValue;
  auto kern = softmax_tc_kernel<D>;
  const int smem = SoftmaxSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int T = (p.N + 1) / 2;
  const long long blocks = p.BH * T;
  kern<<<(unsigned)blocks, 256, smem, st>>>(mq, mk, mv, nprev, sel_idx, sel, p.L, p.N, T, p.BH,
                                            p.scale * 1.4426950408889634f, o_s, err);
  return cudaGetLastError();
}

cudaError_t launch_softmax_tc(const Problem& p, const void* q, const void* k, const void* v,
                              const int32_t* nprev, const int32_t* sel_idx, const uint8_t* sel, float* o_s,
                              int* err, cudaStream_t st) {
  if (p.BH == 0 || p.N == 0) return cudaSuccess;
  return p.d == 64 ? launch_tc_t<64>(p, q, k, v, nprev, sel_idx, sel, o_s, err, st)
                   : launch_tc_t<128>(p, q, k, v, nprev, sel_idx, sel, o_s, err, st);
}

}  // namespace nats
