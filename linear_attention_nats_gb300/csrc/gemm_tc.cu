// gemm_tc.cu - the dense projections around the layer on the 5th-generation
// tensor cores (tcgen05.mma, fp32 accumulators in TMEM, operands staged by
// TMA), with the per-token work of the projections fused into the epilogue.
//
// "Neural Attention Search Linear (NAtS-L)", technical summary,
// "Kernmechanismen" item 4: the merge weights come from projections of the
// query.  The projections themselves follow the plain Gated DeltaNet form
// (the reading stated beside nats_hybrid_fwd_x in the header):
//   [q | k' | v] = bf16(x W_qkv), k = bf16(k' / |k'|) per head,
//   [a | b] = x W_ab, g = -a_scale softplus(a + b_a), beta = sigmoid(b + b_b),
//   y = bf16(o_flat W_o), o_flat[t] = [o_t,0 | o_t,1 | ...].
//
// One kernel serves both products.  C[M, N] = A[M, K] B[K, N], bf16
// operands, fp32 accumulate; A is K-major (rows of x, or rows of the layer
// output read head by head straight from its [B, H, L, d] layout), B is
// N-major (the weight matrices as stored, [K, N] row-major).  Tiles are
// 128 rows x 256 columns, K in blocks of 64.  A tile's columns are whole
// heads of [q | k' | v] (so the key norm is a per-thread reduction; a tile
// may hold heads of two thirds), or gate columns (the 2H columns of W_ab,
// copied zero-padded to a multiple of 64 and read through their own tensor
// map; the MMA's N is the tile's padded width), or columns of y.
//
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ...
// (columns fastest, so the CTAs in flight share their A rows in L2).
// Roles (256 threads):
//   warp 0     TMA producer: the A tile and the B tile of each K block into
//              a 4-deep ring
//   warp 1     TMEM owner (two 256-column accumulators) and MMA issuer
//              (M = 128, N = 256 or the gate width, K = 16 per instruction)
//   warps 4-7  epilogue: thread r owns row r (its TMEM lane); it reads the
//              tile's accumulator while the next tile's products run into
//              the other accumulator, and stores the rows to their
//              destinations
// Every wait is bounded (tc::kWaitLimitNs); on expiry the kernel records an
// error, drains what it issued and exits.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, NSTAGE = 4;
constexpr int kABytes = BM * BK * 2;        // 16 KiB: 128 lines of 128 B
constexpr int kBBlock = BK * 64 * 2;        // 8 KiB: one 64-column block of a K block
constexpr int kBBytes = (BN / 64) * kBBlock;  // 32 KiB
constexpr int kStage = kABytes + kBBytes;
constexpr int offBar = NSTAGE * kStage;
constexpr int kNumBars = 2 * NSTAGE + 4 + 1;
constexpr int offTmem = offBar + kNumBars * 8;
constexpr int kSmemBytes = offTmem + 16 + 1024;

enum { G_FULL = 0, G_EMPTY = NSTAGE, G_AF = 2 * NSTAGE, G_AE = G_AF + 2, G_DONE = G_AE + 2 };

enum { kModeQKV = 0, kModeOut = 1 };

struct GemmArgs {
  int M, K;         // rows (tokens B L) and reduction length
  int n_main;       // column tiles of 256 over the main B matrix
  int n_cols;       // columns of the main B matrix (stores stop there)
  int gate_cols;    // padded gate columns (multiple of 64), 0: no gate tiles
  int mode;
  int B, H, L, d;
  // kModeQKV epilogue
  __nv_bfloat16 *q, *k, *v;
  float *g, *beta;
  const float *b_a, *a_scale, *b_b;
  int HD;  // H d: width of one third of [q | k' | v]
  // kModeOut epilogue
  __nv_bfloat16* y;
  int ldy;
  int* err;
};

// The first n (a multiple of 8) of the NF values f, as bf16 with 16-byte
// stores (unrolled, so f stays in registers)
template <int NF>
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16* dst, const float (&f)[NF], int n) {
#pragma unroll
  for (int c = 0; c < NF; c += 8) {
    if (c >= n) break;
    uint4 pk;
    pk.x = tc::pack_bf16x2(f[c], f[c + 1]);
    pk.y = tc::pack_bf16x2(f[c + 2], f[c + 3]);
    pk.z = tc::pack_bf16x2(f[c + 4], f[c + 5]);
    pk.w = tc::pack_bf16x2(f[c + 6], f[c + 7]);
    *(uint4*)(dst + c) = pk;
  }
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

template <int D>
__global__ void __launch_bounds__(256, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_bg, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + offBar);
  uint32_t* tmem_slot = (uint32_t*)(smem + offTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_gate = (a.gate_cols + BN - 1) / BN;
  const int nt = a.n_main + n_gate;  // column tiles per row block
  const int mt = (a.M + BM - 1) / BM;
  const long long n_tiles = (long long)mt * nt;
  const int kb_n = (a.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      tc::mbar_init(&bars[G_FULL + s], 1);
      tc::mbar_init(&bars[G_EMPTY + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars[G_AF + b], 1);
      tc::mbar_init(&bars[G_AE + b], 128);
    }
    tc::mbar_init(&bars[G_DONE], 1);
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
      tc::prefetch_tensormap(&tm_a);
      tc::prefetch_tensormap(&tm_b);
      if (a.gate_cols) tc::prefetch_tensormap(&tm_bg);
      long long it = 0;  // K blocks issued so far
      bool ok = true;
      for (long long t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int m = (int)(t / nt), n = (int)(t % nt);
        const bool gate = n >= a.n_main;
        const int gcol0 = (n - a.n_main) * BN;
        const int nblk = gate ? min(BN, a.gate_cols - gcol0) / 64 : BN / 64;
        const int row0 = m * BM;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = (int)(it % NSTAGE);
          const uint32_t par = (uint32_t)(((it / NSTAGE) & 1) ^ 1);
          if (!(ok = tc::mbar_wait(&bars[G_EMPTY + s], par, a.err))) break;
          uint8_t* As = smem + s * kStage;
          uint8_t* Bs = As + kABytes;
          tc::mbar_arrive_expect_tx(&bars[G_FULL + s], kABytes + nblk * kBBlock);
          if (a.mode == kModeOut) {
            // A = o_flat: K index h d + j of row (b, l) is o[b, h, l, j];
            // two 64-row boxes of the [B H, L, d] view (L % 64 == 0, so a box
            // never straddles two sequences; rows past M read as zero)
            const int h = (kb * BK) / D, j0 = (kb * BK) % D;
            for (int half = 0; half < 2; ++half) {
              const int r = row0 + 64 * half;
              const int b = r / a.L, l = r - b * a.L;
              const int bh = b < a.B ? b * a.H + h : a.B * a.H;  // past the end: zero fill
              asm volatile(
                  "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
                  "%4}], [%5];" ::"r"(tc::smem_u32(As + half * (kABytes / 2))),
                  "l"((uint64_t)&tm_a), "r"(j0), "r"(l), "r"(bh), "r"(tc::smem_u32(&bars[G_FULL + s]))
                  : "memory");
            }
          } else {
            tc::tma_load_2d(As, &tm_a, kb * BK, row0, &bars[G_FULL + s]);
          }
          const CUtensorMap* tb = gate ? &tm_bg : &tm_b;
          const int col0 = gate ? gcol0 : n * BN;
          for (int nb = 0; nb < nblk; ++nb)
            tc::tma_load_2d(Bs + nb * kBBlock, tb, col0 + 64 * nb, kb * BK, &bars[G_FULL + s]);
        }
      }
      // drain: every load landed and was consumed
      for (int s = 0; s < NSTAGE; ++s) {
        const long long uses = it > s ? (it - 1 - s) / NSTAGE + 1 : 0;
        if (uses > 0) {
          tc::mbar_wait(&bars[G_FULL + s], (uint32_t)((uses - 1) & 1), nullptr);
          if (ok) tc::mbar_wait(&bars[G_EMPTY + s], (uint32_t)((uses - 1) & 1), a.err);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint64_t ad0 = tc::smem_desc_sw128(tc::smem_u32(smem), 16, 1024);
      const uint64_t bd0 = tc::smem_desc_sw128(tc::smem_u32(smem + kABytes), kBBlock, 1024);
      long long it = 0, tl = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tl) {
        const int n = (int)(t % nt);
        const bool gate = n >= a.n_main;
        const int width = gate ? min(BN, a.gate_cols - (n - a.n_main) * BN) : BN;
        const uint32_t idesc = tc::idesc_bf16_f32(BM, width, false, true);
        const int buf = (int)(tl & 1);
        // the epilogue has read this accumulator's previous tile
        if (tl >= 2 && !(ok = tc::mbar_wait(&bars[G_AE + buf], (uint32_t)(((tl - 2) >> 1) & 1), a.err))) break;
        tc::fence_after();
        const uint32_t tacc = tmem + buf * BN;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = (int)(it % NSTAGE);
          if (!(ok = tc::mbar_wait(&bars[G_FULL + s], (uint32_t)((it / NSTAGE) & 1), a.err))) break;
          tc::fence_after();
          const uint64_t ad = tc::desc_add(ad0, s * kStage), bd = tc::desc_add(bd0, s * kStage);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(tacc, tc::desc_add(ad, kk * 32), tc::desc_add(bd, kk * 2048), idesc, (kb | kk) != 0);
          tc::mma_commit(&bars[G_EMPTY + s]);
        }
        if (!ok) break;
        tc::mma_commit(&bars[G_AF + buf]);
      }
      tc::mma_commit(&bars[G_DONE]);
      tc::mbar_wait(&bars[G_DONE], 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int r = threadIdx.x - 128;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    long long tl = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
      const int m = (int)(t / nt), n = (int)(t % nt);
      const bool gate = n >= a.n_main;
      const int buf = (int)(tl & 1);
      if (!(ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[G_AF + buf], (uint32_t)((tl >> 1) & 1), a.err))))
        break;
      tc::fence_after();
      const uint32_t tacc = tmem + buf * BN + lane_off;
      const int row = m * BM + r;
      const bool valid = row < a.M;
      const int b = row / a.L, l = row - b * a.L;
      if (a.mode == kModeOut) {
        __nv_bfloat16* dst = a.y + (size_t)row * a.ldy + (size_t)n * BN;
        const int ncol = min(BN, a.n_cols - n * BN);  // a multiple of 8
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 64) {
          float f[64];
          tc::tmem_ld32_at<0>(tacc + c0, f);
          tc::tmem_ld32_at<32>(tacc + c0 + 32, f);
          tc::tmem_ld_wait();
          if (valid) store_bf16_row(dst + c0, f, min(64, ncol - c0));
        }
      } else if (gate) {
        // gate columns 0 .. H-1: a of head h; H .. 2H-1: b of head h
        const int gcol0 = (n - a.n_main) * BN;
        const int width = min(BN, a.gate_cols - gcol0);
#pragma unroll 1
        for (int c0 = 0; c0 < width; c0 += 32) {
          float f[32];
          tc::tmem_ld32(tacc + c0, f);
          tc::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              const int col = gcol0 + c0 + x;
              if (col < a.H) {
                const float av = f[x] + (a.b_a ? a.b_a[col] : 0.f);
                const float sp = av > 20.f ? av : log1pf(__expf(av));  // softplus
                a.g[((size_t)b * a.H + col) * a.L + l] = -(a.a_scale ? a.a_scale[col] : 1.f) * sp;
              } else if (col < 2 * a.H) {
                const int hh = col - a.H;
                const float bv = f[x] + (a.b_b ? a.b_b[hh] : 0.f);
                a.beta[((size_t)b * a.H + hh) * a.L + l] = 1.f / (1.f + __expf(-bv));
              }
            }
          }
        }
      } else {
        // whole heads of [q | k' | v]
#pragma unroll 1
        for (int hh = 0; hh < BN / D; ++hh) {
          const int col = n * BN + hh * D;
          if (col >= a.n_cols) break;  // warp-uniform
          const int third = col / a.HD, h = (col % a.HD) / D;
          __nv_bfloat16* base = third == 0 ? a.q : (third == 1 ? a.k : a.v);
          float f[D];
#pragma unroll
          for (int c = 0; c < D; c += 32)
            tc::tmem_ld32(tacc + hh * D + c, *reinterpret_cast<float(*)[32]>(&f[c]));
          tc::tmem_ld_wait();
          if (third == 1) {
            // k = bf16(k' / |k'|), k' the bf16 projection (a zero row stays zero)
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) {
              f[c] = bf16_round(f[c]);
              ss = fmaf(f[c], f[c], ss);
            }
            const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) f[c] *= inv;
          }
          if (valid) store_bf16_row(base + (((size_t)b * a.H + h) * a.L + l) * D, f, D);
        }
      }
      // this thread's reads of the accumulator are complete (tcgen05.wait::ld above)
      tc::fence_before();
      tc::mbar_arrive(&bars[G_AE + buf]);
    }
    (void)ok;
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

EncodeTiledFn encode() {
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

// bf16 [rows, cols] row-major, box (64 columns, box_rows rows), 128-byte swizzle
bool map_2d(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn enc = encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [BH, L, d] (the layer output), box (64, 64, 1), 128-byte swizzle
bool map_3d(CUtensorMap* m, const void* base, long long BH, int L, int d) {
  EncodeTiledFn enc = encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mbg, const GemmArgs& ga, int d,
                   cudaStream_t st) {
  auto kern = d == 64 ? gemm_tc_kernel<64> : gemm_tc_kernel<128>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long tiles = (long long)((ga.M + BM - 1) / BM) * (ga.n_main + (ga.gate_cols + BN - 1) / BN);
  if (tiles == 0) return cudaSuccess;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  kern<<<grid, 256, kSmemBytes, st>>>(ma, mb, mbg, ga);
  return cudaGetLastError();
}

}  // namespace

// W_ab [hidden, 2H] -> [hidden, gc] (gc = 2H rounded up to 64), zero-padded,
// so that its rows meet the tensor map's 16-byte stride rule for any H
__global__ void pad_gate_weights_kernel(const __nv_bfloat16* __restrict__ w, int hidden, int n2h, int gc,
                                        __nv_bfloat16* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)hidden * gc) return;
  const int r = (int)(i / gc), c = (int)(i % gc);
  out[i] = c < n2h ? w[(size_t)r * n2h + c] : __float2bfloat16_rn(0.f);
}

size_t proj_gate_pad_bytes(int H, int hidden) { return (size_t)hidden * ((2 * H + 63) / 64 * 64) * 2; }

cudaError_t launch_proj_qkv_tc(int B, int H, int L, int d, int hidden, const void* x, const void* w_qkv,
                               const void* w_ab, void* w_ab_pad, const float* b_a, const float* a_scale,
                               const float* b_b, void* q, void* k, void* v, float* g, float* beta, int* err,
                               cudaStream_t st) {
  const long long M = (long long)B * L;
  const int HD = H * d;
  if (M == 0 || H == 0) return cudaSuccess;
  const int gc = (2 * H + 63) / 64 * 64;
  {
    const long long n = (long long)hidden * gc;
    pad_gate_weights_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>((const __nv_bfloat16*)w_ab, hidden, 2 * H,
                                                                        gc, (__nv_bfloat16*)w_ab_pad);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap ma, mb, mbg;
  if (!map_2d(&ma, x, M, hidden, BM) || !map_2d(&mb, w_qkv, hidden, 3LL * HD, BK) ||
      !map_2d(&mbg, w_ab_pad, hidden, gc, BK))
    return cudaErrorInvalidValue;
  GemmArgs ga{};
  ga.M = (int)M;
  ga.K = hidden;
  ga.n_main = (3 * HD + BN - 1) / BN;
  ga.n_cols = 3 * HD;
  ga.gate_cols = gc;
  ga.mode = kModeQKV;
  ga.B = B, ga.H = H, ga.L = L, ga.d = d, ga.HD = HD;
  ga.q = (__nv_bfloat16*)q, ga.k = (__nv_bfloat16*)k, ga.v = (__nv_bfloat16*)v;
  ga.g = g, ga.beta = beta, ga.b_a = b_a, ga.a_scale = a_scale, ga.b_b = b_b;
  ga.err = err;
  return launch(ma, mb, mbg, ga, d, st);
}

cudaError_t launch_proj_out_tc(int B, int H, int L, int d, int hidden, const void* o, const void* w_o, void* y,
                               int* err, cudaStream_t st) {
  const long long M = (long long)B * L;
  if (M == 0 || H == 0) return cudaSuccess;
  if (L % 64 != 0) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!map_3d(&ma, o, (long long)B * H, L, d) || !map_2d(&mb, w_o, (long long)H * d, hidden, BK))
    return cudaErrorInvalidValue;
  GemmArgs ga{};
  ga.M = (int)M;
  ga.K = H * d;
  ga.n_main = (hidden + BN - 1) / BN;
  ga.n_cols = hidden;
  ga.gate_cols = 0;
  ga.mode = kModeOut;
  ga.B = B, ga.H = H, ga.L = L, ga.d = d;
  ga.y = (__nv_bfloat16*)y;
  ga.ldy = hidden;
  ga.err = err;
  return launch(ma, mb, mb, ga, d, st);
}

}  // namespace nats
