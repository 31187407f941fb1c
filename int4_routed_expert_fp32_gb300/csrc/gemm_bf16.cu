// bf16 x bf16 -> fp32 -> bf16 GEMM for the latent projections, y = x W^T with
// the [out, in] weight layout (Kimi K3 latent up-projection page, "Latent
// up-projection"; KimiSparseMoeBlock listing: routed_expert_down_proj and
// routed_expert_up_proj, no bias).
//
// gemm_tc_kernel: persistent CTAs (one per SM) walk 128 x 256 output tiles on
// the 5th-generation tensor cores: a TMA warp streams 128x64 (A) and 256x64
// (B) bf16 tiles with the 128-byte swizzle into a 4-stage ring, one warp
// issues tcgen05.mma (M=128, N=256, K=16) into one of two 256-column TMEM
// accumulators, and four epilogue warps read the other back with tcgen05.ld
// and store bf16 (or fp32) while the next tile's MMAs run.
#include <algorithm>

#include "combine.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace moe {

constexpr int kTcBM = 128, kTcBK = 64, kTcStages = 4;
constexpr int kTcABytes = kTcBM * kTcBK * 2;  // 16 KiB
constexpr int kTcThreads = 192;  // warp 0: TMA, warp 1: MMA + TMEM, warps 2-5: epilogue

template <int BN>
struct TcTile {
  static constexpr int kBBytes = BN * kTcBK * 2;             // 32 KiB (BN 256) .. 16 KiB (128)
  static constexpr int kStageBytes = kTcABytes + kBBytes;
  static constexpr int kSmem = kTcStages * kStageBytes + 1024 + 256;
  // two TMEM accumulators of BN columns, in an allocation of a power of two
  static constexpr uint32_t kCols = 2 * BN <= 256 ? 256u : 512u;
  static_assert(BN % 32 == 0 && 2 * BN <= 512, "accumulator columns");
};

// Persistent: CTA c takes the tiles t = c, c + gridDim.x, ...; tile t is
// (x, y, z) = (t % tn, (t / tn) % tm, t / (tn tm)): the 128 x BN tile (y, x)
// over the K slice [z * kc, min(K, (z + 1) * kc)), stored at columns z * N + n
// of rows of ldc elements (split-K partials side by side; one slice, ldc = N:
// plain C).  Two TMEM accumulators: the epilogue of a tile overlaps the
// MMAs of the next.  The B map is three-dimensional [terms][N][K]: every K
// tile is taken once per term into the same accumulator, so C = A (B_0 + ...
// + B_{terms-1})^T (terms = 1: a plain GEMM).  A second GEMM of the same
// shape and A (mb2, Cout2; tiles after the first GEMM's) can share the
// launch: the shared expert's gate and up projections.
template <bool F32OUT, int BN = 256>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                   const __grid_constant__ CUtensorMap mb2, void* __restrict__ Cout,
                   void* __restrict__ Cout2, int ngemm, int M, int N, int K, int kc, int ldc,
                   int terms, int* status, long long wait_ns) {
  constexpr int kTcBN = BN;
  constexpr int kTcStageBytes = TcTile<BN>::kStageBytes;
  constexpr uint32_t kTcCols = TcTile<BN>::kCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* accfull = empty + kTcStages;  // [2]
  uint64_t* accempty = accfull + 2;       // [2]
  uint64_t* mma_done = accempty + 2;      // the MMA warp's last commit (exit path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, status, wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
    }
    mbar_init(mma_done, 1);
    cta_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int tn = (N + kTcBN - 1) / kTcBN, tm = (M + kTcBM - 1) / kTcBM;
  const int tiles1 = tn * tm * ((K + kc - 1) / kc);  // tiles of one GEMM
  const int tiles = tiles1 * ngemm;
  // K tiles (x terms) of the slice z
  auto ktiles_of = [&](int z) { return (min(K - z * kc, kc) + kTcBK - 1) / kTcBK * terms; };

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensor_map(&ma);
      prefetch_tensor_map(&mb);
      if (ngemm > 1) prefetch_tensor_map(&mb2);
      uint32_t it = 0;
      bool ok = true;
      for (int t2 = blockIdx.x; t2 < tiles && ok; t2 += gridDim.x) {
        const bool second = t2 >= tiles1;
        const int t = second ? t2 - tiles1 : t2;
        const CUtensorMap* bmap = second ? &mb2 : &mb;
        const int n0 = (t % tn) * kTcBN, m0 = ((t / tn) % tm) * kTcBM, z = t / (tn * tm);
        const int ktiles = ktiles_of(z);
        for (int kt = 0; kt < ktiles; ++kt, ++it) {
          const int s = it % kTcStages;
          const uint32_t ph = (it / kTcStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, wt)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kTcStageBytes;
          const int kk = z * kc + (kt / terms) * kTcBK, term = kt % terms;
          mbar_arrive_expect_tx(&full[s], kTcStageBytes);
          tma_g2s_2d(st, &ma, &full[s], kk, m0);
          tma_g2s_3d(st + kTcABytes, bmap, &full[s], kk, n0, term);
        }
      }
      // the issued copies land before the CTA can leave (error path included)
      drain_ring(full, it, kTcStages, status);
    }
  } else if (warp == 1) {
    // the whole warp walks the loop; one elected lane issues (see umma_f16_warp)
    constexpr uint32_t idesc = idesc_bf16(kTcBM, kTcBN);
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int t2 = blockIdx.x; t2 < tiles && ok; t2 += gridDim.x, ++uc) {
      const int b = uc & 1;
      const int t = t2 >= tiles1 ? t2 - tiles1 : t2;
      const int ktiles = ktiles_of(t / (tn * tm));
      if (!__all_sync(0xffffffffu, mbar_wait(&accempty[b], ((uc >> 1) & 1u) ^ 1u, wt))) break;
      tc_fence_after();
      const uint32_t acc = tbase + b * kTcBN;
      for (int kt = 0; kt < ktiles; ++kt, ++it) {
        const int s = it % kTcStages;
        const uint32_t ph = (it / kTcStages) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, wt))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + s * kTcStageBytes;
        const uint64_t da = smem_desc_sw128(st);
        const uint64_t db = smem_desc_sw128(st + kTcABytes);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          umma_f16_warp(acc, da + 2 * kk, db + 2 * kk, idesc, (kt | kk) != 0);
        umma_commit_warp(&empty[s]);
      }
      if (ok) umma_commit_warp(&accfull[b]);
    }
    // every issued MMA completes before TMEM is freed, on the error path too
    umma_commit_warp(mma_done);
    mbar_drain(mma_done, 0, status);
  } else {
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31
    const int q = warp & 3;
    uint32_t uc = 0;
    for (int t2 = blockIdx.x; t2 < tiles; t2 += gridDim.x, ++uc) {
      const int b = uc & 1;
      const bool second = t2 >= tiles1;
      const int t = second ? t2 - tiles1 : t2;
      void* const Cout_t = second ? Cout2 : Cout;
      const int n0 = (t % tn) * kTcBN, m0 = ((t / tn) % tm) * kTcBM, z = t / (tn * tm);
      const int row = m0 + 32 * q + lane;
      // warp-uniform outcome: tcgen05.ld needs the whole warp
      if (!__all_sync(0xffffffffu, mbar_wait(&accfull[b], (uc >> 1) & 1u, wt))) break;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < kTcBN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tbase + (static_cast<uint32_t>(32 * q) << 16) + b * kTcBN + c0, r);
        tmem_ld_wait();
        if (c0 + 32 == kTcBN) {  // the accumulator goes back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[b]);
        }
        const int col = n0 + c0;
        if (F32OUT && row < M && col < N) {
          float* dst = static_cast<float*>(Cout_t) + (size_t)row * ldc + (size_t)z * N + col;
          if (col + 32 <= N && (N & 3) == 0 && (ldc & 3) == 0) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              d4[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                  __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col + i < N) dst[i] = __uint_as_float(r[i]);
          }
        } else if (!F32OUT && row < M && col < N) {
          uint16_t* dst = static_cast<uint16_t*>(Cout_t) + (size_t)row * ldc + (size_t)z * N + col;
          if (col + 32 <= N && (N & 7) == 0 && (ldc & 7) == 0) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w[i] = static_cast<uint32_t>(f32_to_bf16_bits(__uint_as_float(r[8 * v + 2 * i]))) |
                       (static_cast<uint32_t>(f32_to_bf16_bits(__uint_as_float(r[8 * v + 2 * i + 1])))
                        << 16);
              d4[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col + i < N) dst[i] = f32_to_bf16_bits(__uint_as_float(r[i]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTcCols);
  }
}

static bool bf16_map(CUtensorMap* m, const uint16_t* base, int rows, int K, int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(kTcBK), static_cast<uint32_t>(box_rows)};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

// [terms][rows][K] bf16, one box of box_rows rows of one term.
static bool bf16_map3(CUtensorMap* m, const uint16_t* base, int terms, int rows, int K,
                      int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(terms)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(rows) * K * 2};
  const uint32_t box[3] = {static_cast<uint32_t>(kTcBK), static_cast<uint32_t>(box_rows), 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

// y = x w^T, and with w2 set also y2 = x w2^T in the same launch.
template <bool F32OUT, int BN = 256>
static int launch_tc_gemm(const uint16_t* x, const uint16_t* w, int M, int N, int K, int kc,
                          int ldc, int terms, void* y, cudaStream_t s,
                          const uint16_t* w2 = nullptr, void* y2 = nullptr) {
  if (M == 0) return MOE_OK;
  if (kc <= 0 || kc % kTcBK != 0) return MOE_ERR_INVALID;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  CUtensorMap ma, mb, mb2;
  if (!bf16_map(&ma, x, M, K, kTcBM) || !bf16_map3(&mb, w, terms, N, K, BN)) return MOE_ERR_CUDA;
  const int ngemm = w2 ? 2 : 1;
  if (w2) {
    if (!bf16_map3(&mb2, w2, terms, N, K, BN)) return MOE_ERR_CUDA;
  } else {
    mb2 = mb;
  }
  auto kern = gemm_tc_kernel<F32OUT, BN>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    TcTile<BN>::kSmem));
  const long tiles =
      (long)((N + BN - 1) / BN) * ((M + kTcBM - 1) / kTcBM) * ((K + kc - 1) / kc) * ngemm;
  const int grid = static_cast<int>(std::min<long>(tiles, num_sms()));
  kern<<<grid, kTcThreads, TcTile<BN>::kSmem, s>>>(ma, mb, mb2, y, w2 ? y2 : y, ngemm, M, N, K,
                                                     kc, ldc, terms, status, kDefaultWaitNs);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// Tile width of a bf16 GEMM: 256 columns, or 192 when the last wave of
// 256-column tiles would leave more SMs idle (a 2048 x 3584 output: 224 tiles
// of 128 x 256 take two waves of 152 SMs, 304 tiles of 128 x 192 fill two
// exactly); a 192-column tile is taken as 5% slower per column.
static int gemm_tile_n(int M, int N) {
  const long sms = num_sms(), tm = (M + kTcBM - 1) / kTcBM;
  auto cost = [&](int bn) {
    const long tiles = tm * ((N + bn - 1) / bn);
    return static_cast<double>((tiles + sms - 1) / sms) * bn * (bn == 192 ? 1.05 : 1.0);
  };
  return cost(192) < cost(256) ? 192 : 256;
}

int launch_linear_tc(const uint16_t* x, const uint16_t* w, int M, int N, int K, uint16_t* y,
                     cudaStream_t s) {
  const int kc = (K + kTcBK - 1) / kTcBK * kTcBK;
  if (gemm_tile_n(M, N) == 192) return launch_tc_gemm<false, 192>(x, w, M, N, K, kc, N, 1, y, s);
  return launch_tc_gemm<false>(x, w, M, N, K, kc, N, 1, y, s);
}

int launch_linear_tc_f32_splitk(const uint16_t* x, const uint16_t* w, int M, int N, int K, int kc,
                                float* y, cudaStream_t s, const uint16_t* w2, float* y2) {
  const int splits = (K + kc - 1) / kc;
  return launch_tc_gemm<true>(x, w, M, N, K, kc, splits * N, 1, y, s, w2, y2);
}

int launch_linear_tc_f32_terms(const uint16_t* x, const uint16_t* w, int terms, int M, int N, int K,
                               int kc, float* y, cudaStream_t s) {
  const int splits = (K + kc - 1) / kc;
  // 192-column tiles when they divide N (a router of 384 experts: two tiles):
  // an M = 128, N = 192 MMA reads 10 KiB of shared memory per 96 cycles,
  // where N = 128 reads 8 KiB per 64 cycles, the whole shared-memory bandwidth
  if (N % 192 == 0) return launch_tc_gemm<true, 192>(x, w, M, N, K, kc, splits * N, terms, y, s);
  return launch_tc_gemm<true, 128>(x, w, M, N, K, kc, splits * N, terms, y, s);
}

int launch_linear_bf16(const uint16_t* x, const uint16_t* w, int M, int N, int K, uint16_t* y,
                       cudaStream_t s) {
  return launch_linear_tc(x, w, M, N, K, y, s);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_linear_bf16(const uint16_t* x, const uint16_t* w, int M, int N, int K,
                               uint16_t* y, void* stream) {
  moe::Range range_("moe_linear_bf16");
  if (M < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID;
  if (K % 32 != 0 || N % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (!x || !w || !y || !aligned(x, 16) || !aligned(w, 16) || !aligned(y, 4)) return MOE_ERR_INVALID;
  return launch_linear_bf16(x, w, M, N, K, y, static_cast<cudaStream_t>(stream));
}
