// Grouped W4A16 expert GEMMs on the tensor cores of two SMs at once
// (cta_group::2), for prefill-shaped batches with act_bits 16.  Same
// computation as ffn_tc_kernel (Kimi exact-generator adaptation page, "The
// preserved forward form"; Kimi K2.5 donor-reference "SwiGLU-style gated
// feed-forward projection"), laid out for a CTA pair.
//
// A cluster of two CTAs walks units: a chunk of <= 256 token rows of one
// expert x 256 weight rows (gate/up: 128 outputs, each CTA 64 gate + 64 up
// rows of the same outputs; down: 256 outputs, 128 per CTA), in K stages of
// 128 columns.  Every MMA is M = 256 (weight rows, 128 in each CTA's tensor
// memory) x N = the chunk's rows rounded up to 32 (token rows, half of them
// in each CTA's shared memory) x K = 16, so each SM dequantises 128 weight
// rows per stage for 256 token columns: half the conversion per MAC of the
// one-CTA kernel, whose 128-row blocks see 128 token columns, with the same
// shared-memory bytes per MAC.  Per CTA:
//   * warp 0 (one thread): TMA of the CTA's half of the token tile (two
//     128 x 64 fp16 boxes, 128-byte swizzle, pair order) and of its 128
//     weight rows x 128 columns of packed int4 (64-byte swizzle) into a
//     5-stage ring, completing on the CTA's own barrier;
//   * warps 2-17: dequantisation, one weight row and one 32-column group per
//     thread, to fp16 q * scale (exact for scales in [2^-17, 8160], else
//     MOE_ERR_UNSUPPORTED) written with tcgen05.st into a 4-slot TMEM ring;
//     each warp then arrives on rank 0's barrier of that slot;
//   * warp 1 of rank 0 (whole warp, one elected lane issues): per stage 8
//     MMAs into one 256-column fp32 accumulator, and commits that arrive on
//     the barriers of both CTAs (shared-memory slot free, TMEM slot free,
//     accumulator full);
//   * warps 18-25 (18-29 for down): the epilogue of the CTA's 128 rows (lane = weight row,
//     column = token).  Gate/up lane quarters hold 16 gate rows (lanes 0-15)
//     and the up rows of the same outputs (lanes 16-31): one shuffle per
//     token pairs them, the gate lane finishing the first 8 tokens of a
//     16-token slice and the up lane the other 8; h = SiLU(G) * U is packed
//     in registers, the accumulator released (an arrival on rank 0's
//     barrier), then stored in fp16, pair order.  Down units store y (bf16,
//     or fp32).
// Every wait is bounded.  Each CTA's copies complete on its own barriers, so
// each producer drains only its own ring; rank 0's last commit arrives in
// both CTAs, and both wait for it before the pair's closing cluster barrier
// and the TMEM release.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "ffn_tc.cuh"
#include "int4_f16.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kPM = 128;                        // weight rows per CTA (TMEM lanes); 256 per pair
constexpr int kPTN = 256;                       // token rows per unit (largest MMA N)
constexpr int kPBK = 128;                       // K per stage
constexpr int kPXK = 64;                        // K per token box (one 128-byte swizzle atom)
constexpr int kPStages = 5;                     // shared-memory ring
constexpr int kPAStages = 4;                    // TMEM ring of dequantised weights
constexpr int kPXBoxBytes = (kPTN / 2) * kPXK * 2;  // 16 KiB: 128 tokens x 64 columns
constexpr int kPXBytes = 2 * kPXBoxBytes;       // 32 KiB: the CTA's half of the token tile
constexpr int kPQBytes = kPM * kPBK / 2;        // 8 KiB packed int4 (128 rows x 64 bytes)
constexpr int kPStageBytes = kPXBytes + kPQBytes;
constexpr int kPDqWarps = 16;                   // (lane quarter, 32-column group of the stage)
constexpr int kPEpWarp0 = 2 + kPDqWarps;
// Epilogue warps: two per lane quarter for gate/up (whose h packing needs the
// registers), three for down, whose accumulator then drains in two thirds of
// the time (2 + 16 + 12 warps: 960 threads).
constexpr int pair_ep_warps(int mode) { return mode == 0 ? 8 : 12; }
constexpr int pair_threads(int mode) { return (2 + kPDqWarps + pair_ep_warps(mode)) * 32; }
constexpr uint32_t kPCols = 512;
constexpr uint32_t kPACol = kPTN;               // A ring after the 256-column accumulator
constexpr uint32_t kPASlot = kPBK / 2;          // 64 columns: 128 fp16 per row
constexpr int kPSmem = kPStages * kPStageBytes + 1024 + 256;
static_assert(kPStageBytes % 1024 == 0, "stage alignment");
static_assert(kPDqWarps * 32 == kPM * (kPBK / kGroup), "one thread per row and group");
static_assert((2 + kPDqWarps + 12) * 32 <= 1024, "threads per CTA");
static_assert(kPACol + kPAStages * kPASlot <= kPCols, "TMEM budget");

enum PMode { kPGateUp = 0, kPDown = 1, kPLinear = 2 };

// Whether q * scale is exact in fp16 for every q in [-8, 7] (one bf16 scale;
// see scales_exact_f16).
__device__ __forceinline__ bool scale_exact_f16(uint32_t s) {
  const uint32_t f = (s >> 7) & 0xFFu;
  return (s & 0x7FFFu) == 0 || (f - 110u) <= 29u;
}

// MMA N of a chunk: its rows rounded up to a multiple of 32 (16 per CTA).
__device__ __forceinline__ int pair_n(int rows) { return rows <= 32 ? 32 : (rows + 31) / 32 * 32; }

// STALL (tests only): each CTA's producer stops before its stage p.stall_at,
// as if its copies never arrived, so that the other roles' waits run out.
template <int MODE, bool STALL = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(MODE), 1)
    ffn_tc_pair_kernel(const __grid_constant__ TxMaps maps, const TxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPStages * kPStageBytes);
  uint64_t* sfree = full + kPStages;
  uint64_t* aready = sfree + kPStages;   // rank 0: both CTAs' conversion warps
  uint64_t* afree = aready + kPAStages;
  uint64_t* accfull = afree + kPAStages;
  uint64_t* accempty = accfull + 1;      // rank 0: both CTAs' epilogue warps
  uint64_t* mma_done = accempty + 1;     // rank 0's last commit (exit path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, p.status, p.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], 1);
    }
    for (int a = 0; a < kPAStages; ++a) {
      mbar_init(&aready[a], 2 * kPDqWarps);
      mbar_init(&afree[a], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, 2 * pair_ep_warps(MODE));
    mbar_init(mma_done, 1);
    cta_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers exist before either CTA arrives on the other's
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int K = p.K, N = p.N;
  const int tile_n = (MODE == kPGateUp) ? kPM : 2 * kPM;  // outputs per unit (pair)
  const int n_tiles = (N + tile_n - 1) / tile_n;
  const int units = (*p.n_chunks) * n_tiles;
  const int ksteps = (K + kPBK - 1) / kPBK;
  const int G_all = K / kGroup;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&maps.a);
      prefetch_tensor_map(&maps.q0);
      if (MODE == kPGateUp) prefetch_tensor_map(&maps.q1);
      uint32_t it = 0;
      bool ok = true;
      for (int u = pair; u < units && ok; u += n_pairs) {
        const int q = u / n_tiles, jt = u - q * n_tiles;
        const int e = p.chunk_e[q];
        // this CTA's half of the token columns
        const int trow = p.chunk_row0[q] + static_cast<int>(rank) * (pair_n(p.chunk_rows[q]) / 2);
        const int n0 = jt * tile_n;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % kPStages;
          const uint32_t ph = (it / kPStages) & 1u;
          if ((STALL && static_cast<int>(it) == p.stall_at) ||
              !mbar_wait(&sfree[s], ph ^ 1u, wt)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kPStageBytes;
          uint8_t* qd = st + kPXBytes;
          mbar_arrive_expect_tx(&full[s], kPStageBytes);
          // columns beyond K (a last half stage) and rows beyond the
          // activations read as zeros
          tma_g2s_2d(st, &maps.a, &full[s], ks * kPBK, trow);
          tma_g2s_2d(st + kPXBoxBytes, &maps.a, &full[s], ks * kPBK + kPXK, trow);
          if (MODE == kPGateUp) {
            const int nr = n0 + 64 * static_cast<int>(rank);
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kPBK / 8), nr, e);
            tma_g2s_3d(qd + kPQBytes / 2, &maps.q1, &full[s], ks * (kPBK / 8), nr, e);
          } else {
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kPBK / 8), n0 + kPM * static_cast<int>(rank), e);
          }
        }
      }
      // on every exit let the issued copies land before the CTA can leave
      drain_ring(full, it, kPStages, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (rank == 0) {
      uint32_t it = 0, uc = 0;
      bool ok = true;
      for (int u = pair; u < units && ok; u += n_pairs, ++uc) {
        const int q = u / n_tiles;
        const uint32_t idesc = idesc_f16(2 * kPM, pair_n(p.chunk_rows[q]));
        if (!__all_sync(0xffffffffu, mbar_wait(accempty, (uc & 1u) ^ 1u, wt))) break;
        tc_fence_after();
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % kPStages, a = it % kPAStages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&aready[a], (it / kPAStages) & 1u, wt))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t db0 = smem_desc_sw128(smem + s * kPStageBytes);
          const uint64_t db1 = smem_desc_sw128(smem + s * kPStageBytes + kPXBoxBytes);
          const uint32_t ta = tbase + kPACol + a * kPASlot;
#pragma unroll
          for (int kk = 0; kk < kPBK / 16; ++kk) {
            const uint64_t db = (kk < kPXK / 16 ? db0 : db1) + 2 * (kk % (kPXK / 16));
            umma_pair_f16_ts_warp(tbase, ta + 8 * kk, db, idesc, (ks | kk) != 0);
          }
          umma_pair_commit_warp(&sfree[s]);
          umma_pair_commit_warp(&afree[a]);
        }
        if (ok) umma_pair_commit_warp(accfull);
      }
      // every MMA issued (reading both CTAs' shared and tensor memory)
      // completes before either CTA frees its TMEM or leaves (below)
      umma_pair_commit_warp(mma_done);
    }
  } else if (warp < kPEpWarp0) {
    // ----------------------------------------------------- dequantisation
    // lane quarter warp % 4; group gq of each stage (K columns 32 gq ..)
    const int qd = warp & 3;
    const int gq = (warp - 2) >> 2;
    const int m = 32 * qd + lane;  // TMEM lane = weight row of this CTA
    // shared-memory row of this lane's weights: gate/up stages hold the
    // CTA's 64 gate rows, then its 64 up rows
    int srow, nloc;
    if (MODE == kPGateUp) {
      nloc = 64 * static_cast<int>(rank) + 16 * qd + (lane & 15);
      srow = (lane < 16 ? 0 : 64) + 16 * qd + (lane & 15);
    } else {
      nloc = kPM * static_cast<int>(rank) + m;
      srow = m;
    }
    // 64-byte rows with the 64-byte swizzle: 16-byte chunk c of row r sits
    // at chunk c ^ ((r >> 1) & 3)
    const uint32_t qoff = static_cast<uint32_t>(srow * 64 + ((gq ^ ((srow >> 1) & 3)) << 4));
    const uint16_t* sb = (MODE == kPGateUp && lane >= 16) ? p.scale1 : p.scale0;
    const uint32_t t_col = (static_cast<uint32_t>(32 * qd) << 16) + kPACol + gq * 16;
    const uint32_t leader_aready = mapa_shared(aready, 0);
    uint32_t it = 0;
    bool ok = true;
    for (int u = pair; u < units && ok; u += n_pairs) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      const int e = p.chunk_e[q];
      const int n = jt * tile_n + nloc;
      const bool valid = n < N;
      // bf16 scale of this thread's group of stage ks, fetched three stages
      // ahead; groups beyond K (a last half stage) are 0
      const uint16_t* srw = sb + ((size_t)e * N + (valid ? n : 0)) * G_all + gq;
      auto scale_of = [&](int ks2) -> uint32_t {
        return (valid && 4 * ks2 + gq < G_all) ? static_cast<uint32_t>(srw[4 * ks2]) : 0u;
      };
      uint32_t s_a = scale_of(0), s_b = scale_of(1), s_c = scale_of(2);
      bool exact = true;  // every scale of this unit's row converts exactly
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const uint32_t sw = s_a;
        s_a = s_b;
        s_b = s_c;
        s_c = scale_of(ks + 3);
        const int s = it % kPStages, a = it % kPAStages;
        // warp-uniform outcome: the tcgen05.st below needs the whole warp
        const bool got = mbar_wait(&full[s], (it / kPStages) & 1u, wt) &&
                         mbar_wait(&afree[a], ((it / kPAStages) & 1u) ^ 1u, wt);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint4 w4 = *reinterpret_cast<const uint4*>(smem + s * kPStageBytes + kPXBytes + qoff);
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
        exact &= scale_exact_f16(sw);
        const uint32_t s2 = scale_f16x2(sw);
        uint32_t av[16];  // pair order: column 4c + j holds weight columns 8c + j, 8c + j + 4
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w = wv[c];
          const uint32_t w8 = w >> 8;
          av[4 * c + 0] = nib_lo_f16(w, s2);   // (n0, n4)
          av[4 * c + 1] = nib_hi_f16(w, s2);   // (n1, n5)
          av[4 * c + 2] = nib_lo_f16(w8, s2);  // (n2, n6)
          av[4 * c + 3] = nib_hi_f16(w8, s2);  // (n3, n7)
        }
        tmem_st16(tbase + t_col + a * kPASlot, av);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(leader_aready + 8u * a);
      }
      if (!exact) record_status(p.status, MOE_ERR_UNSUPPORTED);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // nq warps per TMEM lane quarter: warp eh of a quarter takes the 16-token
    // slices 16 eh, 16 eh + 16 nq, ...
    constexpr int nq = pair_ep_warps(MODE) / 4;
    const int qd = warp & 3;
    const int eh = (warp - kPEpWarp0) >> 2;
    const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
    const uint32_t leader_accempty = mapa_shared(accempty, 0);
    uint32_t uc = 0;
    for (int u = pair; u < units; u += n_pairs, ++uc) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      const int row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
      const int n0 = jt * tile_n;
      // warp-uniform outcome: tcgen05.ld needs the whole warp
      if (!__all_sync(0xffffffffu, mbar_wait(accfull, uc & 1u, wt, 256))) break;
      tc_fence_after();
      if (MODE == kPGateUp) {
        const bool up = lane >= 16;
        const int n = n0 + 64 * static_cast<int>(rank) + 16 * qd + (lane & 15);
        const int tsh = up ? 8 : 0;  // first token of a slice this lane finishes
        bool fin = true;
        uint32_t hb[8][4];
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
          const int c0 = 16 * eh + 32 * sl;
#pragma unroll
          for (int i = 0; i < 4; ++i) hb[sl][i] = 0u;
          if (c0 < rows) {  // warp-uniform
            uint32_t v[16];
            tmem_ld16(tbase + t_lane + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              // the gate lane sends U's partner value for tokens 8-15, the up
              // lane its U for tokens 0-7
              const uint32_t other = __shfl_xor_sync(0xffffffffu, up ? v[i] : v[8 + i], 16);
              const float G = __uint_as_float(up ? other : v[i]);
              const float U = __uint_as_float(up ? v[8 + i] : other);
              if (c0 + tsh + i >= rows || n >= N) continue;
              const float h = silu_mul(G, U);
              fin &= fabsf(h) <= 65504.0f;
              const uint32_t hbits = __half_as_ushort(__float2half_rn(h));
              hb[sl][i >> 1] |= hbits << (16 * (i & 1));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(leader_accempty);
        if (n < N) {
          uint16_t* hcol = static_cast<uint16_t*>(p.out) + pair_pos(n);
#pragma unroll
          for (int sl = 0; sl < 8; ++sl) {
            const int t0 = 16 * eh + 32 * sl + tsh;
            size_t o = (size_t)(row0 + t0) * N;
#pragma unroll
            for (int i = 0; i < 8; ++i, o += N) {
              if (t0 + i >= rows) break;
              hcol[o] = static_cast<uint16_t>(hb[sl][i >> 1] >> (16 * (i & 1)));
            }
          }
        }
        if (!fin) record_status(p.status, MOE_ERR_UNSUPPORTED);
      } else {
        const int n = n0 + kPM * static_cast<int>(rank) + 32 * qd + lane;
#pragma unroll 1
        for (int c0 = 16 * eh; c0 < rows; c0 += 16 * nq) {
          uint32_t v[16];
          tmem_ld16(tbase + t_lane + c0, v);
          tmem_ld_wait();
          if (c0 + 16 * nq >= rows) {
            // the last slice is in registers: release the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(leader_accempty);
          }
          // y is finite: its inputs are finite fp16 values (checked where
          // they are made) and |q * scale| is bounded, so no check here
          if (n < N) {
            size_t o = (size_t)(row0 + c0) * N + n;
#pragma unroll
            for (int i = 0; i < 16; ++i, o += N) {
              if (c0 + i >= rows) break;
              const float y = __uint_as_float(v[i]);
              if (MODE == kPDown)
                static_cast<uint16_t*>(p.out)[o] = f32_to_bf16_bits(y);
              else
                static_cast<float*>(p.out)[o] = y;
            }
          }
        }
        if (16 * eh >= rows) {
          // no slice for this warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(leader_accempty);
        }
      }
    }
  }
  // every pair MMA is done, and every arrival on the other CTA's barriers
  // made, before either CTA releases the pair's tensor memory or leaves
  tc_fence_before();
  __syncthreads();
  if (warp == 1) mbar_drain(mma_done, 0, p.status);
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, kPCols);
  }
}

static bool pair_act_map(CUtensorMap* m, const uint16_t* x16, int rows, int K) {
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(kPXK), static_cast<uint32_t>(kPTN / 2)};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

static bool pair_packed_map(CUtensorMap* m, const int32_t* w, int E, int N, int K, int rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K / 8) * 4,
                               static_cast<uint64_t>(N) * (K / 8) * 4};
  const uint32_t box[3] = {static_cast<uint32_t>(kPBK / 8), static_cast<uint32_t>(rows), 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, w, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

// Pairs of this kernel that fit on the device at once (0: none).
template <int MODE, bool STALL = false>
static int pair_grid_clusters() {
  auto kern = ffn_tc_pair_kernel<MODE, STALL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * ((num_sms() + 1) / 2));
  cfg.blockDim = dim3(pair_threads(MODE));
  cfg.dynamicSmemBytes = kPSmem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int MODE, bool STALL = false>
static int launch_pair(const TxMaps& maps, const TxParams& p, cudaStream_t s) {
  static int clusters[64] = {};  // per device: pairs resident at once (0: not yet known)
  int dev = 0;
  MOE_TRY_CUDA(cudaGetDevice(&dev));
  int& n = clusters[dev & 63];
  if (n == 0) n = pair_grid_clusters<MODE, STALL>();
  if (n <= 0) return MOE_ERR_UNSUPPORTED;
  auto kern = ffn_tc_pair_kernel<MODE, STALL>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem));
  kern<<<2 * n, pair_threads(MODE), kPSmem, s>>>(maps, p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

int launch_tc_pair_gateup(const uint16_t* x16, int rows_max, int E, int D, int I,
                          const int32_t* gate_packed, const uint16_t* gate_scale,
                          const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                          const int32_t* chunk_e, const int32_t* chunk_row0,
                          const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                          cudaStream_t s) {
  TxMaps maps{};
  if (!pair_act_map(&maps.a, x16, rows_max, D) ||
      !pair_packed_map(&maps.q0, gate_packed, E, I, D, kPM / 2) ||
      !pair_packed_map(&maps.q1, up_packed, E, I, D, kPM / 2))
    return MOE_ERR_CUDA;
  TxParams p{};
  p.scale0 = gate_scale;
  p.scale1 = up_scale;
  p.out = h;
  p.chunk_e = chunk_e;
  p.chunk_row0 = chunk_row0;
  p.chunk_rows = chunk_rows;
  p.n_chunks = n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = D;
  p.N = I;
  return launch_pair<kPGateUp>(maps, p, s);
}

int launch_tc_pair_down(const uint16_t* h16, int rows_max, int E, int D, int I,
                        const int32_t* down_packed, const uint16_t* down_scale, void* y,
                        bool y_f32, const int32_t* chunk_e, const int32_t* chunk_row0,
                        const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                        cudaStream_t s) {
  TxMaps maps{};
  if (!pair_act_map(&maps.a, h16, rows_max, I) ||
      !pair_packed_map(&maps.q0, down_packed, E, D, I, kPM))
    return MOE_ERR_CUDA;
  maps.q1 = maps.q0;
  TxParams p{};
  p.scale0 = down_scale;
  p.scale1 = down_scale;
  p.out = y;
  p.chunk_e = chunk_e;
  p.chunk_row0 = chunk_row0;
  p.chunk_rows = chunk_rows;
  p.n_chunks = n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = I;
  p.N = D;
  return y_f32 ? launch_pair<kPLinear>(maps, p, s) : launch_pair<kPDown>(maps, p, s);
}

int launch_tc_pair_linear_stalled(const uint16_t* x16, int rows_max, int E, int N, int K,
                                  const int32_t* w_packed, const uint16_t* w_scale, float* y,
                                  const int32_t* chunk_e, const int32_t* chunk_row0,
                                  const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                                  long long wait_ns, int stall_at, cudaStream_t s) {
  TxMaps maps{};
  if (!pair_act_map(&maps.a, x16, rows_max, K) || !pair_packed_map(&maps.q0, w_packed, E, N, K, kPM))
    return MOE_ERR_CUDA;
  maps.q1 = maps.q0;
  TxParams p{};
  p.scale0 = w_scale;
  p.scale1 = w_scale;
  p.out = y;
  p.chunk_e = chunk_e;
  p.chunk_row0 = chunk_row0;
  p.chunk_rows = chunk_rows;
  p.n_chunks = n_chunks;
  p.status = status;
  p.wait_ns = wait_ns;
  p.stall_at = stall_at;
  p.K = K;
  p.N = N;
  return launch_pair<kPLinear, true>(maps, p, s);
}

bool tc_pair_available() {
  static int avail[64] = {};  // per device: 0 unknown, 1 yes, -1 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int& a = avail[dev & 63];
  if (a == 0) a = pair_grid_clusters<kPGateUp>() > 0 && pair_grid_clusters<kPDown>() > 0 ? 1 : -1;
  return a > 0;
}

}  // namespace moe
