// Grouped W4A16 expert GEMMs on the 5th-generation tensor cores, for experts
// with many rows (prefill-shaped loads).  Same computation as the stream
// kernel (Kimi exact-generator adaptation page, "The preserved forward form";
// Kimi K2.5 donor-reference "SwiGLU-style gated feed-forward projection"),
// with the weights dequantised once per 128-row token tile.  One persistent
// CTA per SM walks units (token chunk x 256 weight rows: 128 gate + 128 up
// outputs, or 256 down outputs) in K stages of 128 columns:
//   * warp 0 (one thread): TMA of the fp16 activation tile (two 128 x 64
//     boxes, 128-byte swizzle) and of the 256-row x 128-column packed int4
//     tile (64-byte swizzle) into a 4-stage shared-memory ring;
//   * warps 2-17: dequantisation, one weight row and half a stage (two scale
//     groups) per thread, to fp16 q * scale written with tcgen05.st into a
//     2-slot TMEM ring (the A operand).  The activation rows are in pair
//     order (each block of 8 columns stored c0 c4 c1 c5 c2 c6 c3 c7), so the
//     weights are written in the same order, the order of the nibble pairs
//     of a word.  With a bf16 scale (8 significant bits) and |q| <= 8,
//     q * scale has at most 11 significant bits: it is exact in fp16 for
//     scales in [2^-17, 8160] (and zero); a scale outside that range records
//     MOE_ERR_UNSUPPORTED (the stream kernel, which applies scales in fp32,
//     takes any scale).  The activations arrive in fp16 (a copy made once per
//     call; bf16 values are exact in fp16 for 2^-17 <= |x| <= 65504), and the
//     gate/up tiles write h in fp16 for the down tiles.  So, as in the stream
//     kernel, the weights are never rounded silently; a value beyond the fp16
//     range makes its output non-finite and records MOE_ERR_UNSUPPORTED;
//   * warp 1 (whole warp, one elected lane issues): tcgen05.mma kind::f16,
//     A from TMEM (M = 128 weight rows per block, two blocks), B the token
//     tile (N = the chunk's rows rounded up to 16), K = 16, into two
//     128-column fp32 accumulators;
//   * warps 18-25: tcgen05.ld of the accumulators; gate/up units store
//     h = SiLU(G) * U (fp16), releasing the accumulators before the stores;
//     down units store y (bf16, or fp32).
// K stages of 128 columns halve the per-stage barrier waits and handoffs
// against 64-column stages (each mbarrier wait costs a dequantisation warp
// ~130 cycles even on a completed phase).
// act_bits 8 has its own kernel (ffn_tc_q8.cu), which keeps the integer
// partial of every weight group.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "ffn_tc.cuh"
#include "int4_f16.cuh"
#include "tcgen05.cuh"

namespace moe {

constexpr int kTxWM = 128;                     // weight rows per MMA block (M, TMEM lanes)
constexpr int kTxBK = 128;                     // K per stage
constexpr int kTxXK = 64;                      // K per activation box (one 128-byte swizzle atom)
constexpr int kTxQBytes = 2 * kTxWM * kTxBK / 2;  // 16 KiB packed int4 (256 rows x 64 bytes)
constexpr int kTxDqWarps = 16;                 // (lane quarter, block, half of the stage)
constexpr int kTxEpWarps = 8;                  // two per TMEM lane quarter
constexpr int kTxThreads = (2 + kTxDqWarps + kTxEpWarps) * 32;
constexpr uint32_t kTxCols = 512;
constexpr uint32_t kTxASlot = 2 * (kTxBK / 2);  // A columns per stage: 2 blocks x 64
static_assert(kTxDqWarps * 32 == 2 * 2 * kTxWM, "one dequantisation thread per row and half stage");

// Layout for token tiles of at most TN rows.  TN = 128: 4 stages of 48 KiB,
// two 128-column accumulators and two A slots.  TN = 64 (experts of at most
// 64 rows): 6 stages of 32 KiB, two 64-column accumulators and three A slots,
// and the conversion warps in two teams of eight that take alternate stages
// (a warp converts a whole 128-column row of its stages).  Measured on
// GB300 (int4_linear, 128 experts x 64 rows, K = 7168): 0.332 ms with the
// TN = 128 layout, 0.304 ms with this one; each of its three changes alone
// gained 1-3%.
template <int TN>
struct TxCfg {
  static constexpr int kXBoxBytes = TN * kTxXK * 2;         // 16 KiB (TN 128) / 8 KiB (TN 64)
  static constexpr int kXBytes = 2 * kXBoxBytes;
  static constexpr int kStageBytes = kXBytes + kTxQBytes;
  static constexpr int kStages = TN == 128 ? 4 : 6;         // shared-memory ring
  static constexpr int kAStages = TN == 128 ? 2 : 3;        // TMEM ring of dequantised weights
  static constexpr uint32_t kAcc1 = TN;                     // column of the second accumulator
  static constexpr uint32_t kACol = 2 * TN;                 // first A column
  static constexpr bool kTeams = TN != 128;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kACol + kAStages * kTxASlot <= kTxCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory");
  static_assert((2 * kStages + 2 * kAStages + 3) * 8 + 4 <= 256, "barrier area");
};

enum TxMode { kTxGateUp = 0, kTxDown = 1, kTxLinear = 2 };

// STALL (tests only): the producer stops before stage p.stall_at, as if its
// copies never arrived, so that the other roles' waits run out.
template <int MODE, int TN = 128, bool STALL = false>
__global__ void __launch_bounds__(kTxThreads, 1)
    ffn_tc_kernel(const __grid_constant__ TxMaps maps, const TxParams p) {
  using C = TxCfg<TN>;
  constexpr int kTxStages = C::kStages, kTxAStages = C::kAStages;
  constexpr int kTxStageBytes = C::kStageBytes, kTxXBytes = C::kXBytes;
  constexpr int kTxXBoxBytes = C::kXBoxBytes;
  constexpr uint32_t kTxAcc1 = C::kAcc1, kTxACol = C::kACol;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTxStages * kTxStageBytes);
  uint64_t* sfree = full + kTxStages;
  uint64_t* aready = sfree + kTxStages;
  uint64_t* afree = aready + kTxAStages;
  uint64_t* accfull = afree + kTxAStages;
  uint64_t* accempty = accfull + 1;
  uint64_t* mma_done = accempty + 1;  // the MMA warp's last commit (exit path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, p.status, p.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], 1);
    }
    for (int a = 0; a < kTxAStages; ++a) {
      mbar_init(&aready[a], C::kTeams ? kTxDqWarps / 2 : kTxDqWarps);
      mbar_init(&afree[a], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, kTxEpWarps);
    mbar_init(mma_done, 1);
    cta_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTxCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int K = p.K, N = p.N;
  const int tile_n = (MODE == kTxGateUp) ? kTxWM : 2 * kTxWM;  // outputs per unit
  const int n_tiles = (N + tile_n - 1) / tile_n;
  const int units = (*p.n_chunks) * n_tiles;
  const int ksteps = (K + kTxBK - 1) / kTxBK;
  const int G_all = K / kGroup;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&maps.a);
      prefetch_tensor_map(&maps.q0);
      if (MODE == kTxGateUp) prefetch_tensor_map(&maps.q1);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int q = u / n_tiles, jt = u - q * n_tiles;
        const int e = p.chunk_e[q], row0 = p.chunk_row0[q];
        const int n0 = jt * tile_n;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % kTxStages;
          const uint32_t ph = (it / kTxStages) & 1u;
          if ((STALL && static_cast<int>(it) == p.stall_at) || !mbar_wait(&sfree[s], ph ^ 1u, wt)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kTxStageBytes;
          uint8_t* qd = st + kTxXBytes;
          mbar_arrive_expect_tx(&full[s], kTxStageBytes);
          // columns beyond K (a last half stage) read as zeros
          tma_g2s_2d(st, &maps.a, &full[s], ks * kTxBK, row0);
          tma_g2s_2d(st + kTxXBoxBytes, &maps.a, &full[s], ks * kTxBK + kTxXK, row0);
          if (MODE == kTxGateUp) {
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kTxBK / 8), n0, e);
            tma_g2s_3d(qd + kTxQBytes / 2, &maps.q1, &full[s], ks * (kTxBK / 8), n0, e);
          } else {
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kTxBK / 8), n0, e);
          }
        }
      }
      // on every exit (a wait that gave up included) let the issued copies
      // land before the CTA can leave
      drain_ring(full, it, kTxStages, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp walks the loop (uniform operands); one elected lane
    // issues each MMA and commit.
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const int q = u / n_tiles;
      const int rows = p.chunk_rows[q];
      const int nn = rows <= 16 ? 16 : (rows + 15) / 16 * 16;  // MMA N: tokens, multiple of 16
      const uint32_t idesc = idesc_f16(kTxWM, nn);
      if (!__all_sync(0xffffffffu, mbar_wait(accempty, (uc & 1u) ^ 1u, wt)))
        break;
      tc_fence_after();
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const int s = it % kTxStages, a = it % kTxAStages;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&aready[a], (it / kTxAStages) & 1u, wt))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t db0 = smem_desc_sw128(smem + s * kTxStageBytes);
        const uint64_t db1 = smem_desc_sw128(smem + s * kTxStageBytes + kTxXBoxBytes);
        const uint32_t ta = tbase + kTxACol + a * kTxASlot;  // block 0; block 1 at +64
#pragma unroll
        for (int kk = 0; kk < kTxBK / 16; ++kk) {
          const uint64_t db = (kk < kTxXK / 16 ? db0 : db1) + 2 * (kk % (kTxXK / 16));
          umma_f16_ts_warp(tbase, ta + 8 * kk, db, idesc, (ks | kk) != 0);
          umma_f16_ts_warp(tbase + kTxAcc1, ta + kTxBK / 2 + 8 * kk, db, idesc, (ks | kk) != 0);
        }
        umma_commit_warp(&sfree[s]);
        umma_commit_warp(&afree[a]);
      }
      if (ok) umma_commit_warp(accfull);
    }
    // every MMA issued (reading shared memory and TMEM) completes before the
    // CTA frees its TMEM or leaves, on the error path too
    umma_commit_warp(mma_done);
    mbar_drain(mma_done, 0, p.status);
  } else if (warp < 2 + kTxDqWarps) {
    // ----------------------------------------------------- dequantisation
    if constexpr (C::kTeams) {
      // Two teams of eight warps take alternate stages (team = parity of the
      // stage counter); a thread converts its row's whole stage (4 groups).
      // Warps 2-5 / 10-13: team 0, blocks 0 / 1; warps 6-9 / 14-17: team 1.
      const int qd = warp & 3;
      const int blk = (warp - 2) >> 3;
      const int team = ((warp - 2) >> 2) & 1;
      const int m = 32 * qd + lane;
      const int r = blk * kTxWM + m;
      const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
      const int qsw = (r >> 1) & 3;
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int q = u / n_tiles, jt = u - q * n_tiles;
        const int e = p.chunk_e[q];
        const int n0 = jt * tile_n;
        int n;
        const uint16_t* sb;
        if (MODE == kTxGateUp) {
          n = n0 + m;
          sb = blk == 0 ? p.scale0 : p.scale1;
        } else {
          n = n0 + r;
          sb = p.scale0;
        }
        const bool valid = n < N;
        // bf16 scales of groups 4 ks + 2 h and + 1 (h = 0, 1; one 4-byte word
        // each), fetched one of this team's stages ahead; groups beyond K are 0
        const uint16_t* srow = sb + ((size_t)e * N + (valid ? n : 0)) * G_all;
        auto scale_word = [&](int ks2, int h) -> uint32_t {
          return (valid && ks2 < ksteps && 4 * ks2 + 2 * h < G_all)
                     ? *reinterpret_cast<const uint32_t*>(srow + 4 * ks2 + 2 * h)
                     : 0u;
        };
        const int ks0 = (team - static_cast<int>(it)) & 1;  // first stage of this team
        uint32_t pa0 = scale_word(ks0, 0), pa1 = scale_word(ks0, 1);
        bool exact = true;
        for (int ks = ks0; ks < ksteps; ks += 2) {
          const uint32_t sw0 = pa0, sw1 = pa1;
          pa0 = scale_word(ks + 2, 0);
          pa1 = scale_word(ks + 2, 1);
          const uint32_t itk = it + ks;
          const int s = itk % kTxStages, a = itk % kTxAStages;
          // warp-uniform outcome: the tcgen05.st below needs the whole warp
          const bool got = mbar_wait(&full[s], (itk / kTxStages) & 1u, wt) &&
                           mbar_wait(&afree[a], ((itk / kTxAStages) & 1u) ^ 1u, wt);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint8_t* qt = smem + s * kTxStageBytes + kTxXBytes;
          exact &= scales_exact_f16(sw0) && scales_exact_f16(sw1);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // chunks 2h and 2h + 1 of the row (64-byte swizzle: chunk c at c ^ qsw)
            const uint4 w0 = *reinterpret_cast<const uint4*>(qt + r * 64 + (((2 * h) ^ qsw) << 4));
            const uint4 w1 =
                *reinterpret_cast<const uint4*>(qt + r * 64 + (((2 * h + 1) ^ qsw) << 4));
            const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            const uint32_t sw = h ? sw1 : sw0;
            const uint32_t s_lo = scale_f16x2(sw & 0xffffu);
            const uint32_t s_hi = scale_f16x2(sw >> 16);
            uint32_t av[32];  // pair order, as below
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t w = wv[c];
              const uint32_t sc = c < 4 ? s_lo : s_hi;
              const uint32_t w8 = w >> 8;
              av[4 * c + 0] = nib_lo_f16(w, sc);
              av[4 * c + 1] = nib_hi_f16(w, sc);
              av[4 * c + 2] = nib_lo_f16(w8, sc);
              av[4 * c + 3] = nib_hi_f16(w8, sc);
            }
            tmem_st32(tbase + t_lane + kTxACol + a * kTxASlot + blk * (kTxBK / 2) + h * 32, av);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&aready[a]);
        }
        it += ksteps;
        if (!exact) record_status(p.status, MOE_ERR_UNSUPPORTED);
      }
    } else {
      // TMEM lane quarter of this warp: warp % 4.  Warps 2-5: block 0, first
      // half of each stage (K columns 0-63, scale groups 0 and 1); 6-9: block 0,
      // second half (64-127, groups 2 and 3); 10-13 and 14-17: the same for
      // block 1.
      const int qd = warp & 3;
      const int blk = (warp - 2) >> 3;
      const int gh = ((warp - 2) >> 2) & 1;  // half of the stage
      const int m = 32 * qd + lane;        // TMEM lane = row within the block
      const int r = blk * kTxWM + m;       // row within the 256-row tile
      const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
      // int4 rows of 64 bytes, stored with the 64-byte swizzle: 16-byte chunk c
      // of row r sits at chunk c ^ ((r >> 1) & 3); this thread reads chunks
      // 2 gh and 2 gh + 1
      const int qsw = (r >> 1) & 3;
      const uint32_t qoff0 = static_cast<uint32_t>(r * 64 + (((2 * gh) ^ qsw) << 4));
      const uint32_t qoff1 = static_cast<uint32_t>(r * 64 + (((2 * gh + 1) ^ qsw) << 4));
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int q = u / n_tiles, jt = u - q * n_tiles;
        const int e = p.chunk_e[q];
        const int n0 = jt * tile_n;
        int n;
        const uint16_t* sb;
        if (MODE == kTxGateUp) {
          n = n0 + m;
          sb = blk == 0 ? p.scale0 : p.scale1;
        } else {
          n = n0 + r;
          sb = p.scale0;
        }
        const bool valid = n < N;
        // bf16 scales of this thread's two groups of stage ks (4 ks + 2 gh and
        // + 1: one 4-byte word), fetched three stages ahead; groups beyond K
        // (a last half stage) are 0
        const uint16_t* srow = sb + ((size_t)e * N + (valid ? n : 0)) * G_all + 2 * gh;
        auto scale_word = [&](int ks2) -> uint32_t {
          return (valid && ks2 < ksteps && 4 * ks2 + 2 * gh < G_all)
                     ? *reinterpret_cast<const uint32_t*>(srow + 4 * ks2)
                     : 0u;
        };
        uint32_t s_a = scale_word(0), s_b = scale_word(1), s_c = scale_word(2);
        bool exact = true;  // every scale of this unit's row converts exactly
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t sw = s_a;
          s_a = s_b;
          s_b = s_c;
          s_c = scale_word(ks + 3);
          const int s = it % kTxStages, a = it % kTxAStages;
          // warp-uniform outcome: the tcgen05.st below needs the whole warp
          const bool got = mbar_wait(&full[s], (it / kTxStages) & 1u, wt) &&
                           mbar_wait(&afree[a], ((it / kTxAStages) & 1u) ^ 1u, wt);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint8_t* qt = smem + s * kTxStageBytes + kTxXBytes;
          const uint4 w0 = *reinterpret_cast<const uint4*>(qt + qoff0);
          const uint4 w1 = *reinterpret_cast<const uint4*>(qt + qoff1);
          const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          exact &= scales_exact_f16(sw);
          const uint32_t s_lo = scale_f16x2(sw & 0xffffu);  // group 4 ks + 2 gh
          const uint32_t s_hi = scale_f16x2(sw >> 16);      // group 4 ks + 2 gh + 1
          uint32_t av[32];  // pair order: column 4c + j holds weight columns 8c + j, 8c + j + 4
  #pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t w = wv[c];
            const uint32_t sc = c < 4 ? s_lo : s_hi;
            const uint32_t w8 = w >> 8;
            av[4 * c + 0] = nib_lo_f16(w, sc);   // (n0, n4)
            av[4 * c + 1] = nib_hi_f16(w, sc);   // (n1, n5)
            av[4 * c + 2] = nib_lo_f16(w8, sc);  // (n2, n6)
            av[4 * c + 3] = nib_hi_f16(w8, sc);  // (n3, n7)
          }
          tmem_st32(tbase + t_lane + kTxACol + a * kTxASlot + blk * (kTxBK / 2) + gh * 32, av);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&aready[a]);
        }
        if (!exact) record_status(p.status, MOE_ERR_UNSUPPORTED);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // two warps per TMEM lane quarter: half eh takes the 16-token slices
    // 16 eh, 16 eh + 32, ...
    const int qd = warp & 3;
    const int eh = (warp - 2 - kTxDqWarps) >> 2;
    const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
    uint32_t uc = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++uc) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      const int row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
      const int n0 = jt * tile_n;
      // warp-uniform outcome: tcgen05.ld needs the whole warp
      if (!__all_sync(0xffffffffu, mbar_wait(accfull, uc & 1u, wt, 256))) break;
      tc_fence_after();
      bool fin = true;
      if (MODE == kTxGateUp) {
        // h of this lane's feature for the warp's (up to) four 16-token
        // slices, packed in registers; the accumulator is released before the
        // global stores, so the next unit's MMAs start meanwhile
        const int n = n0 + 32 * qd + lane;  // output feature of this lane
        uint32_t hb[4][8];
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const int c0 = 16 * eh + 32 * sl;
#pragma unroll
          for (int i = 0; i < 8; ++i) hb[sl][i] = 0u;
          if (c0 < rows) {  // warp-uniform
            uint32_t g[16], v[16];
            tmem_ld16(tbase + t_lane + c0, g);
            tmem_ld16(tbase + t_lane + kTxAcc1 + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int tok = c0 + i;
              if (tok >= rows || n >= N) continue;
              const float G = __uint_as_float(g[i]), U = __uint_as_float(v[i]);
              // SiLU through the hardware tanh approximation (relative error
              // ~2^-11, the size of h's fp16 rounding)
              const float h = silu_mul(G, U);
              fin &= fabsf(h) <= 65504.0f;
              const uint32_t hbits = __half_as_ushort(__float2half_rn(h));
              hb[sl][i >> 1] |= hbits << (16 * (i & 1));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty);
        if (n < N) {
          uint16_t* hcol = static_cast<uint16_t*>(p.out) + pair_pos(n);
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const int c0 = 16 * eh + 32 * sl;
            size_t o = (size_t)(row0 + c0) * N;
#pragma unroll
            for (int i = 0; i < 16; ++i, o += N) {
              if (c0 + i >= rows) break;
              hcol[o] = static_cast<uint16_t>(hb[sl][i >> 1] >> (16 * (i & 1)));
            }
          }
        }
        if (!fin) record_status(p.status, MOE_ERR_UNSUPPORTED);
      } else {
#pragma unroll 1
        for (int c0 = 16 * eh; c0 < rows; c0 += 32) {
          uint32_t g[16], v[16];
          tmem_ld16(tbase + t_lane + c0, g);
          tmem_ld16(tbase + t_lane + kTxAcc1 + c0, v);
          tmem_ld_wait();
          {
            // y is finite: its inputs are finite fp16 values (checked where
            // they are made) and |q * scale| is bounded, so no check here
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
              const int n = n0 + b2 * kTxWM + 32 * qd + lane;
              if (n >= N) continue;
              size_t o = (size_t)(row0 + c0) * N + n;
#pragma unroll
              for (int i = 0; i < 16; ++i, o += N) {
                if (c0 + i >= rows) break;
                const float y = __uint_as_float(b2 ? v[i] : g[i]);
                if (MODE == kTxDown)
                  static_cast<uint16_t*>(p.out)[o] = f32_to_bf16_bits(y);
                else
                  static_cast<float*>(p.out)[o] = y;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTxCols);
  }
}

static bool act_map(CUtensorMap* m, const uint16_t* x16, int rows, int K, int box_rows = 128) {
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(kTxXK), static_cast<uint32_t>(box_rows)};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

// int8 pair (bytes at bit offsets a, b of w) -> fp16x2, exactly.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t w, int a, int b) {
  const float lo = static_cast<float>(static_cast<int8_t>((w >> a) & 0xffu));
  const float hi = static_cast<float>(static_cast<int8_t>((w >> b) & 0xffu));
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 copy of the bf16 (I8 = false) or int8 (I8 = true) rows below
// *row_count (one warp per row, 8 values per lane step).
template <bool I8>
__global__ void __launch_bounds__(256) to_f16_rows_kernel(const void* __restrict__ src, int R,
                                                          int C, const int32_t* row_count,
                                                          uint16_t* __restrict__ dst) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= R || r >= *row_count) return;
  uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)r * C);
  if (!I8) {
    const uint4* s4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + (size_t)r * C);
    for (int v = lane; v < C / 8; v += 32) {
      uint4 x = s4[v];
      x.x = bf16x2_to_f16x2(x.x);
      x.y = bf16x2_to_f16x2(x.y);
      x.z = bf16x2_to_f16x2(x.z);
      x.w = bf16x2_to_f16x2(x.w);
      d4[v] = x;
    }
  } else {
    const uint2* s2 = reinterpret_cast<const uint2*>(static_cast<const int8_t*>(src) + (size_t)r * C);
    for (int v = lane; v < C / 8; v += 32) {
      const uint2 q = s2[v];
      d4[v] = make_uint4(i8x2_to_f16x2(q.x, 0, 8), i8x2_to_f16x2(q.x, 16, 24),
                         i8x2_to_f16x2(q.y, 0, 8), i8x2_to_f16x2(q.y, 16, 24));
    }
  }
}

// Pair-ordered copy of natural-order rows below *row_count (one warp per
// row): each 8-column block c0..c7 becomes c0 c4 c1 c5 c2 c6 c3 c7, bf16 ->
// fp16 (I8 = false) or int8 -> int8 (I8 = true).
template <bool I8>
__global__ void __launch_bounds__(256) to_pair_rows_kernel(const void* __restrict__ src, int R,
                                                           int C, const int32_t* row_count,
                                                           void* __restrict__ dst, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= R || r >= *row_count) return;
  if (!I8) {
    const uint4* s4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + (size_t)r * C);
    uint4* d4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + (size_t)r * C);
    bool fin = true;
    for (int v = lane; v < C / 8; v += 32) {
      const uint4 x = s4[v];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        fin &= fabsf(f[j]) <= 65504.0f && fabsf(f[j + 4]) <= 65504.0f;
        const __half2 h = __floats2half2_rn(f[j], f[j + 4]);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      d4[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (!fin) record_status(status, MOE_ERR_UNSUPPORTED);
  } else {
    const uint2* s2 = reinterpret_cast<const uint2*>(static_cast<const int8_t*>(src) + (size_t)r * C);
    uint2* d2 = reinterpret_cast<uint2*>(static_cast<int8_t*>(dst) + (size_t)r * C);
    for (int v = lane; v < C / 8; v += 32) {
      const uint2 q = s2[v];
      d2[v] = make_uint2(__byte_perm(q.x, q.y, 0x5140u), __byte_perm(q.x, q.y, 0x7362u));
    }
  }
}

int launch_to_pair_rows(const void* src, bool src_i8, int R, int C, const int32_t* row_count,
                        void* dst, int* status, cudaStream_t s) {
  if (R == 0) return MOE_OK;
  if (src_i8)
    to_pair_rows_kernel<true><<<(R + 7) / 8, 256, 0, s>>>(src, R, C, row_count, dst, status);
  else
    to_pair_rows_kernel<false><<<(R + 7) / 8, 256, 0, s>>>(src, R, C, row_count, dst, status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_to_f16_rows(const void* src, bool src_i8, int R, int C, const int32_t* row_count,
                       uint16_t* dst, cudaStream_t s) {
  if (R == 0) return MOE_OK;
  if (src_i8)
    to_f16_rows_kernel<true><<<(R + 7) / 8, 256, 0, s>>>(src, R, C, row_count, dst);
  else
    to_f16_rows_kernel<false><<<(R + 7) / 8, 256, 0, s>>>(src, R, C, row_count, dst);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static bool packed_map(CUtensorMap* m, const int32_t* w, int E, int N, int K, int rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K / 8) * 4,
                               static_cast<uint64_t>(N) * (K / 8) * 4};
  const uint32_t box[3] = {static_cast<uint32_t>(kTxBK / 8), static_cast<uint32_t>(rows), 1};
  // 64-byte rows with the 64-byte swizzle: conflict-free 16-byte reads per row
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, w, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int MODE, int TN = 128, bool STALL = false>
static int launch_tc(const TxMaps& maps, const TxParams& p, cudaStream_t s) {
  auto kern = ffn_tc_kernel<MODE, TN, STALL>;
  constexpr int smem = TxCfg<TN>::kSmem;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  kern<<<num_sms(), kTxThreads, smem, s>>>(maps, p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// K a multiple of 64: a last half stage reads zero weights and activations
// beyond K.
bool tc_path_supported(int K) { return K % kTxXK == 0; }

int launch_tc_gateup(const uint16_t* x16, int rows_max, int E, int D, int I,
                     const int32_t* gate_packed, const uint16_t* gate_scale,
                     const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                     const int32_t* chunk_e,
                     const int32_t* chunk_row0, const int32_t* chunk_rows, const int32_t* n_chunks,
                     int* status, cudaStream_t s, bool small) {
  TxMaps maps{};
  if (!act_map(&maps.a, x16, rows_max, D, small ? 64 : 128) ||
      !packed_map(&maps.q0, gate_packed, E, I, D, kTxWM) ||
      !packed_map(&maps.q1, up_packed, E, I, D, kTxWM))
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
  return small ? launch_tc<kTxGateUp, 64>(maps, p, s) : launch_tc<kTxGateUp>(maps, p, s);
}

int launch_tc_down(const uint16_t* h16, int rows_max, int E, int D, int I,
                   const int32_t* down_packed, const uint16_t* down_scale, void* y, bool y_f32,
                   const int32_t* chunk_e, const int32_t* chunk_row0, const int32_t* chunk_rows,
                   const int32_t* n_chunks, int* status, cudaStream_t s, bool small) {
  TxMaps maps{};
  if (!act_map(&maps.a, h16, rows_max, I, small ? 64 : 128) ||
      !packed_map(&maps.q0, down_packed, E, D, I, 2 * kTxWM))
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
  if (small)
    return y_f32 ? launch_tc<kTxLinear, 64>(maps, p, s) : launch_tc<kTxDown, 64>(maps, p, s);
  return y_f32 ? launch_tc<kTxLinear>(maps, p, s) : launch_tc<kTxDown>(maps, p, s);
}

int launch_tc_q8_linear_stalled(const uint16_t* x16, const float* x_scale, int rows_max, int E,
                                int N, int K, const int32_t* w_packed, const uint16_t* w_scale,
                                float* y, const int32_t* chunk_e, const int32_t* chunk_row0,
                                const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                                long long wait_ns, int stall_at, cudaStream_t s);

int launch_tc_linear_stalled(const uint16_t* x16, const float* x_scale, int rows_max, int E, int N,
                             int K, const int32_t* w_packed, const uint16_t* w_scale, float* y,
                             const int32_t* chunk_e, const int32_t* chunk_row0,
                             const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                             long long wait_ns, int stall_at, cudaStream_t s, bool small) {
  if (x_scale)
    return launch_tc_q8_linear_stalled(x16, x_scale, rows_max, E, N, K, w_packed, w_scale, y,
                                       chunk_e, chunk_row0, chunk_rows, n_chunks, status, wait_ns,
                                       stall_at, s);
  TxMaps maps{};
  if (!act_map(&maps.a, x16, rows_max, K, small ? 64 : 128) ||
      !packed_map(&maps.q0, w_packed, E, N, K, 2 * kTxWM))
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
  return small ? launch_tc<kTxLinear, 64, true>(maps, p, s) : launch_tc<kTxLinear, 128, true>(maps, p, s);
}

}  // namespace moe
