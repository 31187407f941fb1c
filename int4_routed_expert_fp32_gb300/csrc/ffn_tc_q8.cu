// Exact-mode (act_bits 8) grouped int4 x int8 expert GEMMs on the
// 5th-generation tensor cores, for experts with many rows.  The Kimi
// exact-generator adaptation page ("Sources & provenance": an exact int4
// multiply-accumulate; "The preserved forward form": activation quantisation,
// scales and accumulator bounds are part of the form) fixes what is computed:
// for every output n, row r and 32-column weight group g the integer partial
//   P[r, n, g] = sum over the group's columns c of q_x[r, c] * q_w[n, c]
// is exact, and the output is
//   y[r, n] = sc_x[r] * ( ... fma(s_w[n, 1], P[r,n,1], fma(s_w[n, 0], P[r,n,0], 0)) ... )
// in fp32, the groups taken in K order (the stream kernel forms the same chain,
// so both kernels give the same bits).
//
// The integer partials come from the tensor cores: tcgen05.mma kind::f16 on
// fp16 operands that hold integers exactly (|q_w| <= 8, |q_x| <= 127), with
// fp32 accumulation restarted for every group: two K = 16 MMAs per group, so
// every partial sum is an integer of magnitude <= 32 * 8 * 127 < 2^24 and the
// accumulator holds P exactly.  Whole-K integer sums stay far inside int32
// (K * 8 * 127 = 7,282,688 at K = 7168), and the kernel never forms one.
//
// One persistent CTA per SM walks units (a chunk of <= 128 token rows x 128
// weight rows: 64 gate + 64 up rows of the same outputs, or 128 down rows) in
// K stages of 128 columns (4 groups):
//   * warp 0 (one thread): TMA of the fp16 copy of the int8 rows (two 128 x 64
//     boxes, 128-byte swizzle) and of the 128-row x 128-column packed int4
//     tile (64-byte swizzle) into a 4-stage shared-memory ring;
//   * warps 2-5: the integer codes q as exact fp16 (pair order), one row of
//     a stage per thread, written with tcgen05.st into a 2-slot TMEM ring
//     (the MMA's A operand, M = 128 weight rows);
//   * warp 1 (whole warp, one elected lane issues): per group two MMAs into
//     one of three 128-column TMEM group buffers, committed per group;
//   * warps 6-13: per group, tcgen05.ld of the partials (lane = weight row,
//     column = token) in four 16-token pieces, each accumulated as
//     y = fma(s_w, P, y) in registers (64 tokens per thread, two warps per
//     lane quarter), and release of the buffer after the last piece is read.  After the last group a gate/up unit pairs each gate
//     lane with its up lane (lanes i and i + 16 of a lane quarter) and stores
//     h = SiLU(G) * U in bf16, pair order; a down unit stores y (bf16, or
//     fp32 for the plain linear).
// WP (tests only): every partial P is also stored, as int32, to p.partials
// [rows_max, N, K/32].
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "ffn_tc.cuh"
#include "tcgen05.cuh"

namespace moe {

constexpr int kQM = 128;                        // weight rows per unit (TMEM lanes, MMA M)
constexpr int kQTN = 128;                       // token rows per unit (largest MMA N)
constexpr int kQBK = 128;                       // K per stage
constexpr int kQXK = 64;                        // K per token box (one 128-byte swizzle atom)
constexpr int kQStages = 4;                     // shared-memory ring
constexpr int kQAStages = 2;                    // TMEM ring of the integer weight codes
constexpr int kQGBufs = 3;                      // TMEM group buffers
constexpr int kQXBoxBytes = kQTN * kQXK * 2;    // 16 KiB
constexpr int kQXBytes = 2 * kQXBoxBytes;       // 32 KiB token tile
constexpr int kQQBytes = kQM * kQBK / 2;        // 8 KiB packed int4 (128 rows x 64 bytes)
constexpr int kQStageBytes = kQXBytes + kQQBytes;
constexpr int kQDqWarps = 4;                    // one per lane quarter, a whole stage per row
constexpr int kQEpWarps = 8;                    // (lane quarter, half of the tokens)
constexpr int kQThreads = (2 + kQDqWarps + kQEpWarps) * 32;
constexpr uint32_t kQCols = 512;
constexpr uint32_t kQACol = kQGBufs * kQTN;     // A ring after the group buffers
constexpr uint32_t kQASlot = kQBK / 2;          // 64 columns: 128 fp16 per row
constexpr int kQSmem = kQStages * kQStageBytes + 1024 + 256;
constexpr int kQEpCols = kQTN / 2;              // tokens per epilogue thread
static_assert(kQStageBytes % 1024 == 0, "stage alignment");
static_assert(kQDqWarps * 32 == kQM, "one conversion thread per row");
static_assert(kQACol + kQAStages * kQASlot <= kQCols, "TMEM budget");

enum QMode { kQGateUp = 0, kQDown = 1, kQLinear = 2 };

// Two nibbles (bits 0-3 and 16-19 of v, two's complement) -> fp16x2 q,
// exactly: (n ^ 8) in the low mantissa bits of 1024.0 gives 1032 + q, minus
// 1032.
__device__ __forceinline__ uint32_t q_lo_f16(uint32_t v) {
  uint32_t m, r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64086408, 0x6a;" : "=r"(m) : "r"(v));  // (v & a) ^ b
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(0x64086408u));
  return r;
}

// Nibbles at bits 4-7 and 20-23: the half is 1024 + 16 (n ^ 8); times 1/16
// minus 72 gives q, exactly.
__device__ __forceinline__ uint32_t q_hi_f16(uint32_t v) {
  uint32_t m, r;
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64806480, 0x6a;" : "=r"(m) : "r"(v));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(m), "r"(0x2C002C00u), "r"(0xD480D480u));
  return r;
}

// STALL (tests only): the producer stops before stage p.stall_at, as if its
// copies never arrived, so that the other roles' waits run out.
template <int MODE, bool WP, bool STALL = false>
__global__ void __launch_bounds__(kQThreads, 1)
    ffn_tc_q8_kernel(const __grid_constant__ TxMaps maps, const TxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQStages * kQStageBytes);
  uint64_t* sfree = full + kQStages;
  uint64_t* aready = sfree + kQStages;
  uint64_t* afree = aready + kQAStages;
  uint64_t* gfull = afree + kQAStages;
  uint64_t* gempty = gfull + kQGBufs;
  uint64_t* mma_done = gempty + kQGBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, p.status, p.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], 1);
    }
    for (int a = 0; a < kQAStages; ++a) {
      mbar_init(&aready[a], kQDqWarps);
      mbar_init(&afree[a], 1);
    }
    for (int b = 0; b < kQGBufs; ++b) {
      mbar_init(&gfull[b], 1);
      mbar_init(&gempty[b], kQEpWarps);
    }
    mbar_init(mma_done, 1);
    cta_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kQCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int K = p.K, N = p.N;
  const int tile_n = (MODE == kQGateUp) ? kQM / 2 : kQM;  // outputs per unit
  const int n_tiles = (N + tile_n - 1) / tile_n;
  const int units = (*p.n_chunks) * n_tiles;
  const int ksteps = (K + kQBK - 1) / kQBK;
  const int G_all = K / kGroup;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&maps.a);
      prefetch_tensor_map(&maps.q0);
      if (MODE == kQGateUp) prefetch_tensor_map(&maps.q1);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int q = u / n_tiles, jt = u - q * n_tiles;
        const int e = p.chunk_e[q], row0 = p.chunk_row0[q];
        const int n0 = jt * tile_n;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % kQStages;
          const uint32_t ph = (it / kQStages) & 1u;
          if ((STALL && static_cast<int>(it) == p.stall_at) || !mbar_wait(&sfree[s], ph ^ 1u, wt)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kQStageBytes;
          uint8_t* qd = st + kQXBytes;
          mbar_arrive_expect_tx(&full[s], kQStageBytes);
          // columns beyond K (a last half stage) and rows beyond N read as zeros
          tma_g2s_2d(st, &maps.a, &full[s], ks * kQBK, row0);
          tma_g2s_2d(st + kQXBoxBytes, &maps.a, &full[s], ks * kQBK + kQXK, row0);
          if (MODE == kQGateUp) {
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kQBK / 8), n0, e);
            tma_g2s_3d(qd + kQQBytes / 2, &maps.q1, &full[s], ks * (kQBK / 8), n0, e);
          } else {
            tma_g2s_3d(qd, &maps.q0, &full[s], ks * (kQBK / 8), n0, e);
          }
        }
      }
      drain_ring(full, it, kQStages, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    uint32_t it = 0, gi = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int q = u / n_tiles;
      const int rows = p.chunk_rows[q];
      const int nn = rows <= 16 ? 16 : (rows + 15) / 16 * 16;  // MMA N: tokens, multiple of 16
      const uint32_t idesc = idesc_f16(kQM, nn);
      for (int ks = 0; ks < ksteps && ok; ++ks, ++it) {
        const int s = it % kQStages, a = it % kQAStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&aready[a], (it / kQAStages) & 1u, wt))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t db0 = smem_desc_sw128(smem + s * kQStageBytes);
        const uint64_t db1 = smem_desc_sw128(smem + s * kQStageBytes + kQXBoxBytes);
        const uint32_t ta = tbase + kQACol + a * kQASlot;
        const int ng = min(kQBK / kGroup, G_all - ks * (kQBK / kGroup));
        for (int gg = 0; gg < ng; ++gg, ++gi) {
          const int b = gi % kQGBufs;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&gempty[b], ((gi / kQGBufs) & 1u) ^ 1u, wt))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int kx = 2 * gg + kk;  // K = 16 step within the stage
            const uint64_t db = (kx < kQXK / 16 ? db0 : db1) + 2 * (kx % (kQXK / 16));
            umma_f16_ts_warp(tbase + b * kQTN, ta + 8 * kx, db, idesc, kk);
          }
          umma_commit_warp(&gfull[b]);
        }
        umma_commit_warp(&sfree[s]);
        umma_commit_warp(&afree[a]);
      }
    }
    // every issued MMA completes before the CTA frees its TMEM or leaves
    umma_commit_warp(mma_done);
    mbar_drain(mma_done, 0, p.status);
  } else if (warp < 2 + kQDqWarps) {
    // ---------------------------------------------- integer codes as fp16
    const int qd = warp & 3;
    const int m = 32 * qd + lane;  // TMEM lane = row of the MMA block
    // shared-memory row of this lane's weights: gate/up blocks hold gate rows
    // in lanes 0-15 and the matching up rows in lanes 16-31 of each quarter
    const int r = (MODE == kQGateUp) ? ((lane < 16) ? 16 * qd + lane : 64 + 16 * qd + lane - 16) : m;
    const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
    const int qsw = (r >> 1) & 3;  // 64-byte swizzle phase of the row
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const int s = it % kQStages, a = it % kQAStages;
        const bool got = mbar_wait(&full[s], (it / kQStages) & 1u, wt) &&
                         mbar_wait(&afree[a], ((it / kQAStages) & 1u) ^ 1u, wt);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint8_t* qt = smem + s * kQStageBytes + kQXBytes + r * 64;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // columns 64 hh .. 64 hh + 63
          const uint4 w0 = *reinterpret_cast<const uint4*>(qt + (((2 * hh) ^ qsw) << 4));
          const uint4 w1 = *reinterpret_cast<const uint4*>(qt + (((2 * hh + 1) ^ qsw) << 4));
          const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          uint32_t av[32];  // pair order: column 4c + j holds weight columns 8c + j, 8c + j + 4
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t w = wv[c];
            const uint32_t w8 = w >> 8;
            av[4 * c + 0] = q_lo_f16(w);
            av[4 * c + 1] = q_hi_f16(w);
            av[4 * c + 2] = q_lo_f16(w8);
            av[4 * c + 3] = q_hi_f16(w8);
          }
          tmem_st32(tbase + t_lane + kQACol + a * kQASlot + hh * 32, av);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aready[a]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;
    const int eh = (warp - 2 - kQDqWarps) >> 2;  // tokens 64 eh .. 64 eh + 63
    const uint32_t t_lane = static_cast<uint32_t>(32 * qd) << 16;
    // output of this lane: gate/up units pair lane i (gate) with lane i + 16
    // (up) of the same quarter
    const bool up_lane = (MODE == kQGateUp) && lane >= 16;
    const int o_off = (MODE == kQGateUp) ? 16 * qd + (lane & 15) : 32 * qd + lane;
    const uint16_t* sbase = up_lane ? p.scale1 : p.scale0;
    uint32_t gi = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      const int e = p.chunk_e[q], row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
      const int o = jt * tile_n + o_off;
      const bool valid = o < N;
      const int c0 = kQEpCols * eh;   // first token column of this warp
      const bool any = c0 < rows;     // warp-uniform
      const uint32_t* srow = reinterpret_cast<const uint32_t*>(
          sbase + ((size_t)e * N + (valid ? o : 0)) * G_all);  // G_all even: 4-byte aligned
      float y[kQEpCols];
#pragma unroll
      for (int j = 0; j < kQEpCols; ++j) y[j] = 0.f;
      // bf16 scales of groups 2i (low half) and 2i + 1 in word i, loaded four
      // words (eight groups) ahead of their use
      const int n_sw = G_all / 2;
      auto scale_word = [&](int i) -> uint32_t { return (valid && i < n_sw) ? srow[i] : 0u; };
      uint32_t sq0 = scale_word(0), sq1 = scale_word(1), sq2 = scale_word(2), sq3 = scale_word(3);
      uint32_t sw = 0;
      for (int g = 0; g < G_all; ++g, ++gi) {
        if ((g & 1) == 0) {
          sw = sq0;
          sq0 = sq1;
          sq1 = sq2;
          sq2 = sq3;
          sq3 = scale_word((g >> 1) + 4);
        }
        const float sg = __uint_as_float((g & 1) ? (sw & 0xffff0000u) : (sw << 16));
        const uint64_t sg2 = pair_f32(sg);
        const int b = gi % kQGBufs;
        if (!__all_sync(0xffffffffu, mbar_wait(&gfull[b], (gi / kQGBufs) & 1u, wt))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (any) {
          // four 16-token pieces; the buffer is released once all are read
          const uint32_t ta = tbase + t_lane + b * kQTN + c0;
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            uint32_t vc[16];
            tmem_ld16(ta + 16 * pc, vc);
            tmem_ld_wait();
            if (pc == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&gempty[b]);
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2)
              fma_f32x2(y[16 * pc + j], y[16 * pc + j + 1], sg2, __uint_as_float(vc[j]),
                        __uint_as_float(vc[j + 1]));
            if (WP) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = c0 + 16 * pc + j;
                if (valid && col < rows)
                  p.partials[((size_t)(row0 + col) * N + o) * G_all + g] =
                      static_cast<int32_t>(__uint_as_float(vc[j]));
              }
            }
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&gempty[b]);
        }
      }
      if (!ok || !any) continue;
      if (MODE == kQGateUp) {
        // lanes i and i + 16 hold G and U of output o for the warp's 64
        // tokens; the gate lane finishes tokens 0-31, the up lane 32-63
        uint16_t* hcol = static_cast<uint16_t*>(p.out) + pair_pos(o);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float mine = up_lane ? y[j] : y[32 + j];
          const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
          const int col = c0 + (up_lane ? 32 + j : j);
          if (!valid || col >= rows) continue;
          const float xs = p.x_scale[row0 + col];
          const float G = (up_lane ? other : y[j]) * xs;
          const float U = (up_lane ? y[32 + j] : other) * xs;
          hcol[(size_t)(row0 + col) * N] = f32_to_bf16_bits(silu_mul(G, U));
        }
      } else if (valid) {
#pragma unroll
        for (int j = 0; j < kQEpCols; ++j) {
          const int col = c0 + j;
          if (col >= rows) break;
          const float v = y[j] * p.x_scale[row0 + col];
          const size_t idx = (size_t)(row0 + col) * N + o;
          if (MODE == kQDown)
            static_cast<uint16_t*>(p.out)[idx] = f32_to_bf16_bits(v);
          else
            static_cast<float*>(p.out)[idx] = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kQCols);
  }
}

static bool q8_act_map(CUtensorMap* m, const uint16_t* x16, int rows, int K) {
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(kQXK), static_cast<uint32_t>(kQTN)};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

static bool q8_packed_map(CUtensorMap* m, const int32_t* w, int E, int N, int K, int rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K / 8) * 4,
                               static_cast<uint64_t>(N) * (K / 8) * 4};
  const uint32_t box[3] = {static_cast<uint32_t>(kQBK / 8), static_cast<uint32_t>(rows), 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, w, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int MODE, bool WP, bool STALL = false>
static int launch_q8(const TxMaps& maps, const TxParams& p, cudaStream_t s) {
  auto kern = ffn_tc_q8_kernel<MODE, WP, STALL>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem));
  kern<<<num_sms(), kQThreads, kQSmem, s>>>(maps, p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_tc_q8_gateup(const uint16_t* x16, const float* x_scale, int rows_max, int E, int D,
                        int I, const int32_t* gate_packed, const uint16_t* gate_scale,
                        const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                        const int32_t* chunk_e, const int32_t* chunk_row0,
                        const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                        cudaStream_t s) {
  TxMaps maps{};
  if (!q8_act_map(&maps.a, x16, rows_max, D) ||
      !q8_packed_map(&maps.q0, gate_packed, E, I, D, kQM / 2) ||
      !q8_packed_map(&maps.q1, up_packed, E, I, D, kQM / 2))
    return MOE_ERR_CUDA;
  TxParams p{};
  p.scale0 = gate_scale;
  p.scale1 = up_scale;
  p.x_scale = x_scale;
  p.out = h;
  p.chunk_e = chunk_e;
  p.chunk_row0 = chunk_row0;
  p.chunk_rows = chunk_rows;
  p.n_chunks = n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = D;
  p.N = I;
  return launch_q8<kQGateUp, false>(maps, p, s);
}

int launch_tc_q8_down(const uint16_t* h16, const float* h_scale, int rows_max, int E, int D, int I,
                      const int32_t* down_packed, const uint16_t* down_scale, void* y, bool y_f32,
                      const int32_t* chunk_e, const int32_t* chunk_row0,
                      const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                      cudaStream_t s, int32_t* partials) {
  TxMaps maps{};
  if (!q8_act_map(&maps.a, h16, rows_max, I) ||
      !q8_packed_map(&maps.q0, down_packed, E, D, I, kQM))
    return MOE_ERR_CUDA;
  maps.q1 = maps.q0;
  TxParams p{};
  p.scale0 = down_scale;
  p.scale1 = down_scale;
  p.x_scale = h_scale;
  p.out = y;
  p.partials = partials;
  p.chunk_e = chunk_e;
  p.chunk_row0 = chunk_row0;
  p.chunk_rows = chunk_rows;
  p.n_chunks = n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = I;
  p.N = D;
  if (partials) return launch_q8<kQLinear, true>(maps, p, s);
  return y_f32 ? launch_q8<kQLinear, false>(maps, p, s) : launch_q8<kQDown, false>(maps, p, s);
}

int launch_tc_q8_linear_stalled(const uint16_t* x16, const float* x_scale, int rows_max, int E,
                                int N, int K, const int32_t* w_packed, const uint16_t* w_scale,
                                float* y, const int32_t* chunk_e, const int32_t* chunk_row0,
                                const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                                long long wait_ns, int stall_at, cudaStream_t s) {
  TxMaps maps{};
  if (!q8_act_map(&maps.a, x16, rows_max, K) || !q8_packed_map(&maps.q0, w_packed, E, N, K, kQM))
    return MOE_ERR_CUDA;
  maps.q1 = maps.q0;
  TxParams p{};
  p.scale0 = w_scale;
  p.scale1 = w_scale;
  p.x_scale = x_scale;
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
  return launch_q8<kQLinear, false, true>(maps, p, s);
}

}  // namespace moe
