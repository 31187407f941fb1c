// Grouped PackedInt4Linear kernels over expert-sorted rows: the gated expert
// MLP down(SiLU(gate(x)) * up(x)) (Kimi exact-generator adaptation page,
// "The proposed substitution", "The preserved forward form", "Sources &
// provenance"; Kimi K2.5 donor-reference equation "SwiGLU-style gated
// feed-forward projection").
//
// Design (one persistent CTA per SM):
//   * a producer warp streams, per K step of 256 columns, a 256-row tile of
//     packed int4 weights with one 3-D TMA copy (128-byte swizzle), the
//     matching bf16 group scales with 4-byte cp.async, and the rows of the
//     current token chunk (<= 32 expert-sorted rows) with 1-D bulk copies,
//     into a 4-stage shared-memory ring guarded by mbarriers;
//   * eight consumer warps each own 32 weight rows.  One ldmatrix gives a
//     lane its packed words; each word becomes four bf16x2 registers holding
//     136 + q exactly (nibble | 0x4300 magic), the A operand of m16n8k16
//     tensor-core MMAs against up to 2 blocks of 8 token rows.  The constant
//     136 is removed through the accumulator: each chain starts from the MMA
//     of a constant -136 tile with the same activations, i.e. -136 * (sum of
//     the group's activations).  The 32-column group's fp32 partial is then
//     multiplied by its bf16 scale and accumulated in fp32, so the
//     dequantised weight q * scale is never rounded;
//   * the gate/up variant holds gate and up rows of the same outputs in one
//     warp and writes h = SiLU(G) * U (bf16); the down variant writes y.
// act_bits 8: the int8 activations become exact bf16 integers, the group
// partials are exact integers (|P| <= 32*8*127 < 2^24) and the row scale is
// applied in the epilogue.
#include <math.h>

#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"

namespace moe {

constexpr int kFsKc = 256;                 // K columns per stage
constexpr int kFsGroups = kFsKc / kGroup;  // 8 scale groups per stage
constexpr int kFsMc = 16;                  // token rows per chunk
constexpr int kFsTb = kFsMc / 8;           // token blocks of 8 (MMA N)
constexpr int kFsCWarps = 8;               // consumer warps
constexpr int kFsThreads = (kFsCWarps + 1) * 32;
constexpr int kFsRows = 256;               // weight rows per stage tile
constexpr int kFsStages = 5;
constexpr int kFsWBytes = kFsRows * 128;   // 32 KiB of packed int4 per stage
constexpr int kFsSBytes = kFsRows * 16;    // 8 bf16 scales per row per stage
constexpr int kFsXStride16 = kFsKc * 2 + 64;  // bf16 row stride in shared memory
constexpr int kFsXStride8 = kFsKc + 32;       // int8 row stride in shared memory
constexpr int kFsXBytes = kFsMc * kFsXStride16;
constexpr int kFsStageBytes = kFsWBytes + kFsSBytes + kFsXBytes;  // 46080 = 45 KiB
constexpr int kFsSmemBytes = kFsStages * kFsStageBytes + 1024 + 128;
static_assert(kFsStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");

enum FsMode { kGateUp = 0, kDown = 1, kLinear = 2 };

struct FsParams {
  const void* x;          // bf16 or int8 rows [rows_max, K]
  const float* x_scale;   // act_bits 8 row scales
  const uint16_t* scale0; // bf16 [E, N, K/32] (gate, or the single matrix)
  const uint16_t* scale1; // bf16 [E, N, K/32] (up)
  void* out;              // bf16 h / bf16 y / fp32 [rows_max, N]
  const int32_t* chunk_e;
  const int32_t* chunk_row0;
  const int32_t* chunk_rows;
  const int32_t* n_chunks;
  int* status;
  long long wait_ns;
  int K;
  int N;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void ldsm_x4(const void* addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(addr)));
}

// Eight two's-complement nibbles n -> four bf16x2 holding 128 + (n ^ 8), i.e.
// 136 + value, exactly: out[i] = (nibble i, nibble i+4), low half = nibble i.
// The constant 136 is removed through the MMA accumulator (see kNeg136).
__device__ __forceinline__ void dequant_magic(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = ((w >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
}

// bf16x2 (-136, -136): A operand of the MMA that forms -136 * (sum of the
// group's activations), the start value of every weight MMA chain.
constexpr uint32_t kNeg136 = 0xC308C308u;

__device__ __forceinline__ uint32_t i8pair_bf16x2(uint32_t lo_byte_word, int lo_shift,
                                                  uint32_t hi_byte_word, int hi_shift) {
  const float lo = static_cast<float>(static_cast<int8_t>((lo_byte_word >> lo_shift) & 0xffu));
  const float hi = static_cast<float>(static_cast<int8_t>((hi_byte_word >> hi_shift) & 0xffu));
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// B fragments (8 tokens x 32 columns of one group) for the two K=16 halves.
// Column permutation shared with the A side: MMA half j, logical k = 2t, 2t+1
// <-> group columns 8t+2j, 8t+2j+4; logical 2t+8, 2t+9 <-> 8t+2j+1, 8t+2j+5.
template <bool Q8>
__device__ __forceinline__ void load_b_frag(const uint8_t* xrow, int G, int t, uint32_t (&b)[4]) {
  if (!Q8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xrow + G * 64 + t * 16);
    b[0] = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
    b[1] = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
    b[2] = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
    b[3] = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(xrow + G * 32 + t * 8);
    b[0] = i8pair_bf16x2(v.x, 0, v.y, 0);    // (x0, x4)
    b[1] = i8pair_bf16x2(v.x, 8, v.y, 8);    // (x1, x5)
    b[2] = i8pair_bf16x2(v.x, 16, v.y, 16);  // (x2, x6)
    b[3] = i8pair_bf16x2(v.x, 24, v.y, 24);  // (x3, x7)
  }
}

// Per-thread constants of a consumer warp.
struct Lane {
  int g, t;            // MMA group id (row / token) and thread in group
  int li;              // row of this lane's 8x8 ldmatrix tile (swizzle phase)
  uint32_t lrow_off;   // byte offset of that row in a stage's weight tile
  int rlo[2];          // tile row of each m16 block's upper half (scales)
};

// One K stage: up to 8 groups of 32 columns for this warp's two m16 blocks
// and NTB blocks of 8 tokens.  FULL: all 8 groups present (no tail checks).
template <bool Q8, int NTB, bool FULL>
__device__ __forceinline__ void stage_compute(const uint8_t* W, const uint8_t* S, const uint8_t* X,
                                              int ng, const Lane& L, float (&acc)[2][NTB][4]) {
  constexpr int xstride = Q8 ? kFsXStride8 : kFsXStride16;
  uint4 sc[2][2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    sc[b][0] = *reinterpret_cast<const uint4*>(S + L.rlo[b] * 16);
    sc[b][1] = *reinterpret_cast<const uint4*>(S + (L.rlo[b] + 8) * 16);
  }
  const uint32_t neg[4] = {kNeg136, kNeg136, kNeg136, kNeg136};
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int G = 0; G < kFsGroups; ++G) {
    if (!FULL && G >= ng) break;
    uint32_t bfr[NTB][4];
    float corr[NTB][4];
#pragma unroll
    for (int tb = 0; tb < NTB; ++tb) {
      load_b_frag<Q8>(X + (tb * 8 + L.g) * xstride, G, L.t, bfr[tb]);
      mma_bf16_16816(corr[tb], neg, bfr[tb][0], bfr[tb][1], zero);
      mma_bf16_16816(corr[tb], neg, bfr[tb][2], bfr[tb][3], corr[tb]);
    }
    uint32_t wr[4];  // words of (block 0 row g, row g+8, block 1 row g, row g+8)
    ldsm_x4(W + L.lrow_off + ((G ^ L.li) << 4), wr);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t P[4], Q[4];
      dequant_magic(wr[2 * b], P);
      dequant_magic(wr[2 * b + 1], Q);
      const uint32_t a0[4] = {P[0], Q[0], P[1], Q[1]};
      const uint32_t a1[4] = {P[2], Q[2], P[3], Q[3]};
      const uint32_t slo_w = (&sc[b][0].x)[G >> 1];
      const uint32_t shi_w = (&sc[b][1].x)[G >> 1];
      const float s_lo = __uint_as_float((G & 1) ? (slo_w & 0xffff0000u) : (slo_w << 16));
      const float s_hi = __uint_as_float((G & 1) ? (shi_w & 0xffff0000u) : (shi_w << 16));
#pragma unroll
      for (int tb = 0; tb < NTB; ++tb) {
        float c[4];
        mma_bf16_16816(c, a0, bfr[tb][0], bfr[tb][1], corr[tb]);
        mma_bf16_16816(c, a1, bfr[tb][2], bfr[tb][3], c);
        acc[b][tb][0] = fmaf(s_lo, c[0], acc[b][tb][0]);
        acc[b][tb][1] = fmaf(s_lo, c[1], acc[b][tb][1]);
        acc[b][tb][2] = fmaf(s_hi, c[2], acc[b][tb][2]);
        acc[b][tb][3] = fmaf(s_hi, c[3], acc[b][tb][3]);
      }
    }
  }
}

// All K stages of one unit (expert chunk x row tile) for NTB token blocks,
// then the epilogue.  Returns false when a wait gave up.
template <int MODE, bool Q8, int NTB>
__device__ __forceinline__ bool consume_unit(uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             uint32_t& it, int ksteps, int row0, int rows, int n0,
                                             int cw, int lane, const Lane& L, const FsParams& p) {
  const int K = p.K, N = p.N;
  float acc[2][NTB][4];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int tb = 0; tb < NTB; ++tb)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[b][tb][c] = 0.f;

  for (int ks = 0; ks < ksteps; ++ks, ++it) {
    const int s = it % kFsStages;
    const uint32_t ph = (it / kFsStages) & 1u;
    if (!mbar_wait(&full[s], ph, p.wait_ns, p.status)) return false;
    const uint8_t* W = smem + s * kFsStageBytes;
    const uint8_t* S = W + kFsWBytes;
    const uint8_t* X = S + kFsSBytes;
    const int ng = min(kFsGroups, (K - ks * kFsKc) / kGroup);
    if (ng == kFsGroups)
      stage_compute<Q8, NTB, true>(W, S, X, ng, L, acc);
    else
      stage_compute<Q8, NTB, false>(W, S, X, ng, L, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  const int g = L.g, t = L.t;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = tb * 8 + 2 * t + (c & 1);
      if (tok >= rows) continue;
      const int row = row0 + tok;
      const float xs = Q8 ? p.x_scale[row] : 1.0f;
      if (MODE == kGateUp) {
        const int n = n0 + 16 * cw + g + ((c & 2) ? 8 : 0);
        if (n >= N) continue;
        const float G = acc[0][tb][c] * xs;
        const float U = acc[1][tb][c] * xs;
        const float h = G / (1.0f + expf(-G)) * U;
        static_cast<uint16_t*>(p.out)[(size_t)row * N + n] = f32_to_bf16_bits(h);
      } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int n = n0 + 32 * cw + 16 * b + g + ((c & 2) ? 8 : 0);
          if (n >= N) continue;
          const float y = acc[b][tb][c] * xs;
          if (MODE == kDown)
            static_cast<uint16_t*>(p.out)[(size_t)row * N + n] = f32_to_bf16_bits(y);
          else
            static_cast<float*>(p.out)[(size_t)row * N + n] = y;
        }
      }
    }
  }
  return true;
}

template <int MODE, bool Q8>
__global__ void __launch_bounds__(kFsThreads, 1)
    ffn_stream_kernel(const __grid_constant__ CUtensorMap wmap0,
                      const __grid_constant__ CUtensorMap wmap1, const FsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFsStages * kFsStageBytes);
  uint64_t* empty = full + kFsStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFsStages; ++s) {
      mbar_init(&full[s], 1 + 32);     // producer arrive.expect_tx + 32 cp.async arrivals
      mbar_init(&empty[s], kFsCWarps); // one arrival per consumer warp
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  const int K = p.K, N = p.N;
  const int tile_n = (MODE == kGateUp) ? kFsRows / 2 : kFsRows;
  const int n_tiles = (N + tile_n - 1) / tile_n;
  const int units = (*p.n_chunks) * n_tiles;
  const int ksteps = (K + kFsKc - 1) / kFsKc;
  const int G_all = K / kGroup;
  constexpr int elem = Q8 ? 1 : 2;
  constexpr int xstride = Q8 ? kFsXStride8 : kFsXStride16;

  if (warp == kFsCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&wmap0);
      if (MODE == kGateUp) prefetch_tensor_map(&wmap1);
    }
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      const int e = p.chunk_e[q], row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
      const int n0 = jt * tile_n;
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const int s = it % kFsStages;
        const uint32_t ph = (it / kFsStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, p.wait_ns, p.status)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * kFsStageBytes;
        const int k0 = ks * kFsKc;
        const int ng = min(kFsGroups, (K - k0) / kGroup);
        const uint32_t xrow_bytes = static_cast<uint32_t>(ng * kGroup * elem);
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], kFsWBytes + static_cast<uint32_t>(rows) * xrow_bytes);
          if (MODE == kGateUp) {
            tma_g2s_3d(st, &wmap0, &full[s], k0 / 8, n0, e);
            tma_g2s_3d(st + kFsWBytes / 2, &wmap1, &full[s], k0 / 8, n0, e);
          } else {
            tma_g2s_3d(st, &wmap0, &full[s], k0 / 8, n0, e);
          }
        }
        __syncwarp();
        if (lane < rows) {
          const uint8_t* src = static_cast<const uint8_t*>(p.x) +
                               ((size_t)(row0 + lane) * K + k0) * elem;
          bulk_g2s(st + kFsWBytes + kFsSBytes + lane * xstride, src, xrow_bytes, &full[s]);
        }
        // scales: row r of the tile, group pair pr (4 bytes)
        uint8_t* sdst = st + kFsWBytes;
        const int g0 = k0 / kGroup;
#pragma unroll 4
        for (int i = 0; i < kFsRows * 4 / 32; ++i) {
          const int c = lane + 32 * i;
          const int r = c >> 2, pr = c & 3;
          if (2 * pr >= ng) continue;
          int n;
          const uint16_t* sbase;
          if (MODE == kGateUp) {
            n = n0 + (r & (kFsRows / 2 - 1));
            sbase = (r < kFsRows / 2) ? p.scale0 : p.scale1;
          } else {
            n = n0 + r;
            sbase = p.scale0;
          }
          if (n >= N) continue;
          cp_async_4(sdst + r * 16 + pr * 4, sbase + ((size_t)e * N + n) * G_all + g0 + 2 * pr);
        }
        cp_async_arrive_noinc(&full[s]);
      }
    }
    if (!ok) {
      // let copies already issued land before the CTA exits (bounded)
      const uint32_t first = it >= kFsStages ? it - kFsStages : 0;
      for (uint32_t i = first; i < it; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&full[i % kFsStages], (i / kFsStages) & 1u)) {
          if (static_cast<int64_t>(global_timer_ns() - t0) > 100000000LL) break;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  Lane L;
  L.g = lane >> 2;
  L.t = lane & 3;
  L.li = lane & 7;
  {
    // ldmatrix: lanes 8m..8m+7 address rows of matrix m = (block m/2, half m%2)
    const int m = lane >> 3;
    const int b = m >> 1, h = m & 1;
    const int base = (MODE == kGateUp) ? b * (kFsRows / 2) + 16 * warp : 32 * warp + 16 * b;
    L.lrow_off = static_cast<uint32_t>((base + 8 * h + L.li) * 128);
    if (MODE == kGateUp) {
      L.rlo[0] = 16 * warp + L.g;                 // gate rows
      L.rlo[1] = kFsRows / 2 + 16 * warp + L.g;   // up rows
    } else {
      L.rlo[0] = 32 * warp + L.g;
      L.rlo[1] = 32 * warp + 16 + L.g;
    }
  }
  uint32_t it = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int q = u / n_tiles, jt = u - q * n_tiles;
    const int row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
    const int n0 = jt * tile_n;
    const int ntb = (rows + 7) >> 3;
    bool ok;
    static_assert(kFsTb == 2, "token-block dispatch below covers 1 or 2 blocks");
    if (ntb == 1)
      ok = consume_unit<MODE, Q8, 1>(smem, full, empty, it, ksteps, row0, rows, n0, warp, lane, L, p);
    else
      ok = consume_unit<MODE, Q8, 2>(smem, full, empty, it, ksteps, row0, rows, n0, warp, lane, L, p);
    if (!ok) return;
  }
}

// Chunk list of the expert-sorted rows: every expert's rows cut into chunks of
// at most kFsMc rows.  One CTA of 1024 threads.  Offsets that are not
// non-decreasing or exceed rows_max record MOE_ERR_INVALID and give no chunk.
__global__ void __launch_bounds__(1024) ffn_schedule_kernel(const int32_t* __restrict__ offsets,
                                                            int E, int rows_max, int max_chunks,
                                                            int32_t* __restrict__ chunk_e,
                                                            int32_t* __restrict__ chunk_row0,
                                                            int32_t* __restrict__ chunk_rows,
                                                            int32_t* __restrict__ n_chunks,
                                                            int* status) {
  __shared__ int32_t nch[kMaxExperts];
  __shared__ int32_t total;
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int a = offsets[e], b = offsets[e + 1];
    const int cnt = b - a;
    if (a < 0 || cnt < 0 || b > rows_max) bad = 1;
    nch[e] = cnt > 0 ? (cnt + kFsMc - 1) / kFsMc : 0;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      record_status(status, MOE_ERR_INVALID);
      *n_chunks = 0;
    }
    return;
  }
  // exclusive scan of nch (n <= 2048) with 1024 threads, two entries each
  {
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, ln = tid & 31, wp = tid >> 5;
    const int i0 = 2 * tid;
    const int a = i0 < E ? nch[i0] : 0;
    const int b = i0 + 1 < E ? nch[i0 + 1] : 0;
    int incl = a + b;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (ln >= o) incl += y;
    }
    if (ln == 31) warp_tot[wp] = incl;
    __syncthreads();
    if (wp == 0) {
      const int w = warp_tot[ln];
      int wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (ln >= o) wi += y;
      }
      warp_tot[ln] = wi - w;
      if (ln == 31) total = wi;
    }
    __syncthreads();
    const int excl = incl - (a + b) + warp_tot[wp];
    __syncthreads();
    if (i0 < E) nch[i0] = excl;
    if (i0 + 1 < E) nch[i0 + 1] = excl + a;
    __syncthreads();
  }
  if (total > max_chunks) {
    if (threadIdx.x == 0) {
      record_status(status, MOE_ERR_INVALID);
      *n_chunks = 0;
    }
    return;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int a = offsets[e], cnt = offsets[e + 1] - a;
    const int base = nch[e];
    for (int i = 0; i * kFsMc < cnt; ++i) {
      chunk_e[base + i] = e;
      chunk_row0[base + i] = a + i * kFsMc;
      chunk_rows[base + i] = min(kFsMc, cnt - i * kFsMc);
    }
  }
  if (threadIdx.x == 0) *n_chunks = total;
}

static int max_chunks_for(int E, int rows_max) { return (rows_max + kFsMc - 1) / kFsMc + E; }

struct Schedule {
  int32_t* chunk_e;
  int32_t* chunk_row0;
  int32_t* chunk_rows;
  int32_t* n_chunks;
  size_t bytes;
};

static Schedule carve_schedule(void* ws, int E, int rows_max) {
  const size_t mc = static_cast<size_t>(max_chunks_for(E, rows_max));
  Schedule s;
  char* b = static_cast<char*>(ws);
  const size_t arr = align_up(mc * sizeof(int32_t), 256);
  s.chunk_e = reinterpret_cast<int32_t*>(b);
  s.chunk_row0 = reinterpret_cast<int32_t*>(b + arr);
  s.chunk_rows = reinterpret_cast<int32_t*>(b + 2 * arr);
  s.n_chunks = reinterpret_cast<int32_t*>(b + 3 * arr);
  s.bytes = 3 * arr + 256;
  return s;
}

static size_t schedule_bytes(int E, int rows_max) {
  const size_t mc = static_cast<size_t>(max_chunks_for(E, rows_max));
  return 3 * align_up(mc * sizeof(int32_t), 256) + 256;
}

// Tensor map of a packed weight [E, N, K/8] int32 with a box of `rows` rows x
// 32 words (128 bytes, 128-byte swizzle).
static bool weight_map(CUtensorMap* m, const int32_t* w, int E, int N, int K, int rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K / 8) * 4,
                               static_cast<uint64_t>(N) * (K / 8) * 4};
  const uint32_t box[3] = {32, static_cast<uint32_t>(rows), 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, w, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE, bool Q8>
static int launch_stream(const CUtensorMap& m0, const CUtensorMap& m1, const FsParams& p,
                         cudaStream_t s) {
  auto kern = ffn_stream_kernel<MODE, Q8>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kFsSmemBytes));
  kern<<<num_sms(), kFsThreads, kFsSmemBytes, s>>>(m0, m1, p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static int run_stream(int mode, bool q8, const CUtensorMap& m0, const CUtensorMap& m1,
                      const FsParams& p, cudaStream_t s) {
  if (mode == kGateUp) return q8 ? launch_stream<kGateUp, true>(m0, m1, p, s)
                                 : launch_stream<kGateUp, false>(m0, m1, p, s);
  if (mode == kDown) return q8 ? launch_stream<kDown, true>(m0, m1, p, s)
                               : launch_stream<kDown, false>(m0, m1, p, s);
  return q8 ? launch_stream<kLinear, true>(m0, m1, p, s) : launch_stream<kLinear, false>(m0, m1, p, s);
}

static int check_width(int v) { return (v > 0 && v % 64 == 0) ? MOE_OK : MOE_ERR_UNSUPPORTED; }

}  // namespace moe

using namespace moe;

extern "C" size_t moe_expert_ffn_workspace_size(int E, int D, int I, int rows_max, int act_bits) {
  if (E <= 0 || D <= 0 || I <= 0 || rows_max < 0) return 256;
  size_t b = schedule_bytes(E, rows_max);
  b += align_up((size_t)rows_max * I * sizeof(uint16_t), 256);  // h (bf16)
  if (act_bits == 8) {
    b += align_up((size_t)rows_max * I, 256);                // h as int8
    b += align_up((size_t)rows_max * sizeof(float), 256);    // its row scales
  }
  return b;
}

int moe::launch_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets,
                           int E, int D, int I, int rows_max, const int32_t* gate_packed,
                           const uint16_t* gate_scale, const int32_t* up_packed,
                           const uint16_t* up_scale, const int32_t* down_packed,
                           const uint16_t* down_scale, int act_bits, void* y, bool y_f32, void* ws,
                           cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  Schedule sch = carve_schedule(ws, E, rows_max);
  char* b = static_cast<char*>(ws) + sch.bytes;
  uint16_t* h = reinterpret_cast<uint16_t*>(b);
  b += align_up((size_t)rows_max * I * sizeof(uint16_t), 256);
  int8_t* hq = nullptr;
  float* hs = nullptr;
  if (act_bits == 8) {
    hq = reinterpret_cast<int8_t*>(b);
    b += align_up((size_t)rows_max * I, 256);
    hs = reinterpret_cast<float*>(b);
  }

  ffn_schedule_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, max_chunks_for(E, rows_max),
                                         sch.chunk_e, sch.chunk_row0, sch.chunk_rows, sch.n_chunks,
                                         status);
  MOE_LAUNCH_CHECK();

  CUtensorMap mg, mu, md;
  if (!weight_map(&mg, gate_packed, E, I, D, kFsRows / 2) ||
      !weight_map(&mu, up_packed, E, I, D, kFsRows / 2) ||
      !weight_map(&md, down_packed, E, D, I, kFsRows))
    return MOE_ERR_CUDA;

  const bool q8 = act_bits == 8;
  FsParams p{};
  p.x = x_sorted;
  p.x_scale = x_scale;
  p.scale0 = gate_scale;
  p.scale1 = up_scale;
  p.out = h;
  p.chunk_e = sch.chunk_e;
  p.chunk_row0 = sch.chunk_row0;
  p.chunk_rows = sch.chunk_rows;
  p.n_chunks = sch.n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = D;
  p.N = I;
  int rc = run_stream(kGateUp, q8, mg, mu, p, s);
  if (rc) return rc;

  FsParams pd = p;
  pd.K = I;
  pd.N = D;
  pd.scale0 = down_scale;
  pd.scale1 = nullptr;
  pd.out = y;
  if (q8) {
    rc = launch_quantize_rows(h, rows_max, I, offsets + E, hq, hs, s);
    if (rc) return rc;
    pd.x = hq;
    pd.x_scale = hs;
  } else {
    pd.x = h;
  }
  return run_stream(y_f32 ? kLinear : kDown, q8, md, md, pd, s);
}

extern "C" int moe_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets,
                              int E, int D, int I, int rows_max, const int32_t* gate_packed,
                              const uint16_t* gate_scale, const int32_t* up_packed,
                              const uint16_t* up_scale, const int32_t* down_packed,
                              const uint16_t* down_scale, int act_bits, uint16_t* y_sorted,
                              void* ws, size_t ws_bytes, void* stream) {
  if (E <= 0 || rows_max < 0) return MOE_ERR_INVALID;
  if (check_width(D) || check_width(I) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x_sorted || !offsets || !gate_packed || !gate_scale || !up_packed || !up_scale ||
      !down_packed || !down_scale || !y_sorted || !ws)
    return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x_sorted, 16) || !aligned(gate_packed, 16) || !aligned(up_packed, 16) ||
      !aligned(down_packed, 16) || !aligned(gate_scale, 4) || !aligned(up_scale, 4) ||
      !aligned(down_scale, 4))
    return MOE_ERR_INVALID;
  if (ws_bytes < moe_expert_ffn_workspace_size(E, D, I, rows_max, act_bits))
    return MOE_ERR_WORKSPACE;
  return launch_expert_ffn(x_sorted, x_scale, offsets, E, D, I, rows_max, gate_packed, gate_scale,
                           up_packed, up_scale, down_packed, down_scale, act_bits, y_sorted, false,
                           ws, static_cast<cudaStream_t>(stream));
}

extern "C" size_t moe_int4_linear_workspace_size(int E, int rows_max) {
  if (E <= 0 || rows_max < 0) return 256;
  return schedule_bytes(E, rows_max);
}

extern "C" int moe_int4_linear(const void* x, const float* x_scale, const int32_t* offsets, int E,
                               int K, int N, int rows_max, const int32_t* w_packed,
                               const uint16_t* w_scale, int act_bits, float* out, void* ws,
                               size_t ws_bytes, void* stream) {
  if (E <= 0 || rows_max < 0 || N <= 0) return MOE_ERR_INVALID;
  if (check_width(K) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x || !offsets || !w_packed || !w_scale || !out || !ws) return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scale, 4)) return MOE_ERR_INVALID;
  if (ws_bytes < moe_int4_linear_workspace_size(E, rows_max)) return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Schedule sch = carve_schedule(ws, E, rows_max);
  ffn_schedule_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, max_chunks_for(E, rows_max),
                                         sch.chunk_e, sch.chunk_row0, sch.chunk_rows, sch.n_chunks,
                                         status);
  MOE_LAUNCH_CHECK();
  CUtensorMap m;
  if (!weight_map(&m, w_packed, E, N, K, kFsRows)) return MOE_ERR_CUDA;
  FsParams p{};
  p.x = x;
  p.x_scale = x_scale;
  p.scale0 = w_scale;
  p.out = out;
  p.chunk_e = sch.chunk_e;
  p.chunk_row0 = sch.chunk_row0;
  p.chunk_rows = sch.chunk_rows;
  p.n_chunks = sch.n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = K;
  p.N = N;
  return run_stream(kLinear, act_bits == 8, m, m, p, s);
}
