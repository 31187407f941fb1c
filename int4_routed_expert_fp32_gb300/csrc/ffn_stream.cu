// Grouped PackedInt4Linear kernels over expert-sorted rows: the gated expert
// MLP down(SiLU(gate(x)) * up(x)) (Kimi exact-generator adaptation page,
// "The proposed substitution", "The preserved forward form", "Sources &
// provenance"; Kimi K2.5 donor-reference equation "SwiGLU-style gated
// feed-forward projection").
//
// Design (one persistent CTA per SM):
//   * a producer warp streams, per K step of 256 columns, a 256-row tile of
//     packed int4 weights and the matching bf16 group scales with 3-D TMA
//     copies (128-byte swizzle for the weights), and the rows of the current
//     token chunk (<= 16 expert-sorted rows) with 1-D bulk copies, into a
//     4-stage shared-memory ring guarded by mbarriers.  When the scale rows
//     are not 16-byte aligned (K not a multiple of 256) the scales go through
//     4-byte cp.async instead;
//   * the activation rows arrive in "pair order": fp16 (int8 with act_bits 8)
//     with each block of 8 columns stored as c0 c4 c1 c5 c2 c6 c3 c7, the
//     order in which one packed int32 word pairs its nibbles.  A lane's
//     16-byte load is then its MMA B fragments as they are;
//   * sixteen consumer warps each own one 16-row block.  One ldmatrix gives a
//     lane its packed words of two groups.  Each word becomes four fp16x2
//     registers with one shift and four masks: the nibble pairs (0,4) and
//     (2,6) land in the low mantissa bits of 1024.0 and hold 1032 + q, the
//     pairs (1,5) and (3,7) in bits 4-7 of 64.0 and hold 72 + q, all
//     exactly.  They are the A operands of one chain of two m16n8k16 fp16
//     MMAs per 32-column group against up to 2 blocks of 8 token rows.  The
//     constants are removed through the accumulator: the chain starts from
//     -(1032 S_lo + 72 S_hi), S the sums of the token's activations that the
//     two kinds of values multiply, computed once per stage for the whole CTA
//     by a start-value warp.  The group's partial is then multiplied by its
//     bf16 scale and accumulated in fp32, so the dequantised weight q * scale
//     is never rounded;
//   * in the gate/up variant warps 0-7 hold gate rows and warps 8-15 the up
//     rows of the same outputs; the up partials go through shared memory and
//     the gate warps write h = SiLU(G) * U in pair order (fp16; bf16 with
//     act_bits 8, for its re-quantisation).  The down variant writes y.
// act_bits 8: the int8 activations become exact fp16 integers; the chain of
// a group stays an exact integer (|partial sums| <= 32 * 1040 * 127 < 2^24),
// so the group partial is the exact integer sum, and the row scale is
// applied in the epilogue.
#include <cuda_fp16.h>
#include <math.h>

#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"
#include "ffn_tc.cuh"

namespace moe {

constexpr int kFsKc = 256;                 // K columns per stage
constexpr int kFsGroups = kFsKc / kGroup;  // 8 scale groups per stage
constexpr int kFsMc = 16;                  // token rows per chunk
constexpr int kFsTb = kFsMc / 8;           // token blocks of 8 (MMA N)
constexpr int kFsCWarps = 16;              // consumer warps, one 16-row block each
constexpr int kFsUnroll = 4;               // group pairs unrolled with one token block
constexpr int kFsThreads = (kFsCWarps + 2) * 32;  // + TMA producer + start-value warp
constexpr int kFsRows = 16 * kFsCWarps;    // weight rows per stage tile
constexpr int kFsStages = 4;
constexpr int kFsWBytes = kFsRows * 128;   // 32 KiB of packed int4 per stage
constexpr int kFsSBytes = kFsRows * 16;    // 8 bf16 scales per row per stage
constexpr int kFsXStride16 = kFsKc * 2 + 64;  // bf16 row stride in shared memory
constexpr int kFsXStride8 = kFsKc + 32;       // int8 row stride in shared memory
constexpr int kFsXBytes = kFsMc * kFsXStride16;
constexpr int kFsCBytes = kFsGroups * kFsMc * 4;  // chain start values [group][token]
constexpr int kFsStageBytes =
    (kFsWBytes + kFsSBytes + kFsXBytes + kFsCBytes + 1023) / 1024 * 1024;  // 1024-byte aligned
constexpr int kFsXchBytes = (kFsRows / 2) * kFsMc * 4;          // up partials of one unit
constexpr int kFsSmemBytes = kFsStages * kFsStageBytes + 2 * kFsXchBytes + 1024 + 256;
static_assert(kFsStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kFsTb == 2, "token-block dispatch covers 1 or 2 blocks");

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
  int tma_scales;         // 1: scales by TMA (K % 256 == 0), 0: 4-byte cp.async
  int32_t* partials;      // act_bits 8, tests only: int32 [rows_max, N, K/32] or null
  int stall_at;           // tests only (STALL instantiation): the producer stops at this stage
};

// Where a consumer thread stores the integer group partials of its MMA
// chains (tests only): token rows tok0, tok0 + 1 of each 8-token block and
// weight rows n, n + 8, K/32 groups per (row, output) pair.
struct PartialsOut {
  int32_t* base;  // partials at (row0 + 2t, n0 + 16 cw + g, group ks * 8)
  int N;          // outputs per row
  int G_all;      // groups per output
  int rows;       // rows of the chunk
  int t2;         // 2t: first token of the thread's pair in each 8-token block
  bool n_ok0, n_ok8;  // weight rows n and n + 8 exist
};

struct FsMaps {
  CUtensorMap w0, w1;     // packed weights (gate/up, or the single matrix twice)
  CUtensorMap s0, s1;     // scales (used when tma_scales)
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
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

// Eight two's-complement nibbles n_0..n_7 of one packed word -> four fp16x2:
//   out[0] = (n0, n4), out[2] = (n2, n6): in the low mantissa bits of 1024.0
//            (ulp 1): 1024 + (n ^ 8) = 1032 + q;
//   out[1] = (n1, n5), out[3] = (n3, n7): in mantissa bits 4-7 of 64.0 (ulp
//            1/16): 64 + (n ^ 8) = 72 + q.
// Low half = the lower nibble of the pair.  One shift and four mask-xor ops;
// every value is exact and carries q with weight 1.
__device__ __forceinline__ void dequant_magic(uint32_t w, uint32_t (&out)[4]) {
  const uint32_t w8 = w >> 8;
  out[0] = (w & 0x000F000Fu) ^ 0x64086408u;
  out[1] = (w & 0x00F000F0u) ^ 0x54805480u;
  out[2] = (w8 & 0x000F000Fu) ^ 0x64086408u;
  out[3] = (w8 & 0x00F000F0u) ^ 0x54805480u;
}

// Two int8 values (bytes selected by `sel` into the low byte of each half)
// -> fp16x2, exactly: 1024 + (x + 128) via the 0x6480 xor, minus 1152.
__device__ __forceinline__ uint32_t i8pair_f16x2(uint32_t w, uint32_t sel) {
  const uint32_t m = __byte_perm(w, 0u, sel) ^ 0x64806480u;
  __half2 h = *reinterpret_cast<const __half2*>(&m);
  h = __hsub2(h, __floats2half2_rn(1152.0f, 1152.0f));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// B fragments (8 tokens x 32 columns of one group) from pair-ordered rows:
// b[0] = (x0, x4), b[1] = (x1, x5), b[2] = (x2, x6), b[3] = (x3, x7) of the
// lane's 8 columns 8t..8t+7 of group G.  The low-nibble MMA takes b[0], b[2],
// the high-nibble MMA b[1], b[3].
template <bool Q8>
__device__ __forceinline__ void load_b_frag(const uint8_t* xrow, int G, int t, uint32_t (&b)[4]) {
  if (!Q8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xrow + G * 64 + t * 16);
    b[0] = v.x;
    b[1] = v.y;
    b[2] = v.z;
    b[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(xrow + G * 32 + t * 8);
    b[0] = i8pair_f16x2(v.x, 0x4140u);
    b[1] = i8pair_f16x2(v.x, 0x4342u);
    b[2] = i8pair_f16x2(v.y, 0x4140u);
    b[3] = i8pair_f16x2(v.y, 0x4342u);
  }
}

// Per-thread constants of a consumer warp.
struct Lane {
  int g, t;            // MMA group id (row / token) and thread in group
  int li;              // row of this lane's 8x8 ldmatrix tile (swizzle phase)
  int gsel;            // which of the two groups this lane's ldmatrix tile holds
  uint32_t lrow_off;   // byte offset of that row in a stage's weight tile
  int rlo;             // tile row of the block's upper half (scales)
};

// One K stage: up to 8 groups of 32 columns for this warp's 16-row block and
// NTB blocks of 8 tokens.  FULL: all 8 groups present (no tail checks).
template <bool Q8, int NTB, bool FULL, bool WP = false>
__device__ __forceinline__ void stage_compute(const uint8_t* W, const uint8_t* S, const uint8_t* X,
                                              const uint8_t* C, int ng, const Lane& L,
                                              float (&acc)[NTB][4],
                                              const PartialsOut& po = PartialsOut{}) {
  constexpr int xstride = Q8 ? kFsXStride8 : kFsXStride16;
  const uint32_t* s_lo_row = reinterpret_cast<const uint32_t*>(S + L.rlo * 16);
  const uint32_t* s_hi_row = reinterpret_cast<const uint32_t*>(S + (L.rlo + 8) * 16);
  const float2* cst = reinterpret_cast<const float2*>(C);  // [group][token pair]
  // two token blocks keep more values live: unroll less there
#pragma unroll(NTB == 1 ? kFsUnroll : 1)
  for (int G2 = 0; G2 < kFsGroups; G2 += 2) {
    if (!FULL && G2 >= ng) break;
    uint32_t wr[4];  // (row g, row g+8) words of groups G2 and G2+1
    ldsm_x4(W + L.lrow_off + (((G2 + L.gsel) ^ L.li) << 4), wr);
    const uint32_t slo_w = s_lo_row[G2 >> 1];  // bf16 scales of groups G2 (low) and G2+1
    const uint32_t shi_w = s_hi_row[G2 >> 1];
#pragma unroll
    for (int gg = 0; gg < 2; ++gg) {
      const int G = G2 + gg;
      uint32_t P[4], Q[4];
      dequant_magic(wr[2 * gg], P);      // row g
      dequant_magic(wr[2 * gg + 1], Q);  // row g + 8
      const uint32_t alo[4] = {P[0], Q[0], P[2], Q[2]};
      const uint32_t ahi[4] = {P[1], Q[1], P[3], Q[3]};
      const float s_lo = __uint_as_float(gg ? (slo_w & 0xffff0000u) : (slo_w << 16));
      const float s_hi = __uint_as_float(gg ? (shi_w & 0xffff0000u) : (shi_w << 16));
#pragma unroll
      for (int tb = 0; tb < NTB; ++tb) {
        uint32_t bfr[4];
        load_b_frag<Q8>(X + (tb * 8 + L.g) * xstride, G, L.t, bfr);
        // start value of tokens 8 tb + 2t and + 1: -(1032 S_lo + 72 S_hi)
        const float2 c2 = cst[G * (kFsMc / 2) + tb * 4 + L.t];
        float c[4] = {c2.x, c2.y, c2.x, c2.y};
        mma_f16_16816(c, alo, bfr[0], bfr[2], c);
        mma_f16_16816(c, ahi, bfr[1], bfr[3], c);
        if (WP) {
          // c holds the exact integer partials of group G: rows n, n + 8 x
          // tokens 8 tb + 2t, + 1
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tk = tb * 8 + po.t2 + (i & 1);
            if (tk < po.rows && ((i & 2) ? po.n_ok8 : po.n_ok0))
              po.base[((size_t)(tb * 8 + (i & 1)) * po.N + ((i & 2) ? 8 : 0)) * po.G_all + G] =
                  static_cast<int32_t>(c[i]);
          }
        }
        acc[tb][0] = fmaf(s_lo, c[0], acc[tb][0]);
        acc[tb][1] = fmaf(s_lo, c[1], acc[tb][1]);
        acc[tb][2] = fmaf(s_hi, c[2], acc[tb][2]);
        acc[tb][3] = fmaf(s_hi, c[3], acc[tb][3]);
      }
    }
  }
}

// Start values of the MMA chains of one stage, for the chunk's token rows:
// C[G][tok] = -(1032 * S_lo + 72 * S_hi), where S_lo sums the token's
// activations that the low-nibble values (1032 + q) of group G multiply and
// S_hi those of the high-nibble values (72 + q).  In pair order (c0 c4 c1 c5
// c2 c6 c3 c7) the low values take positions 0, 1, 4, 5 of each block of 8
// (fragments b[0], b[2]: columns 0 4 2 6) and the high values positions 2,
// 3, 6, 7.  Only the chunk's rows are summed: lane l takes the (token,
// group) pairs l, l + 32, ... of the rows x ng pairs.  With int8
// activations the sums, and the start values, are exact integers.
template <bool Q8>
__device__ __forceinline__ void stage_starts(const uint8_t* X, uint8_t* C, int ng, int rows,
                                             int lane) {
  float* out = reinterpret_cast<float*>(C);
#pragma unroll 1
  for (int idx = lane; idx < rows * ng; idx += 32) {
    const int tk = idx / ng, G = idx - tk * ng;
    float lo = 0.f, hi = 0.f;
    if (!Q8) {
      const uint4* xg = reinterpret_cast<const uint4*>(X + tk * kFsXStride16 + G * 64);
#pragma unroll
      for (int v = 0; v < 4; ++v) {  // one block of 8 per 16 bytes
        const uint4 w = xg[v];
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w.x));  // pos 0, 1
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w.y));  // pos 2, 3
        const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&w.z));  // pos 4, 5
        const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&w.w));  // pos 6, 7
        lo += (f0.x + f0.y) + (f2.x + f2.y);
        hi += (f1.x + f1.y) + (f3.x + f3.y);
      }
    } else {
      const uint2* xg = reinterpret_cast<const uint2*>(X + tk * kFsXStride8 + G * 32);
      int ilo = 0, ihi = 0;
#pragma unroll
      for (int v = 0; v < 4; ++v) {  // one block of 8 per 8 bytes
        const uint2 w = xg[v];
        const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t b = ws[j];
          ilo += static_cast<int8_t>(b & 0xffu) + static_cast<int8_t>((b >> 8) & 0xffu);
          ihi += static_cast<int8_t>((b >> 16) & 0xffu) + static_cast<int8_t>(b >> 24);
        }
      }
      lo = static_cast<float>(ilo);
      hi = static_cast<float>(ihi);
    }
    out[G * kFsMc + tk] = -(1032.0f * lo + 72.0f * hi);
  }
}

__device__ __forceinline__ void named_bar_sync_n(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void consumer_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFsCWarps * 32) : "memory");
}

// All K stages of one unit (expert chunk x row tile) for NTB token blocks,
// then the epilogue.  Returns false when a wait gave up.
template <int MODE, bool Q8, int NTB, bool WP = false>
__device__ __forceinline__ bool consume_unit(uint8_t* smem, float* xch, uint64_t* ready,
                                             uint64_t* empty, uint32_t& it, int ksteps, int row0,
                                             int rows, int n0, int cw, int lane, const Lane& L,
                                             const FsParams& p, const Waiter& wt) {
  const int K = p.K, N = p.N;
  float acc[NTB][4];
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[tb][c] = 0.f;

  bool ok = true;
  for (int ks = 0; ks < ksteps; ++ks, ++it) {
    const int s = it % kFsStages;
    const uint32_t ph = (it / kFsStages) & 1u;
    if (ok && !mbar_wait(&ready[s], ph, wt)) ok = false;
    // The stage is computed whatever the wait's outcome, so every lane runs
    // the warp-collective ldmatrix and MMAs (after a wait that gave up, on
    // data that may be stale, all inside this CTA's ring; the epilogue then
    // stores nothing).
    {
      const uint8_t* W = smem + s * kFsStageBytes;
      const uint8_t* S = W + kFsWBytes;
      const uint8_t* X = S + kFsSBytes;
      const uint8_t* C = X + kFsXBytes;
      const int ng = min(kFsGroups, (K - ks * kFsKc) / kGroup);
      if (WP) {
        const int G_all = K / kGroup;
        const int n = n0 + cw * 16 + L.g;
        PartialsOut po{p.partials + ((size_t)(row0 + 2 * L.t) * N + n) * G_all + ks * kFsGroups,
                       N, G_all, rows, 2 * L.t, n < N, n + 8 < N};
        if (ng == kFsGroups)
          stage_compute<Q8, NTB, true, true>(W, S, X, C, ng, L, acc, po);
        else
          stage_compute<Q8, NTB, false, true>(W, S, X, C, ng, L, acc, po);
      } else if (ng == kFsGroups) {
        stage_compute<Q8, NTB, true>(W, S, X, C, ng, L, acc);
      } else {
        stage_compute<Q8, NTB, false>(W, S, X, C, ng, L, acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  const int g = L.g, t = L.t;
  if (MODE == kGateUp) {
    // up warps (8..15) hand their partials to the gate warps (0..7)
    const int half = kFsCWarps / 2;
    if (cw >= half) {
#pragma unroll
      for (int tb = 0; tb < NTB; ++tb) {
        const int r = (cw - half) * 16 + g;
        const int col = tb * 8 + 2 * t;
        *reinterpret_cast<float2*>(xch + r * kFsMc + col) = make_float2(acc[tb][0], acc[tb][1]);
        *reinterpret_cast<float2*>(xch + (r + 8) * kFsMc + col) = make_float2(acc[tb][2], acc[tb][3]);
      }
    }
    consumer_bar_sync();
    if (cw >= half) return ok;
    {
#pragma unroll
    for (int tb = 0; tb < NTB; ++tb) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int tok = tb * 8 + 2 * t + (c & 1);
        const int rr = cw * 16 + g + ((c & 2) ? 8 : 0);
        const int n = n0 + rr;
        if (!ok || tok >= rows || n >= N) continue;
        const int row = row0 + tok;
        const float xs = Q8 ? p.x_scale[row] : 1.0f;
        const float G = acc[tb][c] * xs;
        const float U = xch[rr * kFsMc + tok] * xs;
        // act_bits 8: the tanh form the tensor-core exact kernel uses, so that
        // both give the same h
        const float h = Q8 ? silu_mul(G, U) : G / (1.0f + expf(-G)) * U;
        uint16_t* hrow = static_cast<uint16_t*>(p.out) + (size_t)row * N;
        if (Q8) {
          hrow[pair_pos(n)] = f32_to_bf16_bits(h);
        } else {
          if (!(fabsf(h) <= 65504.0f)) record_status(p.status, MOE_ERR_UNSUPPORTED);
          hrow[pair_pos(n)] = __half_as_ushort(__float2half_rn(h));
        }
      }
    }
    }
  } else {
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = tb * 8 + 2 * t + (c & 1);
      const int n = n0 + cw * 16 + g + ((c & 2) ? 8 : 0);
      if (!ok || tok >= rows || n >= N) continue;
      const int row = row0 + tok;
      const float xs = Q8 ? p.x_scale[row] : 1.0f;
      const float y = acc[tb][c] * xs;
      if (MODE == kDown)
        static_cast<uint16_t*>(p.out)[(size_t)row * N + n] = f32_to_bf16_bits(y);
      else
        static_cast<float*>(p.out)[(size_t)row * N + n] = y;
    }
  }
  }
  return ok;
}

// Producer side of one unit: for each K stage wait for a free slot, then
// TMA the weight (and scale) tiles and bulk-copy the chunk's activation rows.
// Returns false when a wait gave up.
template <int MODE, bool Q8, bool STALL = false>
__device__ __forceinline__ bool produce_unit(const FsMaps& maps, const FsParams& p, uint8_t* smem,
                                             uint64_t* full, uint64_t* empty, uint32_t& it,
                                             int e, int row0, int rows, int n0, int lane,
                                             const Waiter& wt) {
  constexpr int elem = Q8 ? 1 : 2;
  constexpr int xstride = Q8 ? kFsXStride8 : kFsXStride16;
  const int K = p.K, N = p.N;
  const int ksteps = (K + kFsKc - 1) / kFsKc;
  const int G_all = K / kGroup;
  const bool tma_s = p.tma_scales != 0;
  for (int ks = 0; ks < ksteps; ++ks, ++it) {
    const int s = it % kFsStages;
    const uint32_t ph = (it / kFsStages) & 1u;
    if (STALL && static_cast<int>(it) == p.stall_at) return false;  // tests only
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1u, wt))) return false;  // warp-uniform
    uint8_t* st = smem + s * kFsStageBytes;
    uint8_t* sdst = st + kFsWBytes;
    const int k0 = ks * kFsKc;
    const int ng = min(kFsGroups, (K - k0) / kGroup);
    const uint32_t xrow_bytes = static_cast<uint32_t>(ng * kGroup * elem);
    if (lane == 0) {
      mbar_arrive_expect_tx(&full[s], kFsWBytes + (tma_s ? kFsSBytes : 0) +
                                          static_cast<uint32_t>(rows) * xrow_bytes);
      if (MODE == kGateUp) {
        tma_g2s_3d(st, &maps.w0, &full[s], k0 / 8, n0, e);
        tma_g2s_3d(st + kFsWBytes / 2, &maps.w1, &full[s], k0 / 8, n0, e);
        if (tma_s) {
          tma_g2s_3d(sdst, &maps.s0, &full[s], k0 / kGroup, n0, e);
          tma_g2s_3d(sdst + kFsSBytes / 2, &maps.s1, &full[s], k0 / kGroup, n0, e);
        }
      } else {
        tma_g2s_3d(st, &maps.w0, &full[s], k0 / 8, n0, e);
        if (tma_s) tma_g2s_3d(sdst, &maps.s0, &full[s], k0 / kGroup, n0, e);
      }
    }
    __syncwarp();
    if (lane < rows) {
      const uint8_t* src = static_cast<const uint8_t*>(p.x) + ((size_t)(row0 + lane) * K + k0) * elem;
      bulk_g2s(st + kFsWBytes + kFsSBytes + lane * xstride, src, xrow_bytes, &full[s]);
    }
    if (!tma_s) {
      // scales: row r of the tile, group pair pr (4 bytes)
      const int g0 = k0 / kGroup;
#pragma unroll 4
      for (int i = 0; i < kFsRows * 4 / 32; ++i) {
        const int c = lane + 32 * i;
        const int r = c >> 2, pr = c & 3;
        if (2 * pr >= ng) continue;
        int n;
        const uint16_t* sbase;
        if (MODE == kGateUp) {
          const bool up = r >= kFsRows / 2;
          n = n0 + (up ? r - kFsRows / 2 : r);
          sbase = up ? p.scale1 : p.scale0;
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
  return true;
}

// Start-value side of one unit (see stage_starts).  Returns false when a wait
// gave up.
template <bool Q8>
__device__ __forceinline__ bool starts_unit(const FsParams& p, uint8_t* smem, uint64_t* full,
                                            uint64_t* empty, uint64_t* ready, uint32_t& it,
                                            int rows, int lane, const Waiter& wt) {
  const int K = p.K;
  const int ksteps = (K + kFsKc - 1) / kFsKc;
  for (int ks = 0; ks < ksteps; ++ks, ++it) {
    const int s = it % kFsStages;
    const uint32_t ph = (it / kFsStages) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, wt))) return false;  // warp-uniform
    uint8_t* st = smem + s * kFsStageBytes;
    const int ng = min(kFsGroups, (K - ks * kFsKc) / kGroup);
    stage_starts<Q8>(st + kFsWBytes + kFsSBytes, st + kFsWBytes + kFsSBytes + kFsXBytes, ng, rows,
                     lane);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&ready[s]);
      mbar_arrive(&empty[s]);
    }
  }
  return true;
}

// STALL (tests only): the producer stops before stage p.stall_at, as if its
// copies never arrived, so that the other roles' waits run out.
template <int MODE, bool Q8, bool WP = false, bool STALL = false>
__global__ void __launch_bounds__(kFsThreads, 1)
    ffn_stream_kernel(const __grid_constant__ FsMaps maps, const FsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* xch = reinterpret_cast<float*>(smem + kFsStages * kFsStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFsStages * kFsStageBytes + 2 * kFsXchBytes);
  uint64_t* empty = full + kFsStages;
  uint64_t* ready = empty + kFsStages;  // stage landed and its chain start values written

  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, p.status, p.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tma_s = p.tma_scales != 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFsStages; ++s) {
      // producer arrive.expect_tx (+ 32 cp.async arrivals when scales use cp.async)
      mbar_init(&full[s], tma_s ? 1 : 1 + 32);
      mbar_init(&empty[s], kFsCWarps + 1);  // one arrival per consumer warp + the start-value warp
      mbar_init(&ready[s], 1);
    }
    cta_abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  const int K = p.K, N = p.N;
  const int tile_n = (MODE == kGateUp) ? kFsRows / 2 : kFsRows;
  const int n_tiles = (N + tile_n - 1) / tile_n;
  const int units = (*p.n_chunks) * n_tiles;
  const int ksteps = (K + kFsKc - 1) / kFsKc;

  if (warp == kFsCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&maps.w0);
      if (MODE == kGateUp) prefetch_tensor_map(&maps.w1);
      if (tma_s) {
        prefetch_tensor_map(&maps.s0);
        if (MODE == kGateUp) prefetch_tensor_map(&maps.s1);
      }
    }
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int q = u / n_tiles, jt = u - q * n_tiles;
      ok = produce_unit<MODE, Q8, STALL>(maps, p, smem, full, empty, it, p.chunk_e[q], p.chunk_row0[q],
                                  p.chunk_rows[q], jt * tile_n, lane, wt);
    }
    // on every exit (a wait that gave up included) the issued copies land
    // before the producer leaves, so none is still writing shared memory
    // when the CTA exits
    drain_ring(full, it, kFsStages, p.status);
    return;
  }

  if (warp == kFsCWarps + 1) {
    // --------------------------------------------- chain start values
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x)
      if (!starts_unit<Q8>(p, smem, full, empty, ready, it, p.chunk_rows[u / n_tiles], lane, wt))
        return;
    return;
  }

  // -------------------------------------------------------------- consumers
  Lane L;
  L.g = lane >> 2;
  L.t = lane & 3;
  L.li = lane & 7;
  {
    // ldmatrix x4: lanes 8m..8m+7 address matrix m = (half m&1, group m>>1)
    const int m = lane >> 3;
    const int rb = 16 * warp;  // first tile row of this warp's block
    L.gsel = m >> 1;
    L.lrow_off = static_cast<uint32_t>((rb + 8 * (m & 1) + L.li) * 128);
    L.rlo = rb + L.g;
  }
  uint32_t it = 0;
  int parity = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
    const int q = u / n_tiles, jt = u - q * n_tiles;
    const int row0 = p.chunk_row0[q], rows = p.chunk_rows[q];
    const int n0 = jt * tile_n;
    float* x = xch + parity * (kFsXchBytes / 4);
    // No early exit after a failed wait: the consumer warps meet at named
    // barriers, so all of them walk every unit (the waits then return at once).
    if (rows <= 8)
      consume_unit<MODE, Q8, 1, WP>(smem, x, ready, empty, it, ksteps, row0, rows, n0, warp, lane,
                                    L, p, wt);
    else
      consume_unit<MODE, Q8, 2, WP>(smem, x, ready, empty, it, ksteps, row0, rows, n0, warp, lane,
                                    L, p, wt);
  }
}

// Acquire-load of a completion counter (another CTA's release).
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Gate/up and down of the stream kernel in one persistent launch (act_bits
// 16, scales by TMA).  Every CTA takes its gate/up units first, then its down
// units, so the down phase starts on each SM as soon as that SM is done with
// gate/up and no SM idles at the boundary.  A down unit of chunk q reads the
// h rows of chunk q: its producer waits (bounded) until the gate/up units of
// chunk q have all stored them, as counted in done[q].  Deadlock-free: a CTA
// only waits after finishing all its gate/up units, and the gate/up units
// wait on nothing but their own stages.
template <int DMODE>
__global__ void __launch_bounds__(kFsThreads, 1)
    ffn_stream_fused_kernel(const __grid_constant__ FsMaps mgu, const __grid_constant__ FsMaps mdn,
                            const FsParams pgu, const FsParams pdn, int32_t* done) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* xch = reinterpret_cast<float*>(smem + kFsStages * kFsStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFsStages * kFsStageBytes + 2 * kFsXchBytes);
  uint64_t* empty = full + kFsStages;
  uint64_t* ready = empty + kFsStages;

  __shared__ int cta_abort;
  const Waiter wt{&cta_abort, pgu.status, pgu.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFsStages; ++s) {
      mbar_init(&full[s], 1);               // both phases load their scales by TMA
      mbar_init(&empty[s], kFsCWarps + 1);
      mbar_init(&ready[s], 1);
    }
    cta_abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  const int nt_gu = (pgu.N + kFsRows / 2 - 1) / (kFsRows / 2);
  const int nt_dn = (pdn.N + kFsRows - 1) / kFsRows;
  const int n_ch = *pgu.n_chunks;
  const int units_gu = n_ch * nt_gu;
  const int units = units_gu + n_ch * nt_dn;

  if (warp == kFsCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&mgu.w0);
      prefetch_tensor_map(&mgu.w1);
      prefetch_tensor_map(&mgu.s0);
      prefetch_tensor_map(&mgu.s1);
      prefetch_tensor_map(&mdn.w0);
      prefetch_tensor_map(&mdn.s0);
    }
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      if (u < units_gu) {
        const int q = u / nt_gu, jt = u - q * nt_gu;
        ok = produce_unit<kGateUp, false>(mgu, pgu, smem, full, empty, it, pgu.chunk_e[q],
                                          pgu.chunk_row0[q], pgu.chunk_rows[q],
                                          jt * (kFsRows / 2), lane, wt);
      } else {
        const int d = u - units_gu;
        const int q = d / nt_dn, jt = d - q * nt_dn;
        // h rows of chunk q: wait for all of its gate/up units (bounded)
        if (ld_acquire(done + q) < nt_gu) {
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire(done + q) < nt_gu) {
            if (aborted(wt)) {
              ok = false;
              break;
            }
            if (static_cast<int64_t>(global_timer_ns() - t0) > wt.limit_ns) {
              give_up(wt);
              ok = false;
              break;
            }
            __nanosleep(128);
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        // the rows were stored through the generic proxy; the bulk copies
        // read them through the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        ok = produce_unit<DMODE, false>(mdn, pdn, smem, full, empty, it, pdn.chunk_e[q],
                                        pdn.chunk_row0[q], pdn.chunk_rows[q], jt * kFsRows, lane,
                                        wt);
      }
    }
    drain_ring(full, it, kFsStages, pgu.status);
    return;
  }

  if (warp == kFsCWarps + 1) {
    // --------------------------------------------- chain start values
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const bool gu = u < units_gu;
      const int q = gu ? u / nt_gu : (u - units_gu) / nt_dn;
      if (!starts_unit<false>(gu ? pgu : pdn, smem, full, empty, ready, it, pgu.chunk_rows[q], lane,
                              wt))
        return;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  Lane L;
  L.g = lane >> 2;
  L.t = lane & 3;
  L.li = lane & 7;
  {
    const int m = lane >> 3;
    const int rb = 16 * warp;
    L.gsel = m >> 1;
    L.lrow_off = static_cast<uint32_t>((rb + 8 * (m & 1) + L.li) * 128);
    L.rlo = rb + L.g;
  }
  const int ks_gu = (pgu.K + kFsKc - 1) / kFsKc;
  const int ks_dn = (pdn.K + kFsKc - 1) / kFsKc;
  uint32_t it = 0;
  int parity = 0;
  // No early exit after a failed wait: the consumer warps meet at named
  // barriers, so all of them walk every unit (the waits then return at once).
  for (int u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
    float* x = xch + parity * (kFsXchBytes / 4);
    if (u < units_gu) {
      const int q = u / nt_gu, jt = u - q * nt_gu;
      const int row0 = pgu.chunk_row0[q], rows = pgu.chunk_rows[q];
      if (rows <= 8)
        consume_unit<kGateUp, false, 1>(smem, x, ready, empty, it, ks_gu, row0, rows,
                                        jt * (kFsRows / 2), warp, lane, L, pgu, wt);
      else
        consume_unit<kGateUp, false, 2>(smem, x, ready, empty, it, ks_gu, row0, rows,
                                        jt * (kFsRows / 2), warp, lane, L, pgu, wt);
      if (warp < kFsCWarps / 2) {
        // the gate warps stored this unit's h: publish it to the down units
        __threadfence();
        named_bar_sync_n(2, kFsCWarps / 2 * 32);
        if (warp == 0 && lane == 0) atomicAdd(done + q, 1);
      }
    } else {
      const int d = u - units_gu;
      const int q = d / nt_dn, jt = d - q * nt_dn;
      const int row0 = pdn.chunk_row0[q], rows = pdn.chunk_rows[q];
      if (rows <= 8)
        consume_unit<DMODE, false, 1>(smem, x, ready, empty, it, ks_dn, row0, rows, jt * kFsRows,
                                      warp, lane, L, pdn, wt);
      else
        consume_unit<DMODE, false, 2>(smem, x, ready, empty, it, ks_dn, row0, rows, jt * kFsRows,
                                      warp, lane, L, pdn, wt);
    }
  }
}

// Prefill-shaped batches (an expert holds at least kTcMinBatchRows rows) run
// every expert on the tensor-core kernels: beyond one stream chunk (16 rows)
// the stream kernel would stream an expert's weights again, while one
// tensor-core tile dequantises them once, and the experts of few rows then
// share the tensor-core launch instead of a stream launch that covers too few
// experts to fill the GPU (the latent layer's 36 experts of <= 16 rows: 90 us
// on the stream kernel, 30 us less in the tensor-core launch).  Decode-shaped
// batches run every expert on the stream kernel.  The host launches the
// tensor-core kernels only when an expert can hold kTcMinBatchRows rows (so
// decode pays for no extra launches or fp16 copy); the schedule kernels then
// take the decision on the actual row counts.
constexpr int kTcMinRows = 1;
constexpr int kTcMinBatchRows = 48;
enum ScheduleRule { kAllShapes = 0, kDecodeShaped = 1, kPrefillShaped = 2 };

// Tensor-core kernels of act_bits 16: 1 = the CTA-pair kernels (ffn_tc2.cu)
// where a cluster of two fits, 0 = the one-CTA kernels (ffn_tc.cu).  Set by
// moe_set_tc_pair (tests and measurements compare the two).
static int g_tc_pair = 1;

static bool use_tc_pair(bool q8) { return !q8 && g_tc_pair != 0 && tc_pair_available(); }

// With the CTA-pair kernels, the experts of a prefill-shaped batch with at
// least this many rows run on them (chunks of up to 256 rows); the others stay
// on the one-CTA kernels (chunks of up to 128 rows), which lose less to a
// part-filled token tile.
constexpr int kTcPairMinRows = 129;
// The CTA-pair launches (a schedule and two kernels, ~8 us each when they find
// no expert) are made only for batches whose mean expert load rows_max / E
// reaches this many rows, where experts of kTcPairMinRows rows are expected.
constexpr int kTcPairMinMeanRows = 64;

static bool pair_batch(int rows_max, int E, int max_rows_per_expert) {
  return max_rows_per_expert >= kTcPairMinRows &&
         static_cast<long long>(rows_max) >= static_cast<long long>(kTcPairMinMeanRows) * E;
}

// The tensor-core kernels of a batch that can be prefill-shaped.  act_bits 16:
// the experts of at most kTcSmallChunkRows rows on the small-tile layout of
// the one-CTA kernels, those of kTcPairMinRows rows or more on the CTA pairs
// (pair_batch), the others on the one-CTA kernels; act_bits 8: every expert
// on the exact kernels.
struct TcPlan {
  bool small_one;      // experts of 1 .. kTcSmallChunkRows rows, small-tile layout
  bool pair;           // experts of kTcPairMinRows rows or more, CTA pairs
  int one_lo, one_hi;  // row counts of the experts on the one-CTA (128-row) kernels
};

static TcPlan tc_plan(bool q8, int rows_max, int E, int max_rows_per_expert) {
  TcPlan t{};
  t.small_one = !q8;
  t.pair = use_tc_pair(q8) && pair_batch(rows_max, E, max_rows_per_expert);
  t.one_lo = t.small_one ? kTcSmallChunkRows + 1 : kTcMinRows;
  t.one_hi = t.pair ? kTcPairMinRows - 1 : rows_max;
  return t;
}

struct Schedule;
static int launch_tc_schedules(const int32_t* offsets, int E, int rows_max, const TcPlan& t,
                               const Schedule& one, const Schedule& small_one,
                               const Schedule& pair, int* status, cudaStream_t s);

// Chunk list of the expert-sorted rows: the rows of every expert whose row
// count lies in [lo, hi] cut into chunks of at most mc rows, for a batch of
// the shape `rule` names (no chunk otherwise).  One CTA of 1024 threads.
// Offsets that are not non-decreasing or exceed rows_max record
// MOE_ERR_INVALID and give no chunk.
__global__ void __launch_bounds__(1024) ffn_schedule_kernel(const int32_t* __restrict__ offsets,
                                                            int E, int rows_max, int mc, int lo,
                                                            int hi, int rule, int max_chunks,
                                                            int32_t* __restrict__ chunk_e,
                                                            int32_t* __restrict__ chunk_row0,
                                                            int32_t* __restrict__ chunk_rows,
                                                            int32_t* __restrict__ done,
                                                            int32_t* __restrict__ n_chunks,
                                                            int* status) {
  __shared__ int32_t nch[kMaxExperts];
  __shared__ int32_t total;
  __shared__ int bad;
  __shared__ int max_cnt;
  if (threadIdx.x == 0) {
    bad = 0;
    max_cnt = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int a = offsets[e], b = offsets[e + 1];
    const int cnt = b - a;
    if (a < 0 || cnt < 0 || b > rows_max) bad = 1;
    nch[e] = (cnt > 0 && cnt >= lo && cnt <= hi) ? (cnt + mc - 1) / mc : 0;
    atomicMax(&max_cnt, cnt);
  }
  __syncthreads();
  if (rule != kAllShapes && (rule == kPrefillShaped) != (max_cnt >= kTcMinBatchRows)) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) nch[e] = 0;
    __syncthreads();
  }
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
    if (cnt <= 0 || cnt < lo || cnt > hi) continue;
    const int base = nch[e];
    for (int i = 0; i * mc < cnt; ++i) {
      chunk_e[base + i] = e;
      chunk_row0[base + i] = a + i * mc;
      chunk_rows[base + i] = min(mc, cnt - i * mc);
      done[base + i] = 0;
    }
  }
  if (threadIdx.x == 0) *n_chunks = total;
}

static int max_chunks_for(int E, int rows_max, int mc) { return (rows_max + mc - 1) / mc + E; }

struct Schedule {
  int32_t* chunk_e;
  int32_t* chunk_row0;
  int32_t* chunk_rows;
  int32_t* done;      // per chunk: gate/up units finished (fused kernel), zeroed here
  int32_t* n_chunks;
  int max_chunks;
};

static size_t schedule_bytes_one(int E, int rows_max, int mc) {
  const size_t n = static_cast<size_t>(max_chunks_for(E, rows_max, mc));
  return 4 * align_up(n * sizeof(int32_t), 256) + 256;
}

static Schedule carve_one(char*& b, int E, int rows_max, int mc) {
  Schedule s;
  s.max_chunks = max_chunks_for(E, rows_max, mc);
  const size_t arr = align_up(static_cast<size_t>(s.max_chunks) * sizeof(int32_t), 256);
  s.chunk_e = reinterpret_cast<int32_t*>(b);
  s.chunk_row0 = reinterpret_cast<int32_t*>(b + arr);
  s.chunk_rows = reinterpret_cast<int32_t*>(b + 2 * arr);
  s.done = reinterpret_cast<int32_t*>(b + 3 * arr);
  s.n_chunks = reinterpret_cast<int32_t*>(b + 4 * arr);
  b += 4 * arr + 256;
  return s;
}

size_t row_chunk_bytes(int E, int rows_max, int mc) { return schedule_bytes_one(E, rows_max, mc); }

static int launch_schedule(const int32_t* offsets, int E, int rows_max, int mc, int lo, int hi,
                           const Schedule& sc, int* status, cudaStream_t s,
                           int rule = kAllShapes);

int launch_row_chunks(const int32_t* offsets, int E, int rows_max, int mc, void* ws,
                      RowChunks* rc_out, int* status, cudaStream_t s) {
  char* b = static_cast<char*>(ws);
  const Schedule sc = carve_one(b, E, rows_max, mc);
  rc_out->chunk_e = sc.chunk_e;
  rc_out->chunk_row0 = sc.chunk_row0;
  rc_out->chunk_rows = sc.chunk_rows;
  rc_out->n_chunks = sc.n_chunks;
  rc_out->max_chunks = sc.max_chunks;
  return launch_schedule(offsets, E, rows_max, mc, 1, rows_max, sc, status, s, kAllShapes);
}

// Stream-kernel list plus the three tensor-core lists (one-CTA kernels,
// their small-tile layout, and the CTA-pair kernels).
static size_t schedule_bytes(int E, int rows_max) {
  return schedule_bytes_one(E, rows_max, kFsMc) + schedule_bytes_one(E, rows_max, kTcChunkRows) +
         schedule_bytes_one(E, rows_max, kTcPairChunkRows) +
         schedule_bytes_one(E, rows_max, kTcSmallChunkRows);
}

static int launch_schedule(const int32_t* offsets, int E, int rows_max, int mc, int lo, int hi,
                           const Schedule& sc, int* status, cudaStream_t s,
                           int rule) {
  ffn_schedule_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, mc, lo, hi, rule, sc.max_chunks,
                                         sc.chunk_e, sc.chunk_row0, sc.chunk_rows, sc.done,
                                         sc.n_chunks, status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static int launch_tc_schedules(const int32_t* offsets, int E, int rows_max, const TcPlan& t,
                               const Schedule& one, const Schedule& small_one,
                               const Schedule& pair, int* status, cudaStream_t s) {
  int rc = launch_schedule(offsets, E, rows_max, kTcChunkRows, t.one_lo, t.one_hi, one, status, s,
                           kPrefillShaped);
  if (!rc && t.small_one)
    rc = launch_schedule(offsets, E, rows_max, kTcSmallChunkRows, kTcMinRows, kTcSmallChunkRows,
                         small_one, status, s, kPrefillShaped);
  if (!rc && t.pair)
    rc = launch_schedule(offsets, E, rows_max, kTcPairChunkRows, kTcPairMinRows, rows_max, pair,
                         status, s, kPrefillShaped);
  return rc;
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

// Tensor map of bf16 scales [E, N, K/32] with a box of `rows` rows x 8 groups
// (16 bytes, no swizzle).  Valid when K % 256 == 0 (16-byte row strides).
static bool scale_map(CUtensorMap* m, const uint16_t* sc, int E, int N, int K, int rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K / kGroup), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K / kGroup) * 2,
                               static_cast<uint64_t>(N) * (K / kGroup) * 2};
  const uint32_t box[3] = {static_cast<uint32_t>(kFsGroups), static_cast<uint32_t>(rows), 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, sc, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Scales by TMA: rows of a multiple of 8 groups starting on 16-byte boundaries.
static bool tma_scales_ok(int K, const uint16_t* s0, const uint16_t* s1) {
  return K % kFsKc == 0 && aligned(s0, 16) && aligned(s1, 16);
}

// Maps of one stream launch: w0/s0 the first (or only) matrix, w1/s1 the second.
static bool make_maps(FsMaps* m, const int32_t* w0, const uint16_t* s0, const int32_t* w1,
                      const uint16_t* s1, int E, int N, int K, int rows) {
  if (!weight_map(&m->w0, w0, E, N, K, rows) || !weight_map(&m->w1, w1, E, N, K, rows))
    return false;
  if (tma_scales_ok(K, s0, s1)) {
    if (!scale_map(&m->s0, s0, E, N, K, rows) || !scale_map(&m->s1, s1, E, N, K, rows))
      return false;
  } else {
    m->s0 = m->w0;  // unused
    m->s1 = m->w1;
  }
  return true;
}

template <int MODE, bool Q8, bool WP = false, bool STALL = false>
static int launch_stream(const FsMaps& maps, const FsParams& p, cudaStream_t s) {
  auto kern = ffn_stream_kernel<MODE, Q8, WP, STALL>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kFsSmemBytes));
  kern<<<num_sms(), kFsThreads, kFsSmemBytes, s>>>(maps, p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static int run_stream(int mode, bool q8, const FsMaps& maps, const FsParams& p, cudaStream_t s) {
  if (mode == kGateUp) return q8 ? launch_stream<kGateUp, true>(maps, p, s)
                                 : launch_stream<kGateUp, false>(maps, p, s);
  if (mode == kDown) return q8 ? launch_stream<kDown, true>(maps, p, s)
                               : launch_stream<kDown, false>(maps, p, s);
  return q8 ? launch_stream<kLinear, true>(maps, p, s) : launch_stream<kLinear, false>(maps, p, s);
}

template <int DMODE>
static int launch_fused(const FsMaps& mgu, const FsMaps& mdn, const FsParams& pgu,
                        const FsParams& pdn, int32_t* done, cudaStream_t s) {
  auto kern = ffn_stream_fused_kernel<DMODE>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kFsSmemBytes));
  kern<<<num_sms(), kFsThreads, kFsSmemBytes, s>>>(mgu, mdn, pgu, pdn, done);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static int check_width(int v) { return (v > 0 && v % 64 == 0) ? MOE_OK : MOE_ERR_UNSUPPORTED; }

}  // namespace moe

using namespace moe;

size_t moe::expert_ffn_ws_bytes(int E, int D, int I, int rows_max, int act_bits) {
  size_t b = schedule_bytes(E, rows_max);
  b += align_up((size_t)rows_max * I * sizeof(uint16_t), 256);  // h (fp16, bf16 with act_bits 8)
  if (act_bits == 8) {
    b += align_up((size_t)rows_max * I, 256);                      // h as int8
    b += align_up((size_t)rows_max * sizeof(float), 256);          // its row scales
    b += align_up((size_t)rows_max * D * sizeof(uint16_t), 256);   // fp16 of the int8 x (tensor cores)
    b += align_up((size_t)rows_max * I * sizeof(uint16_t), 256);   // fp16 of the int8 h (tensor cores)
  }
  return b;
}

int moe::launch_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets,
                           int E, int D, int I, int rows_max, int max_rows_per_expert,
                           const int32_t* gate_packed, const uint16_t* gate_scale,
                           const int32_t* up_packed, const uint16_t* up_scale,
                           const int32_t* down_packed, const uint16_t* down_scale, int act_bits,
                           void* y, bool y_f32, void* ws, cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const bool q8 = act_bits == 8;
  char* b = static_cast<char*>(ws);
  Schedule small = carve_one(b, E, rows_max, kFsMc);
  Schedule big = carve_one(b, E, rows_max, kTcChunkRows);
  Schedule big2 = carve_one(b, E, rows_max, kTcPairChunkRows);
  Schedule sm1 = carve_one(b, E, rows_max, kTcSmallChunkRows);
  uint16_t* h = reinterpret_cast<uint16_t*>(b);
  b += align_up((size_t)rows_max * I * sizeof(uint16_t), 256);
  int8_t* hq = nullptr;
  float* hs = nullptr;
  uint16_t* x16 = nullptr;
  uint16_t* h16 = nullptr;
  if (q8) {
    hq = reinterpret_cast<int8_t*>(b);
    b += align_up((size_t)rows_max * I, 256);
    hs = reinterpret_cast<float*>(b);
    b += align_up((size_t)rows_max * sizeof(float), 256);
    x16 = reinterpret_cast<uint16_t*>(b);
    b += align_up((size_t)rows_max * D * sizeof(uint16_t), 256);
    h16 = reinterpret_cast<uint16_t*>(b);
  }

  // the tensor-core kernels run when an expert can hold kTcMinBatchRows rows;
  // the schedules then give every expert to one of the two paths, by the
  // batch's actual shape
  const bool use_tc = tc_path_supported(D) && tc_path_supported(I) &&
                      max_rows_per_expert >= kTcMinBatchRows;
  const TcPlan plan = tc_plan(q8, rows_max, E, max_rows_per_expert);
  int rc = launch_schedule(offsets, E, rows_max, kFsMc, 0, rows_max, small, status, s,
                           use_tc ? kDecodeShaped : kAllShapes);
  if (rc) return rc;
  if (use_tc) {
    rc = launch_tc_schedules(offsets, E, rows_max, plan, big, sm1, big2, status, s);
    if (rc) return rc;
  }

  FsMaps mgu, md;
  if (!make_maps(&mgu, gate_packed, gate_scale, up_packed, up_scale, E, I, D, kFsRows / 2) ||
      !make_maps(&md, down_packed, down_scale, down_packed, down_scale, E, D, I, kFsRows))
    return MOE_ERR_CUDA;

  FsParams p{};
  FsParams pd{};
  p.x = x_sorted;
  p.x_scale = x_scale;
  p.scale0 = gate_scale;
  p.scale1 = up_scale;
  p.out = h;
  p.chunk_e = small.chunk_e;
  p.chunk_row0 = small.chunk_row0;
  p.chunk_rows = small.chunk_rows;
  p.n_chunks = small.n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = D;
  p.N = I;
  p.tma_scales = tma_scales_ok(D, gate_scale, up_scale) ? 1 : 0;
  pd = p;
  pd.K = I;
  pd.N = D;
  pd.tma_scales = tma_scales_ok(I, down_scale, down_scale) ? 1 : 0;
  pd.scale0 = down_scale;
  pd.scale1 = nullptr;
  pd.out = y;
  pd.x = h;
  // act_bits 16 with TMA-loaded scales: gate/up and down of the stream
  // experts in one launch (no re-quantisation of h between them)
  const bool fused = !q8 && p.tma_scales && pd.tma_scales;
  if (fused) {
    rc = y_f32 ? launch_fused<kLinear>(mgu, md, p, pd, small.done, s)
               : launch_fused<kDown>(mgu, md, p, pd, small.done, s);
  } else {
    rc = run_stream(kGateUp, q8, mgu, p, s);
  }
  if (rc) return rc;
  if (use_tc) {
    // both kernels write h in pair order: fp16 (act_bits 16), or bf16 for
    // the re-quantisation below (act_bits 8)
    const uint16_t* xa = static_cast<const uint16_t*>(x_sorted);
    if (q8) {
      rc = launch_to_f16_rows(x_sorted, true, rows_max, D, offsets + E, x16, s);
      if (rc) return rc;
      xa = x16;
    }
    rc = q8 ? launch_tc_q8_gateup(xa, x_scale, rows_max, E, D, I, gate_packed, gate_scale,
                                  up_packed, up_scale, h, big.chunk_e, big.chunk_row0,
                                  big.chunk_rows, big.n_chunks, status, s)
            : launch_tc_gateup(xa, rows_max, E, D, I, gate_packed, gate_scale, up_packed, up_scale,
                               h, big.chunk_e, big.chunk_row0, big.chunk_rows, big.n_chunks,
                               status, s);
    if (rc) return rc;
    if (plan.small_one) {
      rc = launch_tc_gateup(xa, rows_max, E, D, I, gate_packed, gate_scale, up_packed, up_scale,
                            h, sm1.chunk_e, sm1.chunk_row0, sm1.chunk_rows, sm1.n_chunks, status,
                            s, true);
      if (rc) return rc;
    }
    if (plan.pair) {
      rc = launch_tc_pair_gateup(xa, rows_max, E, D, I, gate_packed, gate_scale, up_packed,
                                 up_scale, h, big2.chunk_e, big2.chunk_row0, big2.chunk_rows,
                                 big2.n_chunks, status, s);
      if (rc) return rc;
    }
  }

  if (q8) {
    // the tensor-core down kernel reads the fp16 copy of the codes, written
    // in the same pass
    rc = launch_quantize_rows(h, rows_max, I, offsets + E, hq, hs, s, use_tc ? h16 : nullptr);
    if (rc) return rc;
    pd.x = hq;
    pd.x_scale = hs;
  }
  if (!fused) {
    rc = run_stream(y_f32 ? kLinear : kDown, q8, md, pd, s);
    if (rc) return rc;
  }
  if (use_tc) {
    const uint16_t* ha = q8 ? h16 : h;
    rc = q8 ? launch_tc_q8_down(ha, hs, rows_max, E, D, I, down_packed, down_scale, y, y_f32,
                                big.chunk_e, big.chunk_row0, big.chunk_rows, big.n_chunks, status,
                                s, nullptr)
            : launch_tc_down(ha, rows_max, E, D, I, down_packed, down_scale, y, y_f32,
                             big.chunk_e, big.chunk_row0, big.chunk_rows, big.n_chunks, status, s);
    if (rc) return rc;
    if (plan.small_one) {
      rc = launch_tc_down(ha, rows_max, E, D, I, down_packed, down_scale, y, y_f32, sm1.chunk_e,
                          sm1.chunk_row0, sm1.chunk_rows, sm1.n_chunks, status, s, true);
      if (rc) return rc;
    }
    if (plan.pair) {
      rc = launch_tc_pair_down(ha, rows_max, E, D, I, down_packed, down_scale, y, y_f32,
                               big2.chunk_e, big2.chunk_row0, big2.chunk_rows, big2.n_chunks,
                               status, s);
      if (rc) return rc;
    }
  }
  return MOE_OK;
}

// Argument checks shared by the two expert-FFN entry points.
static int check_ffn_args(const void* x, const float* x_scale, const int32_t* offsets, int E, int D,
                          int I, int rows_max, const int32_t* gate_packed,
                          const uint16_t* gate_scale, const int32_t* up_packed,
                          const uint16_t* up_scale, const int32_t* down_packed,
                          const uint16_t* down_scale, int act_bits, const uint16_t* y, void* ws) {
  if (E <= 0 || rows_max < 0) return MOE_ERR_INVALID;
  if (check_width(D) || check_width(I) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x || !offsets || !gate_packed || !gate_scale || !up_packed || !up_scale || !down_packed ||
      !down_scale || !y || !ws)
    return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(gate_packed, 16) || !aligned(up_packed, 16) ||
      !aligned(down_packed, 16) || !aligned(gate_scale, 4) || !aligned(up_scale, 4) ||
      !aligned(down_scale, 4) || !aligned(ws, 256))
    return MOE_ERR_INVALID;
  return MOE_OK;
}

extern "C" size_t moe_expert_ffn_pairs_workspace_size(int E, int D, int I, int rows_max,
                                                      int act_bits) {
  if (E <= 0 || D <= 0 || I <= 0 || rows_max < 0) return 256;
  return expert_ffn_ws_bytes(E, D, I, rows_max, act_bits);
}

extern "C" int moe_expert_ffn_pairs(const void* x_pairs, const float* x_scale,
                                    const int32_t* offsets, int E, int D, int I, int rows_max,
                                    const int32_t* gate_packed, const uint16_t* gate_scale,
                                    const int32_t* up_packed, const uint16_t* up_scale,
                                    const int32_t* down_packed, const uint16_t* down_scale,
                                    int act_bits, uint16_t* y_sorted, void* ws, size_t ws_bytes,
                                    void* stream) {
  moe::Range range_("moe_expert_ffn_pairs");
  const int rc = check_ffn_args(x_pairs, x_scale, offsets, E, D, I, rows_max, gate_packed,
                                gate_scale, up_packed, up_scale, down_packed, down_scale, act_bits,
                                y_sorted, ws);
  if (rc || rows_max == 0) return rc;
  if (ws_bytes < moe_expert_ffn_pairs_workspace_size(E, D, I, rows_max, act_bits))
    return MOE_ERR_WORKSPACE;
  return launch_expert_ffn(x_pairs, x_scale, offsets, E, D, I, rows_max, rows_max, gate_packed,
                           gate_scale, up_packed, up_scale, down_packed, down_scale, act_bits,
                           y_sorted, false, ws, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_expert_ffn_pairs_bounded(const void* x_pairs, const float* x_scale,
                                            const int32_t* offsets, int E, int D, int I,
                                            int rows_max, int max_rows_per_expert,
                                            const int32_t* gate_packed, const uint16_t* gate_scale,
                                            const int32_t* up_packed, const uint16_t* up_scale,
                                            const int32_t* down_packed,
                                            const uint16_t* down_scale, int act_bits,
                                            uint16_t* y_sorted, void* ws, size_t ws_bytes,
                                            void* stream) {
  moe::Range range_("moe_expert_ffn_pairs_bounded");
  if (max_rows_per_expert < 0) return MOE_ERR_INVALID;
  const int rc = check_ffn_args(x_pairs, x_scale, offsets, E, D, I, rows_max, gate_packed,
                                gate_scale, up_packed, up_scale, down_packed, down_scale, act_bits,
                                y_sorted, ws);
  if (rc || rows_max == 0) return rc;
  if (ws_bytes < moe_expert_ffn_pairs_workspace_size(E, D, I, rows_max, act_bits))
    return MOE_ERR_WORKSPACE;
  // the bound only selects which kernels are launched: every expert still
  // gets a kernel whatever its row count (a bound below 48 puts all of them
  // on the stream kernel)
  return launch_expert_ffn(x_pairs, x_scale, offsets, E, D, I, rows_max,
                           max_rows_per_expert < rows_max ? max_rows_per_expert : rows_max,
                           gate_packed, gate_scale,
                           up_packed, up_scale, down_packed, down_scale, act_bits, y_sorted, false,
                           ws, static_cast<cudaStream_t>(stream));
}

extern "C" size_t moe_expert_ffn_workspace_size(int E, int D, int I, int rows_max, int act_bits) {
  if (E <= 0 || D <= 0 || I <= 0 || rows_max < 0) return 256;
  // + the pair-ordered copy of x_sorted
  return expert_ffn_ws_bytes(E, D, I, rows_max, act_bits) +
         align_up((size_t)rows_max * D * (act_bits == 8 ? 1 : 2), 256);
}

extern "C" int moe_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets,
                              int E, int D, int I, int rows_max, const int32_t* gate_packed,
                              const uint16_t* gate_scale, const int32_t* up_packed,
                              const uint16_t* up_scale, const int32_t* down_packed,
                              const uint16_t* down_scale, int act_bits, uint16_t* y_sorted,
                              void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_expert_ffn");
  const int rc0 = check_ffn_args(x_sorted, x_scale, offsets, E, D, I, rows_max, gate_packed,
                                 gate_scale, up_packed, up_scale, down_packed, down_scale,
                                 act_bits, y_sorted, ws);
  if (rc0 || rows_max == 0) return rc0;
  if (ws_bytes < moe_expert_ffn_workspace_size(E, D, I, rows_max, act_bits))
    return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* xp = static_cast<char*>(ws) + expert_ffn_ws_bytes(E, D, I, rows_max, act_bits);
  int rc = launch_to_pair_rows(x_sorted, act_bits == 8, rows_max, D, offsets + E, xp, status, s);
  if (rc) return rc;
  return launch_expert_ffn(xp, x_scale, offsets, E, D, I, rows_max, rows_max, gate_packed,
                           gate_scale, up_packed, up_scale, down_packed, down_scale, act_bits,
                           y_sorted, false, ws, s);
}

extern "C" size_t moe_int4_linear_partials_workspace_size(int E, int K, int rows_max) {
  if (E <= 0 || K <= 0 || rows_max < 0) return 256;
  return schedule_bytes(E, rows_max) +
         align_up((size_t)rows_max * K, 256) +                     // pair-ordered int8 x
         align_up((size_t)rows_max * K * sizeof(uint16_t), 256);   // its fp16 form
}

extern "C" int moe_int4_linear_partials(const int8_t* x, const float* x_scale,
                                        const int32_t* offsets, int E, int K, int N, int rows_max,
                                        const int32_t* w_packed, const uint16_t* w_scale,
                                        int kernel, float* out, int32_t* partials, void* ws,
                                        size_t ws_bytes, void* stream) {
  moe::Range range_("moe_int4_linear_partials");
  if (E <= 0 || rows_max < 0 || N <= 0) return MOE_ERR_INVALID;
  if (kernel != 0 && kernel != 1) return MOE_ERR_INVALID;
  if (check_width(K) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x || !x_scale || !offsets || !w_packed || !w_scale || !out || !partials || !ws)
    return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scale, 4) || !aligned(out, 16) ||
      !aligned(partials, 4) || !aligned(ws, 256))
    return MOE_ERR_INVALID;
  if (ws_bytes < moe_int4_linear_partials_workspace_size(E, K, rows_max)) return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(ws);
  Schedule sc = carve_one(b, E, rows_max, kernel == 0 ? kFsMc : kTcChunkRows);
  b = static_cast<char*>(ws) + schedule_bytes(E, rows_max);
  void* xp = b;
  b += align_up((size_t)rows_max * K, 256);
  uint16_t* x16 = reinterpret_cast<uint16_t*>(b);
  int rc = launch_to_pair_rows(x, true, rows_max, K, offsets + E, xp, status, s);
  if (rc) return rc;
  // every expert with rows on the chosen kernel
  rc = launch_schedule(offsets, E, rows_max, kernel == 0 ? kFsMc : kTcChunkRows, 1, rows_max, sc,
                       status, s);
  if (rc) return rc;
  if (kernel == 0) {
    FsMaps m;
    if (!make_maps(&m, w_packed, w_scale, w_packed, w_scale, E, N, K, kFsRows)) return MOE_ERR_CUDA;
    FsParams p{};
    p.x = xp;
    p.x_scale = x_scale;
    p.scale0 = w_scale;
    p.out = out;
    p.partials = partials;
    p.chunk_e = sc.chunk_e;
    p.chunk_row0 = sc.chunk_row0;
    p.chunk_rows = sc.chunk_rows;
    p.n_chunks = sc.n_chunks;
    p.status = status;
    p.wait_ns = kDefaultWaitNs;
    p.K = K;
    p.N = N;
    p.tma_scales = tma_scales_ok(K, w_scale, w_scale) ? 1 : 0;
    return launch_stream<kLinear, true, true>(m, p, s);
  }
  rc = launch_to_f16_rows(xp, true, rows_max, K, offsets + E, x16, s);
  if (rc) return rc;
  return launch_tc_q8_down(x16, x_scale, rows_max, E, N, K, w_packed, w_scale, out, true,
                           sc.chunk_e, sc.chunk_row0, sc.chunk_rows, sc.n_chunks, status, s,
                           partials);
}

extern "C" int moe_int4_linear_stall_selftest(const void* x, const float* x_scale,
                                              const int32_t* offsets, int E, int K, int N,
                                              int rows_max, const int32_t* w_packed,
                                              const uint16_t* w_scale, int act_bits, int kernel,
                                              int stall_stage, int64_t limit_ns, float* out,
                                              void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_int4_linear_stall_selftest");
  if (E <= 0 || rows_max <= 0 || N <= 0 || stall_stage < 0) return MOE_ERR_INVALID;
  if (kernel < 0 || kernel > 3) return MOE_ERR_INVALID;
  if (kernel == 2 && (act_bits != 16 || !tc_pair_available())) return MOE_ERR_UNSUPPORTED;
  if (kernel == 3 && act_bits != 16) return MOE_ERR_UNSUPPORTED;
  if (limit_ns < 1000 || limit_ns > 5000000000LL) return MOE_ERR_INVALID;
  if (check_width(K) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!x || !offsets || !w_packed || !w_scale || !out || !ws) return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scale, 4) || !aligned(out, 16) ||
      !aligned(ws, 256))
    return MOE_ERR_INVALID;
  if (ws_bytes < moe_int4_linear_workspace_size(E, K, rows_max)) return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool q8 = act_bits == 8;
  const int mc = kernel == 0   ? kFsMc
                 : kernel == 1 ? kTcChunkRows
                 : kernel == 2 ? kTcPairChunkRows
                               : kTcSmallChunkRows;
  char* b = static_cast<char*>(ws);
  Schedule sc = carve_one(b, E, rows_max, mc);
  b = static_cast<char*>(ws) + schedule_bytes(E, rows_max);
  void* xp = b;
  b += align_up((size_t)rows_max * K * sizeof(uint16_t), 256);
  uint16_t* x16 = reinterpret_cast<uint16_t*>(b);
  int rc = launch_to_pair_rows(x, q8, rows_max, K, offsets + E, xp, status, s);
  if (rc) return rc;
  rc = launch_schedule(offsets, E, rows_max, mc, 1, rows_max, sc, status, s);
  if (rc) return rc;
  if (kernel == 0) {
    FsMaps m;
    if (!make_maps(&m, w_packed, w_scale, w_packed, w_scale, E, N, K, kFsRows)) return MOE_ERR_CUDA;
    FsParams p{};
    p.x = xp;
    p.x_scale = x_scale;
    p.scale0 = w_scale;
    p.out = out;
    p.chunk_e = sc.chunk_e;
    p.chunk_row0 = sc.chunk_row0;
    p.chunk_rows = sc.chunk_rows;
    p.n_chunks = sc.n_chunks;
    p.status = status;
    p.wait_ns = limit_ns;
    p.stall_at = stall_stage;
    p.K = K;
    p.N = N;
    p.tma_scales = tma_scales_ok(K, w_scale, w_scale) ? 1 : 0;
    return q8 ? launch_stream<kLinear, true, false, true>(m, p, s)
              : launch_stream<kLinear, false, false, true>(m, p, s);
  }
  const uint16_t* xa = static_cast<const uint16_t*>(xp);
  if (kernel == 2)
    return launch_tc_pair_linear_stalled(xa, rows_max, E, N, K, w_packed, w_scale, out,
                                         sc.chunk_e, sc.chunk_row0, sc.chunk_rows, sc.n_chunks,
                                         status, limit_ns, stall_stage, s);
  if (q8) {
    rc = launch_to_f16_rows(xp, true, rows_max, K, offsets + E, x16, s);
    if (rc) return rc;
    xa = x16;
  }
  return launch_tc_linear_stalled(xa, q8 ? x_scale : nullptr, rows_max, E, N, K, w_packed, w_scale,
                                  out, sc.chunk_e, sc.chunk_row0, sc.chunk_rows, sc.n_chunks,
                                  status, limit_ns, stall_stage, s, kernel == 3);
}

extern "C" size_t moe_int4_linear_workspace_size(int E, int K, int rows_max) {
  if (E <= 0 || K <= 0 || rows_max < 0) return 256;
  return schedule_bytes(E, rows_max) +
         align_up((size_t)rows_max * K * sizeof(uint16_t), 256) +  // pair-ordered copy of x
         align_up((size_t)rows_max * K * sizeof(uint16_t), 256);   // its fp16 form (int8 x)
}

extern "C" int moe_int4_linear(const void* x, const float* x_scale, const int32_t* offsets, int E,
                               int K, int N, int rows_max, const int32_t* w_packed,
                               const uint16_t* w_scale, int act_bits, float* out, void* ws,
                               size_t ws_bytes, void* stream) {
  moe::Range range_("moe_int4_linear");
  if (E <= 0 || rows_max < 0 || N <= 0) return MOE_ERR_INVALID;
  if (check_width(K) || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x || !offsets || !w_packed || !w_scale || !out || !ws) return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scale, 4) || !aligned(out, 16) ||
      !aligned(ws, 256))
    return MOE_ERR_INVALID;
  if (ws_bytes < moe_int4_linear_workspace_size(E, K, rows_max)) return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool q8 = act_bits == 8;
  char* b = static_cast<char*>(ws);
  Schedule small = carve_one(b, E, rows_max, kFsMc);
  Schedule big = carve_one(b, E, rows_max, kTcChunkRows);
  Schedule big2 = carve_one(b, E, rows_max, kTcPairChunkRows);
  Schedule sm1 = carve_one(b, E, rows_max, kTcSmallChunkRows);
  void* xp = b;
  b += align_up((size_t)rows_max * K * sizeof(uint16_t), 256);
  uint16_t* x16 = reinterpret_cast<uint16_t*>(b);
  const bool use_tc = tc_path_supported(K) && rows_max >= kTcMinBatchRows;
  const TcPlan plan = tc_plan(q8, rows_max, E, rows_max);
  int rc = launch_to_pair_rows(x, q8, rows_max, K, offsets + E, xp, status, s);
  if (rc) return rc;
  rc = launch_schedule(offsets, E, rows_max, kFsMc, 0, rows_max, small, status, s,
                       use_tc ? kDecodeShaped : kAllShapes);
  if (rc) return rc;
  FsMaps m;
  if (!make_maps(&m, w_packed, w_scale, w_packed, w_scale, E, N, K, kFsRows)) return MOE_ERR_CUDA;
  FsParams p{};
  p.x = xp;
  p.x_scale = x_scale;
  p.scale0 = w_scale;
  p.out = out;
  p.chunk_e = small.chunk_e;
  p.chunk_row0 = small.chunk_row0;
  p.chunk_rows = small.chunk_rows;
  p.n_chunks = small.n_chunks;
  p.status = status;
  p.wait_ns = kDefaultWaitNs;
  p.K = K;
  p.N = N;
  p.tma_scales = tma_scales_ok(K, w_scale, w_scale) ? 1 : 0;
  rc = run_stream(kLinear, q8, m, p, s);
  if (rc || !use_tc) return rc;
  rc = launch_tc_schedules(offsets, E, rows_max, plan, big, sm1, big2, status, s);
  if (rc) return rc;
  const uint16_t* xa = static_cast<const uint16_t*>(xp);
  if (q8) {
    rc = launch_to_f16_rows(xp, true, rows_max, K, offsets + E, x16, s);
    if (rc) return rc;
    xa = x16;
  }
  if (q8)
    return launch_tc_q8_down(xa, x_scale, rows_max, E, N, K, w_packed, w_scale, out, true,
                             big.chunk_e, big.chunk_row0, big.chunk_rows, big.n_chunks, status, s,
                             nullptr);
  rc = launch_tc_down(xa, rows_max, E, N, K, w_packed, w_scale, out, true, big.chunk_e,
                      big.chunk_row0, big.chunk_rows, big.n_chunks, status, s);
  if (!rc && plan.small_one)
    rc = launch_tc_down(xa, rows_max, E, N, K, w_packed, w_scale, out, true, sm1.chunk_e,
                        sm1.chunk_row0, sm1.chunk_rows, sm1.n_chunks, status, s, true);
  if (!rc && plan.pair)
    rc = launch_tc_pair_down(xa, rows_max, E, N, K, w_packed, w_scale, out, true, big2.chunk_e,
                             big2.chunk_row0, big2.chunk_rows, big2.n_chunks, status, s);
  return rc;
}

extern "C" int moe_set_tc_pair(int enable) {
  const int prev = g_tc_pair;
  g_tc_pair = enable ? 1 : 0;
  return prev;
}
