// The int16 / int64 reading of act_bits = 16 for one grouped PackedInt4Linear
// (Kimi exact-generator adaptation page, "Sources & provenance": the
// routed experts' PackedInt4Linear with act_bits 16 by default and an "int64
// exact int4 MAC"; the page does not say what the 16 bits hold).  This
// reading quantises each activation row to int16 codes and accumulates code
// products as integers: a = max|x| over the row, sx = a / 32767 (IEEE fp32,
// rounded to nearest), q = clamp(rint(x / sx), -32767, 32767); per 32-column
// weight group the partial P = sum q * q_w is an exact integer (|P| <= 32 *
// 8 * 32767 < 2^23; K * 8 * 32767 < 2^31 keeps a whole-K int32 sum exact
// too); y = sx * acc with acc the fp32 chain fma(scale[n, g], P_g, acc) over
// the groups in K order.  The layer's act_bits 16 path is the other reading,
// bf16 activations times exactly dequantised weights; this entry point
// serves the comparison of the two.
//
// SIMT integer arithmetic: one CTA per (chunk of <= 16 expert rows, 64
// outputs), 256 threads, thread (row, 4 outputs); per group the chunk's
// codes and the tile's packed words are staged in shared memory.
#include <algorithm>

#include "combine.cuh"
#include "common.cuh"

namespace moe {

namespace {

constexpr int kI16Rows = 16;     // rows per chunk
constexpr int kI16Outs = 64;     // outputs per CTA tile
constexpr int kI16MaxK = 8160;   // K * 8 * 32767 < 2^31
constexpr int kI16Max = 32767;

// One warp per row of R rows x C bf16 values: scale and int16 codes.  Rows at
// or beyond *row_count (when given) are skipped.
__global__ void __launch_bounds__(256) quantize_rows_i16_kernel(const uint16_t* __restrict__ v,
                                                                int R, int C,
                                                                const int32_t* row_count,
                                                                int16_t* __restrict__ q,
                                                                float* __restrict__ scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= R || (row_count && r >= *row_count)) return;
  const uint16_t* row = v + (size_t)r * C;
  float a = 0.f;
  for (int c = lane; c < C; c += 32) a = fmaxf(a, fabsf(bf16_bits_to_f32(row[c])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float sc = __fdiv_rn(a, static_cast<float>(kI16Max));
  int16_t* qr = q + (size_t)r * C;
  for (int c = lane; c < C; c += 32) {
    int qi = 0;
    if (sc > 0.f) qi = min(max(__float2int_rn(__fdiv_rn(bf16_bits_to_f32(row[c]), sc)), -kI16Max), kI16Max);
    qr[c] = static_cast<int16_t>(qi);
  }
  if (lane == 0) scale[r] = sc;
}

// Signed nibble j of a packed word.
__device__ __forceinline__ int nib(uint32_t w, int j) {
  return static_cast<int>(w << (28 - 4 * j)) >> 28;
}

__global__ void __launch_bounds__(256) linear_i16_kernel(
    const int16_t* __restrict__ q, const float* __restrict__ sx, const int32_t* chunk_e,
    const int32_t* chunk_row0, const int32_t* chunk_rows, const int32_t* n_chunks, int K, int N,
    const int32_t* __restrict__ w_packed, const uint16_t* __restrict__ w_scale,
    float* __restrict__ out, int32_t* __restrict__ partials) {
  __shared__ int16_t xs[kI16Rows][kGroup];
  __shared__ uint32_t ws[kI16Outs][kGroup / 8];
  const int n_tiles = (N + kI16Outs - 1) / kI16Outs;
  const int units = *n_chunks * n_tiles;
  const int G = K / kGroup;
  const int tr = threadIdx.x >> 4;       // row of the chunk
  const int tn = (threadIdx.x & 15) * 4; // first of this thread's 4 outputs
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int c = u / n_tiles, jt = u - c * n_tiles;
    const int e = chunk_e[c], row0 = chunk_row0[c], rows = chunk_rows[c];
    const int n0 = jt * kI16Outs;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = 0; g < G; ++g) {
      __syncthreads();  // the previous group's tiles are no longer read
      {
        // 16 rows x 32 codes: two codes per thread
        const int r = threadIdx.x >> 4, c2 = (threadIdx.x & 15) * 2;
        int16_t a0 = 0, a1 = 0;
        if (r < rows) {  // rows past the chunk are not read
          const int16_t* src = q + (size_t)(row0 + r) * K + g * kGroup + c2;
          a0 = src[0];
          a1 = src[1];
        }
        xs[r][c2] = a0;
        xs[r][c2 + 1] = a1;
        // 64 weight rows x 4 words: one word per thread
        const int wn = threadIdx.x >> 2, wk = threadIdx.x & 3;
        const int n = n0 + wn;
        ws[wn][wk] = n < N ? static_cast<uint32_t>(
                                 w_packed[((size_t)e * N + n) * (K / 8) + g * 4 + wk])
                           : 0u;
      }
      __syncthreads();
      int P[4] = {0, 0, 0, 0};
#pragma unroll
      for (int wk = 0; wk < 4; ++wk) {
        const uint32_t w[4] = {ws[tn][wk], ws[tn + 1][wk], ws[tn + 2][wk], ws[tn + 3][wk]};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int xv = xs[tr][8 * wk + j];
#pragma unroll
          for (int i = 0; i < 4; ++i) P[i] += xv * nib(w[i], j);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + tn + i;
        if (n >= N || tr >= rows) continue;
        const float s = bf16_bits_to_f32(w_scale[((size_t)e * N + n) * G + g]);
        acc[i] = fmaf(s, static_cast<float>(P[i]), acc[i]);
        if (partials) partials[((size_t)(row0 + tr) * N + n) * G + g] = P[i];
      }
    }
    if (tr < rows) {
      const float scx = sx[row0 + tr];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + tn + i;
        if (n < N) out[(size_t)(row0 + tr) * N + n] = scx * acc[i];
      }
    }
  }
}

struct I16Ws {
  int16_t* q;
  float* sx;
  size_t total;
};

I16Ws i16_carve(int E, int K, int rows_max, void* base) {
  I16Ws w{};
  size_t off = row_chunk_bytes(E, rows_max, kI16Rows);
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? static_cast<char*>(base) + off : nullptr;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return p;
  };
  w.q = static_cast<int16_t*>(take((size_t)rows_max * K * sizeof(int16_t)));
  w.sx = static_cast<float*>(take((size_t)rows_max * sizeof(float)));
  w.total = off;
  return w;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_quantize_rows_int16(const uint16_t* v, int R, int C, int16_t* q, float* scale,
                                       void* stream) {
  moe::Range range_("moe_quantize_rows_int16");
  if (R < 0 || C <= 0) return MOE_ERR_INVALID;
  if (R == 0) return MOE_OK;
  if (!v || !q || !scale || !aligned(v, 2) || !aligned(q, 2) || !aligned(scale, 4))
    return MOE_ERR_INVALID;
  quantize_rows_i16_kernel<<<(R + 7) / 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      v, R, C, nullptr, q, scale);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" size_t moe_int4_linear_int16_workspace_size(int E, int K, int rows_max) {
  if (E <= 0 || K <= 0 || rows_max < 0) return 256;
  return i16_carve(E, K, rows_max, nullptr).total;
}

extern "C" int moe_int4_linear_int16(const uint16_t* x, const int32_t* offsets, int E, int K,
                                     int N, int rows_max, const int32_t* w_packed,
                                     const uint16_t* w_scale, float* out, int32_t* partials,
                                     void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_int4_linear_int16");
  if (E <= 0 || rows_max < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID;
  if (K % kGroup != 0 || K > kI16MaxK || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!x || !offsets || !w_packed || !w_scale || !out || !ws) return MOE_ERR_INVALID;
  if (!aligned(x, 2) || !aligned(w_packed, 4) || !aligned(w_scale, 2) || !aligned(out, 4) ||
      !aligned(partials, 4) || !aligned(ws, 256))
    return MOE_ERR_INVALID;
  if (ws_bytes < moe_int4_linear_int16_workspace_size(E, K, rows_max)) return MOE_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const I16Ws w = i16_carve(E, K, rows_max, ws);
  RowChunks ch{};
  int rc = launch_row_chunks(offsets, E, rows_max, kI16Rows, ws, &ch, status, s);
  if (rc) return rc;
  // the codes of every row below offsets[E]
  quantize_rows_i16_kernel<<<(rows_max + 7) / 8, 256, 0, s>>>(x, rows_max, K, offsets + E, w.q,
                                                              w.sx);
  MOE_LAUNCH_CHECK();
  const int blocks = std::min(ch.max_chunks * ((N + kI16Outs - 1) / kI16Outs), 8 * num_sms());
  linear_i16_kernel<<<blocks, 256, 0, s>>>(w.q, w.sx, ch.chunk_e, ch.chunk_row0, ch.chunk_rows,
                                           ch.n_chunks, K, N, w_packed, w_scale, out, partials);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
