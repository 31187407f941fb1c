// tcgen05 grouped W4A16 expert GEMMs (ffn_tc.cu), used for the experts with
// many rows.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

struct TxParams {
  const uint16_t* scale0;  // bf16 [E, N, K/32] (gate, or the single matrix)
  const uint16_t* scale1;  // bf16 [E, N, K/32] (up)
  const float* x_scale;    // act_bits 8: row scales of the int8 rows
  void* out;               // fp16 h (bf16 h in act_bits 8) / bf16 y / fp32 y  [rows_max, N]
  int32_t* partials;       // act_bits 8, tests only: int32 [rows_max, N, K/32] or null
  const int32_t* chunk_e;
  const int32_t* chunk_row0;
  const int32_t* chunk_rows;
  const int32_t* n_chunks;
  int* status;
  long long wait_ns;
  int K;
  int N;
  int stall_at;            // tests only (STALL instantiation): the producer stops at this stage
};

struct TxMaps {
  CUtensorMap a;   // activations fp16 [rows_max, K], 128 x 64 box, 128-byte swizzle
  CUtensorMap q0;  // packed weights [E, N, K/8], box 16 words x rows, 64-byte swizzle
  CUtensorMap q1;
};

// Rows per token tile of the tensor-core path (chunks of that many rows), and
// of its small-tile layout for experts of at most kTcSmallChunkRows rows.
constexpr int kTcChunkRows = 128;
constexpr int kTcSmallChunkRows = 64;

// Rows per token tile of the CTA-pair kernels (ffn_tc2.cu).
constexpr int kTcPairChunkRows = 256;

// K of the tensor-core path must be a multiple of 64.
bool tc_path_supported(int K);

// Pair-ordered copy (see pair_pos) of natural-order rows [R, C] below
// *row_count: bf16 -> fp16 (src_i8 false; a value beyond the fp16 range
// records MOE_ERR_UNSUPPORTED), or int8 -> int8 (src_i8 true).
int launch_to_pair_rows(const void* src, bool src_i8, int R, int C, const int32_t* row_count,
                        void* dst, int* status, cudaStream_t s);

// fp16 copy of bf16 (src_i8 false) or int8 (src_i8 true) rows [R, C] below
// *row_count (order kept).
int launch_to_f16_rows(const void* src, bool src_i8, int R, int C, const int32_t* row_count,
                       uint16_t* dst, cudaStream_t s);

// h[rows] = SiLU(x W_gate^T) * (x W_up^T) for the listed 128-row chunks
// (act_bits 16); x16 is the fp16 copy of the activations (pair order), h is
// written in fp16, pair order.
// small: chunks of at most kTcSmallChunkRows rows (64-row token tiles, a
// deeper ring; ffn_tc.cu).
int launch_tc_gateup(const uint16_t* x16, int rows_max, int E, int D, int I,
                     const int32_t* gate_packed, const uint16_t* gate_scale,
                     const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                     const int32_t* chunk_e, const int32_t* chunk_row0,
                     const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                     cudaStream_t s, bool small = false);

// act_bits 8 on the tensor cores (ffn_tc_q8.cu): exact int4 x int8 group
// partials, y = sc_x * (fp32 chain of fma(s_w[g], P[g], .) in group order).
// x16 / h16: fp16 copies of the int8 rows.  Gate/up stores h in bf16 (pair
// order) for its re-quantisation.  partials (tests only, down / linear): also
// store every P as int32 [rows_max, N, K/32] (then y is fp32).
int launch_tc_q8_gateup(const uint16_t* x16, const float* x_scale, int rows_max, int E, int D,
                        int I, const int32_t* gate_packed, const uint16_t* gate_scale,
                        const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                        const int32_t* chunk_e, const int32_t* chunk_row0,
                        const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                        cudaStream_t s);
int launch_tc_q8_down(const uint16_t* h16, const float* h_scale, int rows_max, int E, int D, int I,
                      const int32_t* down_packed, const uint16_t* down_scale, void* y, bool y_f32,
                      const int32_t* chunk_e, const int32_t* chunk_row0,
                      const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                      cudaStream_t s, int32_t* partials);

// y[rows] = h16 W_down^T for the listed chunks (act_bits 16); bf16 y, or fp32
// with y_f32.
// Tests only: launch_tc_down's linear (fp32 y) or, with h_scale set, the
// exact kernel's linear, with the producer of every CTA stopping before its
// stage stall_at and every wait limited to wait_ns (the kernels' exit paths).
int launch_tc_linear_stalled(const uint16_t* x16, const float* x_scale, int rows_max, int E, int N,
                             int K, const int32_t* w_packed, const uint16_t* w_scale, float* y,
                             const int32_t* chunk_e, const int32_t* chunk_row0,
                             const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                             long long wait_ns, int stall_at, cudaStream_t s, bool small = false);

int launch_tc_down(const uint16_t* h16, int rows_max, int E, int D, int I,
                   const int32_t* down_packed, const uint16_t* down_scale, void* y, bool y_f32,
                   const int32_t* chunk_e, const int32_t* chunk_row0, const int32_t* chunk_rows,
                   const int32_t* n_chunks, int* status, cudaStream_t s, bool small = false);

// The same two GEMMs (act_bits 16) on CTA pairs (ffn_tc2.cu): chunks of at
// most kTcPairChunkRows rows, MMAs of 256 weight rows over two SMs.
// Returns MOE_ERR_UNSUPPORTED when no cluster of two fits on the device.
bool tc_pair_available();
// Tests only: launch_tc_linear_stalled's act_bits 16 linear on the CTA-pair
// kernel.
int launch_tc_pair_linear_stalled(const uint16_t* x16, int rows_max, int E, int N, int K,
                                  const int32_t* w_packed, const uint16_t* w_scale, float* y,
                                  const int32_t* chunk_e, const int32_t* chunk_row0,
                                  const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                                  long long wait_ns, int stall_at, cudaStream_t s);
int launch_tc_pair_gateup(const uint16_t* x16, int rows_max, int E, int D, int I,
                          const int32_t* gate_packed, const uint16_t* gate_scale,
                          const int32_t* up_packed, const uint16_t* up_scale, uint16_t* h,
                          const int32_t* chunk_e, const int32_t* chunk_row0,
                          const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                          cudaStream_t s);
int launch_tc_pair_down(const uint16_t* h16, int rows_max, int E, int D, int I,
                        const int32_t* down_packed, const uint16_t* down_scale, void* y,
                        bool y_f32, const int32_t* chunk_e, const int32_t* chunk_row0,
                        const int32_t* chunk_rows, const int32_t* n_chunks, int* status,
                        cudaStream_t s);

}  // namespace moe
