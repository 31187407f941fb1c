// Internal launchers shared between translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// out[t] = bf16(sum_j y[inv_row[t,j]] * w[t,j]) with y bf16 (y_f32 false) or
// fp32; with a gain, the fp32 combined row goes through RMSNorm(eps) * gain
// before the single rounding to bf16.
int launch_combine(const void* y, bool y_f32, const int32_t* inv_row, const float* w, int T, int D,
                   int k, const uint16_t* gain, float eps, uint16_t* out, cudaStream_t s);

// Gated expert MLP over expert-sorted rows (validated arguments); y is bf16
// [rows_max, D] or, with y_f32, fp32.  No expert has more than
// max_rows_per_expert rows (the token count when called from the layer).
// Every expert's rows (offsets) cut into chunks of at most mc rows, on the
// device (no host sync): the lists are carved from ws (row_chunk_bytes).
struct RowChunks {
  int32_t* chunk_e;
  int32_t* chunk_row0;
  int32_t* chunk_rows;
  int32_t* n_chunks;
  int max_chunks;
};
size_t row_chunk_bytes(int E, int rows_max, int mc);
int launch_row_chunks(const int32_t* offsets, int E, int rows_max, int mc, void* ws,
                      RowChunks* chunks, int* status, cudaStream_t s);

// Workspace bytes of launch_expert_ffn.
size_t expert_ffn_ws_bytes(int E, int D, int I, int rows_max, int act_bits);

// Expert FFN over expert-sorted rows x_sorted in pair order (fp16, or int8
// with act_bits 8; see pair_pos), y in natural column order.
int launch_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets, int E,
                      int D, int I, int rows_max, int max_rows_per_expert,
                      const int32_t* gate_packed,
                      const uint16_t* gate_scale, const int32_t* up_packed,
                      const uint16_t* up_scale, const int32_t* down_packed,
                      const uint16_t* down_scale, int act_bits, void* y, bool y_f32, void* ws,
                      cudaStream_t s);

// Split-K partials of x[M, K] w[N, K]^T (bf16 operands, tcgen05, fp32
// accumulation over each slice of kc columns, kc a multiple of 64):
// y[m, z * N + n] = sum over k in [z * kc, (z + 1) * kc) of x[m, k] w[n, k],
// z = 0 .. ceil(K / kc) - 1.  With w2 (same shape) also y2 from x w2^T, in
// the same launch.
int launch_linear_tc_f32_splitk(const uint16_t* x, const uint16_t* w, int M, int N, int K, int kc,
                                float* y, cudaStream_t s, const uint16_t* w2 = nullptr,
                                float* y2 = nullptr);

// y = x (W_0 + ... + W_{terms-1})^T with fp32 out, split-K partials as
// launch_linear_tc_f32_splitk; w is [terms][N][K] bf16.
int launch_linear_tc_f32_terms(const uint16_t* x, const uint16_t* w, int terms, int M, int N, int K,
                               int kc, float* y, cudaStream_t s);

// moe_route with, from 512 tokens, the three bf16 terms of the router weight
// (bf16 [3, E, H] from moe_router_prepare) read from w_terms instead of
// split into the workspace on every call (w_terms NULL: split them now).
int route_with_terms(const uint16_t* x, const float* w_router, const uint16_t* w_terms,
                     const float* bias, int T, int H, int E, int k, int renorm, int32_t* topk_idx,
                     float* topk_w, void* ws, size_t ws_bytes, cudaStream_t s);

// y[M, N] = x[M, K] w[N, K]^T in bf16 with fp32 accumulation.
int launch_linear_bf16(const uint16_t* x, const uint16_t* w, int M, int N, int K, uint16_t* y,
                       cudaStream_t s);

// Shared expert (validated arguments): out = bf16((accumulate ? out : 0) +
// down(SiLU(gate x) * up x)), bf16 weights gate/up [I, H], down [H, I].
size_t shared_expert_ws_bytes(int T, int H, int I);
int launch_shared_expert(const uint16_t* x, int T, int H, int I, const uint16_t* gate_w,
                         const uint16_t* up_w, const uint16_t* down_w, int accumulate,
                         uint16_t* out, void* ws, cudaStream_t s);

}  // namespace moe
