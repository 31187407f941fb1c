// Internal helpers exported by dispatch.cu to the other translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Per-row int8 quantisation of R rows of C bf16 values on stream s; rows at or
// beyond *row_count (device pointer, may be null) are skipped.  With q16 the
// fp16 values of the codes are written too (16-byte aligned, [R, C]).
int launch_quantize_rows(const uint16_t* v, int R, int C, const int32_t* row_count, int8_t* q,
                         float* scale, cudaStream_t s, uint16_t* q16 = nullptr);

// Dispatch whose x_sorted rows are in the expert kernels' pair order (fp16,
// or int8 with act_bits 8); ws as for moe_dispatch.  Arguments are checked by
// the caller.
int launch_dispatch_pairs(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                          int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                          int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                          void* ws, cudaStream_t s);

}  // namespace moe
