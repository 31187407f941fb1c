// Internal helpers exported by dispatch.cu to the other translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Per-row int8 quantisation of R rows of C bf16 values on stream s; rows at or
// beyond *row_count (device pointer, may be null) are skipped.
int launch_quantize_rows(const uint16_t* v, int R, int C, const int32_t* row_count, int8_t* q,
                         float* scale, cudaStream_t s);

}  // namespace moe
