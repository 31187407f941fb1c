// Internal launchers shared between translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// out[t] = bf16(sum_j y[inv_row[t,j]] * w[t,j]); with a gain, the rounded row
// then goes through RMSNorm(eps) * gain.
int launch_combine(const uint16_t* y, const int32_t* inv_row, const float* w, int T, int D, int k,
                   const uint16_t* gain, float eps, uint16_t* out, cudaStream_t s);

// y[M, N] = x[M, K] w[N, K]^T in bf16 with fp32 accumulation.
int launch_linear_bf16(const uint16_t* x, const uint16_t* w, int M, int N, int K, uint16_t* y,
                       cudaStream_t s);

}  // namespace moe
