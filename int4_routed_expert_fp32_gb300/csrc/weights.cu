// Weight preparation: bf16 weights -> the packed int4 + bf16 scale format the
// expert kernels read.  The "Kimi exact-generator adaptation" page (section
// "The proposed substitution") names the conversion, ExactLinear.from_weight
// with a four-bit choice and group size 32, but not its rounding.  Reading,
// per row and 32-column group, in IEEE float32: a = max|w|; s = bf16(a / 7)
// (the division rounded to nearest, then rounded to bf16, ties to even);
// q = clamp(rint(w / s), -8, 7) with the stored s and ties to even; s = 0
// gives q = 0.  Nibble j of packed word i is column 8 i + j, two's complement.
// The eight-bit choice reads the same way with 127 in place of 7 and the
// codes stored one per byte: since |w| / s <= 127 (1 + 2^-9) < 127.5, the
// codes lie in [-127, 127].
#include "common.cuh"

namespace moe {

// One thread per (row, group): 64 bytes of bf16 in, 16 bytes of packed int4
// and one bf16 scale out.  A non-finite weight records MOE_ERR_UNSUPPORTED.
__global__ void __launch_bounds__(256) quantize_int4_kernel(const uint16_t* __restrict__ w, int N,
                                                            int K, int32_t* __restrict__ packed,
                                                            uint16_t* __restrict__ scale,
                                                            int* status) {
  const int G = K / kGroup;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(N) * G) return;
  const int n = static_cast<int>(idx / G), g = static_cast<int>(idx - static_cast<long long>(n) * G);
  const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)n * K + (size_t)g * kGroup);
  float f[kGroup];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = src[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
    }
  }
  float a = 0.0f;
  bool fin = true;
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    fin &= fabsf(f[i]) <= 3.4028235e38f;
    a = fmaxf(a, fabsf(f[i]));
  }
  if (!fin) {
    record_status(status, MOE_ERR_UNSUPPORTED);
    a = 0.0f;
  }
  const uint16_t sb = f32_to_bf16_bits(__fdiv_rn(a, 7.0f));
  const float s = __uint_as_float(static_cast<uint32_t>(sb) << 16);
  uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    int q = 0;
    if (s > 0.0f) q = min(max(__float2int_rn(__fdiv_rn(f[i], s)), -8), 7);
    word[i >> 3] |= (static_cast<uint32_t>(q) & 0xFu) << (4 * (i & 7));
  }
  *reinterpret_cast<uint4*>(packed + (size_t)n * (K / 8) + (size_t)g * 4) =
      make_uint4(word[0], word[1], word[2], word[3]);
  scale[(size_t)n * G + g] = sb;
}

// One thread per (row, group): 64 bytes of bf16 in, 32 int8 codes and one
// bf16 scale out.  A non-finite weight records MOE_ERR_UNSUPPORTED.
__global__ void __launch_bounds__(256) quantize_int8_kernel(const uint16_t* __restrict__ w, int N,
                                                            int K, int8_t* __restrict__ q8,
                                                            uint16_t* __restrict__ scale,
                                                            int* status) {
  const int G = K / kGroup;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(N) * G) return;
  const int n = static_cast<int>(idx / G), g = static_cast<int>(idx - static_cast<long long>(n) * G);
  const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)n * K + (size_t)g * kGroup);
  float f[kGroup];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = src[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
    }
  }
  float a = 0.0f;
  bool fin = true;
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    fin &= fabsf(f[i]) <= 3.4028235e38f;
    a = fmaxf(a, fabsf(f[i]));
  }
  if (!fin) {
    record_status(status, MOE_ERR_UNSUPPORTED);
    a = 0.0f;
  }
  const uint16_t sb = f32_to_bf16_bits(__fdiv_rn(a, 127.0f));
  const float s = __uint_as_float(static_cast<uint32_t>(sb) << 16);
  uint32_t word[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    int q = 0;
    if (s > 0.0f) q = min(max(__float2int_rn(__fdiv_rn(f[i], s)), -127), 127);
    word[i >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i & 3));
  }
  uint4* dst = reinterpret_cast<uint4*>(q8 + (size_t)n * K + (size_t)g * kGroup);
  dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
  dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
  scale[(size_t)n * G + g] = sb;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_quantize_int4(const uint16_t* w, int N, int K, int32_t* packed,
                                 uint16_t* scale, void* stream) {
  moe::Range range_("moe_quantize_int4");
  if (N < 0 || K <= 0) return MOE_ERR_INVALID;
  if (K % kGroup != 0) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!w || !packed || !scale || !aligned(w, 16) || !aligned(packed, 16) || !aligned(scale, 2))
    return MOE_ERR_INVALID;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const long long total = static_cast<long long>(N) * (K / kGroup);
  const long long blocks = (total + 255) / 256;
  if (blocks > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  quantize_int4_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      w, N, K, packed, scale, status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_quantize_int8(const uint16_t* w, int N, int K, int8_t* q, uint16_t* scale,
                                 void* stream) {
  moe::Range range_("moe_quantize_int8");
  if (N < 0 || K <= 0) return MOE_ERR_INVALID;
  if (K % kGroup != 0) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!w || !q || !scale || !aligned(w, 16) || !aligned(q, 16) || !aligned(scale, 2))
    return MOE_ERR_INVALID;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const long long total = static_cast<long long>(N) * (K / kGroup);
  const long long blocks = (total + 255) / 256;
  if (blocks > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  quantize_int8_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      w, N, K, q, scale, status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
