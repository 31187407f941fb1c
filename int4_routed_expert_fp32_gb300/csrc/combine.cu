// Un-permute + weighted top-k combine (Kimi K3 latent up-projection page,
// KimiSparseMoeBlock.moe_infer listing: scatter back, cast to the routing
// weights' fp32, multiply, sum over the k slots, cast back; Kimi K2.5
// donor-reference equation "Sum the selected expert outputs with their routing
// weights"), optionally fused with the latent RMSNorm (donor-reference
// equations "RMSNorm mean square ...", "Normalize by the root mean square",
// "Apply learned per-feature RMSNorm gains").
#include <math.h>

#include "combine.cuh"
#include "common.cuh"

namespace moe {

constexpr int kCbThreads = 128;

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = static_cast<uint32_t>(f32_to_bf16_bits(f[2 * i])) |
           (static_cast<uint32_t>(f32_to_bf16_bits(f[2 * i + 1])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float tot = 0.f;
  if (threadIdx.x < 32) {
    tot = lane < (blockDim.x >> 5) ? red[lane] : 0.f;
    tot = warp_sum(tot);
    if (lane == 0) red[0] = tot;
  }
  __syncthreads();
  tot = red[0];
  __syncthreads();
  return tot;
}

__device__ __forceinline__ void load8(const uint16_t* y, size_t row, int nv, int v, float (&f)[8]) {
  unpack8(reinterpret_cast<const uint4*>(y)[row * nv + v], f);
}

__device__ __forceinline__ void load8(const float* y, size_t row, int nv, int v, float (&f)[8]) {
  const float4* p = reinterpret_cast<const float4*>(y) + (row * nv + v) * 2;
  const float4 a = p[0], b = p[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// CTA (t, y) combines the 16-byte column vectors y, y + gridDim.y, ... of
// token t (gridDim.y > 1 spreads few tokens over the SMs).  YT: bf16 bits or
// fp32 expert outputs.  NORM (gridDim.y == 1): RMSNorm of the fp32 combined
// row (no intermediate rounding), times the gain.
template <typename YT, bool NORM>
__global__ void __launch_bounds__(kCbThreads) combine_kernel(
    const YT* __restrict__ y, const int32_t* __restrict__ inv_row, const float* __restrict__ w,
    int T, int D, int k, const uint16_t* __restrict__ gain, float eps,
    uint16_t* __restrict__ out, int* status) {
  extern __shared__ float rowbuf[];  // NORM: D floats
  __shared__ int32_t rows[kMaxTopK];
  __shared__ float wts[kMaxTopK];
  __shared__ float red[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    // y holds T * k rows: a row index outside them is skipped and recorded
    int r = inv_row[(size_t)t * k + threadIdx.x];
    if (r < 0 || r >= T * k) {
      record_status(status, MOE_ERR_INVALID);
      r = -1;
    }
    rows[threadIdx.x] = r;
    wts[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int nv = D / 8;
  uint4* ov = reinterpret_cast<uint4*>(out + (size_t)t * D);
  float ss = 0.f;
  for (int v = blockIdx.y * kCbThreads + threadIdx.x; v < nv; v += kCbThreads * gridDim.y) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      float f[8];
      load8(y, static_cast<size_t>(r), nv, v, f);
      const float wj = wts[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(f[i], wj, acc[i]);
    }
    if (!NORM) {
      ov[v] = pack8(acc);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        rowbuf[8 * v + i] = acc[i];
        ss = fmaf(acc[i], acc[i], ss);
      }
    }
  }
  if (NORM) {
    const float tot = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(D) + eps);
    for (int v = threadIdx.x; v < nv; v += kCbThreads) {
      float f[8];
      const uint4 gv = reinterpret_cast<const uint4*>(gain)[v];
      float gf[8];
      unpack8(gv, gf);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = rowbuf[8 * v + i] * inv * gf[i];
      ov[v] = pack8(f);
    }
  }
}

__global__ void __launch_bounds__(kCbThreads) rmsnorm_kernel(const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ gain,
                                                             int D, float eps,
                                                             uint16_t* __restrict__ out) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int nv = D / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x + (size_t)r * D);
  float ss = 0.f;
  for (int v = threadIdx.x; v < nv; v += kCbThreads) {
    float f[8];
    unpack8(xv[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  const float tot = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(D) + eps);
  uint4* ov = reinterpret_cast<uint4*>(out + (size_t)r * D);
  for (int v = threadIdx.x; v < nv; v += kCbThreads) {
    float f[8], gf[8];
    unpack8(xv[v], f);
    unpack8(reinterpret_cast<const uint4*>(gain)[v], gf);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * inv * gf[i];
    ov[v] = pack8(f);
  }
}

template <typename YT>
static int launch_combine_t(const YT* y, const int32_t* inv_row, const float* w, int T, int D,
                            int k, const uint16_t* gain, float eps, uint16_t* out, cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  if (gain) {
    const size_t smem = (size_t)D * sizeof(float);
    if (smem > 48 * 1024)
      MOE_TRY_CUDA(cudaFuncSetAttribute(combine_kernel<YT, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    combine_kernel<YT, true><<<T, kCbThreads, smem, s>>>(y, inv_row, w, T, D, k, gain, eps, out,
                                                         status);
  } else {
    // few tokens: split each row over CTAs so that about 4 CTAs per SM run
    const int nv = D / 8;
    const int max_split = (nv + kCbThreads - 1) / kCbThreads;
    const int want = (4 * num_sms() + T - 1) / T;
    const dim3 grid(T, want < 1 ? 1 : (want > max_split ? max_split : want));
    combine_kernel<YT, false><<<grid, kCbThreads, 0, s>>>(y, inv_row, w, T, D, k, nullptr, eps,
                                                           out, status);
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_combine(const void* y, bool y_f32, const int32_t* inv_row, const float* w, int T, int D,
                   int k, const uint16_t* gain, float eps, uint16_t* out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  if (y_f32)
    return launch_combine_t(static_cast<const float*>(y), inv_row, w, T, D, k, gain, eps, out, s);
  return launch_combine_t(static_cast<const uint16_t*>(y), inv_row, w, T, D, k, gain, eps, out, s);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine(const uint16_t* y_sorted, const int32_t* inv_row, const float* topk_w,
                           int T, int D, int k, uint16_t* out, void* stream) {
  moe::Range range_("moe_combine");
  if (T < 0 || D <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (D % 64 != 0 || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_sorted || !inv_row || !topk_w || !out) return MOE_ERR_INVALID;
  if (!aligned(y_sorted, 16) || !aligned(out, 16)) return MOE_ERR_INVALID;
  return launch_combine(y_sorted, false, inv_row, topk_w, T, D, k, nullptr, 0.f, out,
                        static_cast<cudaStream_t>(stream));
}

extern "C" int moe_rmsnorm(const uint16_t* x, const uint16_t* gain, int M, int N, float eps,
                           uint16_t* y, void* stream) {
  moe::Range range_("moe_rmsnorm");
  if (M < 0 || N <= 0 || !(eps >= 0.f)) return MOE_ERR_INVALID;
  if (N % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (!x || !gain || !y || !aligned(x, 16) || !aligned(gain, 16) || !aligned(y, 16))
    return MOE_ERR_INVALID;
  rmsnorm_kernel<<<M, kCbThreads, 0, static_cast<cudaStream_t>(stream)>>>(x, gain, N, eps, y);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
