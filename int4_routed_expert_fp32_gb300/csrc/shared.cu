// The always-active shared expert: out += down( SiLU(gate(x)) * up(x) ) with
// bf16 weights on the full-width input ("Kimi K3 latent up-projection" page,
// KimiSparseMoeBlock listing: shared_experts = KimiMLP of
// moe_intermediate_size * num_shared_experts features, y = y +
// shared_experts(identity); "Kimi K2.5 donor reference" page, "Add an
// always-active shared expert"; the exact-generator page keeps shared experts
// as ordinary bf16 linear modules).
//
// Two tcgen05 GEMM launches (gate and up together, then down) with fp32
// split-K partials (the split fills the SMs when T is small), one kernel
// that sums the gate/up partials and stores
// h = bf16(SiLU(g) * u) (the module's dtype), and one that adds the summed
// down partials to the bf16 output with a single rounding.
#include <math.h>

#include "combine.cuh"
#include "common.cuh"

namespace moe {

namespace {

// K slice (a multiple of 64) so that tiles x slices reaches ~ one CTA per SM.
int split_kc(int M, int N, int K) {
  const int tiles = ((N + 255) / 256) * ((M + 127) / 128);
  int splits = (num_sms() + tiles - 1) / tiles;
  const int max_splits = (K + 63) / 64;
  if (splits < 1) splits = 1;
  if (splits > max_splits) splits = max_splits;
  const int per = (K + splits - 1) / splits;
  return (per + 63) / 64 * 64;
}

int n_splits(int K, int kc) { return (K + kc - 1) / kc; }

struct SharedWs {
  float* g;     // [T, sg * I]
  float* u;     // [T, sg * I]
  uint16_t* h;  // [T, I]
  float* s;     // [T, sd * H]
  int kc_gu, sg, kc_d, sd;
  size_t total;
};

SharedWs shared_carve(int T, int H, int I, void* base) {
  SharedWs w{};
  w.kc_gu = split_kc(T, 2 * I, H);  // gate and up share one launch
  w.sg = n_splits(H, w.kc_gu);
  w.kc_d = split_kc(T, H, I);
  w.sd = n_splits(I, w.kc_d);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? static_cast<char*>(base) + off : nullptr;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return p;
  };
  w.g = static_cast<float*>(take((size_t)T * w.sg * I * 4));
  w.u = static_cast<float*>(take((size_t)T * w.sg * I * 4));
  w.h = static_cast<uint16_t*>(take((size_t)T * I * 2));
  w.s = static_cast<float*>(take((size_t)T * w.sd * H * 4));
  w.total = off;
  return w;
}

}  // namespace

// h[t, i] = bf16( SiLU(sum_z g[t, z*I + i]) * sum_z u[t, z*I + i] ), 4 outputs
// per thread.
__global__ void __launch_bounds__(256) shared_silu_mul_kernel(const float* __restrict__ g,
                                                              const float* __restrict__ u,
                                                              int splits, int T, int I,
                                                              uint16_t* __restrict__ h) {
  const long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int per_row = I / 4;
  if (q >= static_cast<long long>(T) * per_row) return;
  const int t = static_cast<int>(q / per_row), i = static_cast<int>(q - (long long)t * per_row) * 4;
  float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
  for (int z = 0; z < splits; ++z) {
    const size_t o = ((size_t)t * splits + z) * I + i;
    const float4 a = *reinterpret_cast<const float4*>(g + o);
    const float4 b = *reinterpret_cast<const float4*>(u + o);
    gs.x += a.x; gs.y += a.y; gs.z += a.z; gs.w += a.w;
    us.x += b.x; us.y += b.y; us.z += b.z; us.w += b.w;
  }
  const float gv[4] = {gs.x, gs.y, gs.z, gs.w}, uv[4] = {us.x, us.y, us.z, us.w};
  uint32_t packed[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float h0 = gv[2 * j] / (1.0f + expf(-gv[2 * j])) * uv[2 * j];
    const float h1 = gv[2 * j + 1] / (1.0f + expf(-gv[2 * j + 1])) * uv[2 * j + 1];
    packed[j] = static_cast<uint32_t>(f32_to_bf16_bits(h0)) |
                (static_cast<uint32_t>(f32_to_bf16_bits(h1)) << 16);
  }
  *reinterpret_cast<uint2*>(h + (size_t)t * I + i) = make_uint2(packed[0], packed[1]);
}

// out[t, n] = bf16( (accumulate ? out[t, n] : 0) + sum_z s[t, z*H + n] ), 4
// outputs per thread.
__global__ void __launch_bounds__(256) shared_add_kernel(const float* __restrict__ s, int splits,
                                                         int T, int H, int accumulate,
                                                         uint16_t* __restrict__ out) {
  const long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int per_row = H / 4;
  if (q >= static_cast<long long>(T) * per_row) return;
  const int t = static_cast<int>(q / per_row), n = static_cast<int>(q - (long long)t * per_row) * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  uint2* o = reinterpret_cast<uint2*>(out + (size_t)t * H + n);
  if (accumulate) {
    const uint2 v = *o;
    acc[0] = __uint_as_float(v.x << 16);
    acc[1] = __uint_as_float(v.x & 0xffff0000u);
    acc[2] = __uint_as_float(v.y << 16);
    acc[3] = __uint_as_float(v.y & 0xffff0000u);
  }
  for (int z = 0; z < splits; ++z) {
    const float4 a = *reinterpret_cast<const float4*>(s + ((size_t)t * splits + z) * H + n);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
  }
  *o = make_uint2(static_cast<uint32_t>(f32_to_bf16_bits(acc[0])) |
                      (static_cast<uint32_t>(f32_to_bf16_bits(acc[1])) << 16),
                  static_cast<uint32_t>(f32_to_bf16_bits(acc[2])) |
                      (static_cast<uint32_t>(f32_to_bf16_bits(acc[3])) << 16));
}

size_t shared_expert_ws_bytes(int T, int H, int I) {
  if (T <= 0) return 256;
  return shared_carve(T, H, I, nullptr).total;
}

int launch_shared_expert(const uint16_t* x, int T, int H, int I, const uint16_t* gate_w,
                         const uint16_t* up_w, const uint16_t* down_w, int accumulate,
                         uint16_t* out, void* ws, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const SharedWs w = shared_carve(T, H, I, ws);
  // gate and up in one launch
  int rc = launch_linear_tc_f32_splitk(x, gate_w, T, I, H, w.kc_gu, w.g, s, up_w, w.u);
  if (rc) return rc;
  const long long n1 = (long long)T * (I / 4);
  shared_silu_mul_kernel<<<static_cast<unsigned>((n1 + 255) / 256), 256, 0, s>>>(w.g, w.u, w.sg, T,
                                                                                 I, w.h);
  MOE_LAUNCH_CHECK();
  rc = launch_linear_tc_f32_splitk(w.h, down_w, T, H, I, w.kc_d, w.s, s);
  if (rc) return rc;
  const long long n2 = (long long)T * (H / 4);
  shared_add_kernel<<<static_cast<unsigned>((n2 + 255) / 256), 256, 0, s>>>(w.s, w.sd, T, H,
                                                                           accumulate, out);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_shared_expert_workspace_size(int T, int H, int I) {
  if (T < 0 || H <= 0 || I <= 0) return 256;
  return shared_expert_ws_bytes(T, H, I);
}

extern "C" int moe_shared_expert(const uint16_t* x, int T, int H, int I, const uint16_t* gate_w,
                                 const uint16_t* up_w, const uint16_t* down_w, int accumulate,
                                 uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_shared_expert");
  if (T < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID;
  if (H % 64 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !gate_w || !up_w || !down_w || !out || !ws) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(gate_w, 16) || !aligned(up_w, 16) || !aligned(down_w, 16) ||
      !aligned(out, 16) || !aligned(ws, 256))
    return MOE_ERR_INVALID;
  if (ws_bytes < shared_expert_ws_bytes(T, H, I)) return MOE_ERR_WORKSPACE;
  return launch_shared_expert(x, T, H, I, gate_w, up_w, down_w, accumulate, out, ws,
                              static_cast<cudaStream_t>(stream));
}
