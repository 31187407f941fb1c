// Router: fp32 logits of the bf16 tokens against the fp32 router weight,
// sigmoid affinities, correction bias for ranking, warp-level top-k and
// renormalisation (Kimi K2.5 donor-reference page, equations
// "MoEGate.forward: logits", "Independent sigmoid scores for the router",
// "Bias the choice of experts while retaining original affinities",
// "MoEGate.forward: topk weight" and "Normalize the selected routing
// affinities").  One expert group: group-limited masking is the identity.
// Few tokens: split-K fp32 SIMT logits (the weight read dominates); up to 32
// tokens one lane per token.  Many tokens: the fp32 weight is split exactly
// into three bf16 terms and the logits come from tcgen05 GEMMs with fp32
// accumulation.
#include <math.h>

#include <algorithm>

#include "combine.cuh"
#include "common.cuh"

namespace moe {

constexpr int kRtTokens = 64;   // tokens per logits tile
constexpr int kRtExperts = 64;  // experts per logits tile
constexpr int kRtK = 32;        // K step staged in shared memory
constexpr int kRtTargetCtas = 304;

struct RouterSplit {
  int splits;  // K slices
  int kslice;  // elements per slice (multiple of kRtK)
};

// K is split so that small token counts still spread the weight read over
// about two CTAs per SM; the partial sums are reduced in a fixed order.
static RouterSplit router_split(int T, int H, int E) {
  const int tiles = ((T + kRtTokens - 1) / kRtTokens) * ((E + kRtExperts - 1) / kRtExperts);
  int s = (kRtTargetCtas + tiles - 1) / tiles;
  const int max_s = H / kRtK;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  int kslice = ((H + s - 1) / s + kRtK - 1) / kRtK * kRtK;
  RouterSplit r;
  r.kslice = kslice;
  r.splits = (H + kslice - 1) / kslice;
  return r;
}

// part[z, t, e] = sum over the z-th K slice of x[t, k] * W[e, k] (fp32 FMA).
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ W, int T,
                                                            int H, int E, int kslice,
                                                            float* __restrict__ part) {
  __shared__ float xs[kRtK][kRtTokens + 1];
  __shared__ float wsm[kRtK][kRtExperts + 1];
  const int t0 = blockIdx.x * kRtTokens;
  const int e0 = blockIdx.y * kRtExperts;
  const int kb = blockIdx.z * kslice;
  const int ke = min(H, kb + kslice);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = kb; k0 < ke; k0 += kRtK) {
    for (int i = tid; i < kRtTokens * kRtK; i += 256) {
      const int r = i / kRtK, c = i % kRtK;
      const int t = t0 + r, kk = k0 + c;
      xs[c][r] = (t < T && kk < ke) ? bf16_bits_to_f32(x[(size_t)t * H + kk]) : 0.f;
    }
    for (int i = tid; i < kRtExperts * kRtK; i += 256) {
      const int r = i / kRtK, c = i % kRtK;
      const int e = e0 + r, kk = k0 + c;
      wsm[c][r] = (e < E && kk < ke) ? W[(size_t)e * H + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kRtK; ++c) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = xs[c][ty * 4 + i];
        b[i] = wsm[c][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) part[((size_t)blockIdx.z * T + t) * E + e] = acc[i][j];
    }
  }
}

// Decode-sized batches (T <= 32): one lane per token.  A CTA of eight warps
// takes 32 experts x 256 columns (336 CTAs at H = 7168, E = 384: four fit on
// an SM, so the whole weight is in flight at once): the fp32 weight tile and the tokens' bf16
// x slice are copied to shared memory up front (16-byte cp.async, all in
// flight at once; x rows padded by 16 bytes so that the lanes' 16-byte reads
// of 32 different rows hit distinct banks), then each lane accumulates its
// token against the four experts of its warp, the weights read as
// shared-memory broadcasts (one 16-byte read per four FMAs).
// part[z, t, e] = the z-th 256-column slice's dot product, in column order.
constexpr int kRwExperts = 32;               // experts per CTA (4 per warp)
constexpr int kRwK = 256;                    // K columns per CTA
constexpr int kRwMaxTokens = 32;             // one lane per token
constexpr int kRwXStride = kRwK * 2 + 16;    // bytes per x row in shared memory
constexpr int kRwSmem = kRwExperts * kRwK * 4 + kRwMaxTokens * kRwXStride;  // 48.5 KiB

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__global__ void __launch_bounds__(256) router_logits_warp_kernel(const uint16_t* __restrict__ x,
                                                                 const float* __restrict__ W,
                                                                 int T, int H, int E,
                                                                 float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t rsm[];
  float* wsm = reinterpret_cast<float*>(rsm);              // [kRwExperts][kRwK]
  uint8_t* xsm = rsm + kRwExperts * kRwK * 4;              // [kRwMaxTokens][kRwXStride]
  const int e0 = blockIdx.x * kRwExperts;
  const int k0 = blockIdx.y * kRwK;
  const int kn = min(kRwK, H - k0);  // multiple of 64 (H % 64 == 0)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // weight tile (rows of experts beyond E are zeros) and x slice (rows of
  // tokens beyond T are never read)
  for (int i = threadIdx.x; i < kRwExperts * (kRwK / 4); i += 256) {
    const int r = i / (kRwK / 4), c4 = i % (kRwK / 4);
    float* dst = wsm + r * kRwK + 4 * c4;
    if (e0 + r < E && 4 * c4 < kn)
      cp_async_16(dst, W + (size_t)(e0 + r) * H + k0 + 4 * c4);
    else
      *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = threadIdx.x; i < T * (kRwK / 8); i += 256) {
    const int t = i / (kRwK / 8), c8 = i % (kRwK / 8);
    if (8 * c8 < kn) cp_async_16(xsm + t * kRwXStride + 16 * c8, x + (size_t)t * H + k0 + 8 * c8);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int t = lane;
  if (t >= T) return;  // no barrier follows
  const uint8_t* xr = xsm + t * kRwXStride;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const float* wr = wsm + (warp * 4) * kRwK;
  for (int c0 = 0; c0 < kn; c0 += 32) {
    float xv[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 q = *reinterpret_cast<const uint4*>(xr + 2 * c0 + 16 * v);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[8 * v + 2 * i] = bf16_bits_to_f32(w4[i] & 0xffffu);
        xv[8 * v + 2 * i + 1] = bf16_bits_to_f32(w4[i] >> 16);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4* w4 = reinterpret_cast<const float4*>(wr + j * kRwK + c0);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 wv = w4[v];  // broadcast: every lane reads the same address
        acc[j] = fmaf(xv[4 * v], wv.x, acc[j]);
        acc[j] = fmaf(xv[4 * v + 1], wv.y, acc[j]);
        acc[j] = fmaf(xv[4 * v + 2], wv.z, acc[j]);
        acc[j] = fmaf(xv[4 * v + 3], wv.w, acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = e0 + warp * 4 + j;
    if (e < E) part[((size_t)blockIdx.y * T + t) * E + e] = acc[j];
  }
}

// Tokens from which the router uses the tensor cores.
constexpr int kRtTcMinTokens = 512;
// K columns per tensor-core accumulation (the three weight terms of those
// columns accumulate together); the slices' fp32 partials are added in order
// afterwards.
constexpr int kRtTcKSlice = 1024;

static int router_tc_splits(int H) { return (H + kRtTcKSlice - 1) / kRtTcKSlice; }

// W fp32 [E, H] -> three bf16 terms [3E, H] with W = W1 + W2 + W3 to the last
// bit of the fp32 significand for 2^-110 <= |W| < 3.38e38 and W = 0 (each
// term is the rounded remainder of the previous ones; below 2^-110 the last
// remainder reaches fp32's subnormal range); x (bf16) times each term is
// exact in fp32.
__global__ void router_split_kernel(const float* __restrict__ W, size_t n, uint16_t* __restrict__ Ws) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const float w = W[i];
    const uint16_t b1 = f32_to_bf16_bits(w);
    const float r1 = w - bf16_bits_to_f32(b1);
    const uint16_t b2 = f32_to_bf16_bits(r1);
    const float r2 = r1 - bf16_bits_to_f32(b2);
    Ws[i] = b1;
    Ws[n + i] = b2;
    Ws[2 * n + i] = f32_to_bf16_bits(r2);
  }
}

// One CTA per token.  Its threads reduce the partial logits of the token in
// order (partial p of (t, e) at part[p * sp + t * st + e]; one thread per
// expert at E <= 384, so that all the partial loads are in flight at once),
// then take the sigmoid and add the bias; warp 0 runs k rounds of warp
// arg-max (equal scores: lower expert id) and renormalises.
constexpr int kTopkThreads = 384;

__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(
    const float* __restrict__ part, int S, size_t sp, size_t st, const float* __restrict__ bias,
    int T, int E, int k, int renorm, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  extern __shared__ float sm[];
  __shared__ float sel[kMaxTopK];
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  float* r = sm;
  float* s = sm + E;
  const float* pt = part + (size_t)t * st;
  for (int e = threadIdx.x; e < E; e += kTopkThreads) {
    const float* pe = pt + e;
    float z = 0.f;
    int p = 0;
    for (; p + 8 <= S; p += 8) {  // loads issued together, summed in order
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = pe[(size_t)(p + i) * sp];
#pragma unroll
      for (int i = 0; i < 8; ++i) z += v[i];
    }
    for (; p < S; ++p) z += pe[(size_t)p * sp];
    const float sg = 1.0f / (1.0f + expf(-z));
    float rv = sg + bias[e];
    if (rv != rv) rv = -INFINITY;  // a NaN score never wins
    s[e] = sg;
    r[e] = rv;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bi = E;
    for (int e = lane; e < E; e += 32) {
      const float v = r[e];
      if (v != v) continue;  // already selected
      if (v > best || (v == best && e < bi)) {
        best = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    if (lane == 0) {
      topk_idx[(size_t)t * k + j] = bi;
      sel[j] = s[bi];
      r[bi] = __int_as_float(0x7fc00000);  // mark selected
    }
    __syncwarp();
  }
  if (lane == 0) {
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += sel[j];
    const float den = sum + 1e-20f;
    for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = renorm ? __fdiv_rn(sel[j], den) : sel[j];
  }
}

// The same reduction, scores and selection with one warp per token and the
// token's E <= 32 NPL scores in registers (expert e = lane + 32 i), 8 tokens
// per CTA: every thread works through the k selection rounds, instead of one
// warp of a 384-thread CTA.  Same sums (partials in order), same sigmoid,
// same ties (lower expert id), so the same bits as router_topk_kernel.
constexpr int kTopkWarpTokens = 8;
// Below this many tokens the one-CTA kernel's 384 threads per token keep more
// loads in flight (decode, T = 32: 33 us against 35 us).
constexpr int kTopkWarpMinTokens = 64;

template <int NPL>
__global__ void __launch_bounds__(32 * kTopkWarpTokens) router_topk_warp_kernel(
    const float* __restrict__ part, int S, size_t sp, size_t st, const float* __restrict__ bias,
    int T, int E, int k, int renorm, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarpTokens + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* pt = part + (size_t)t * st;
  float z[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) z[i] = 0.f;
  for (int p = 0; p < S; ++p) {  // each partial's loads issued together, summed in order
    const float* pp = pt + (size_t)p * sp;
    float v[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? pp[e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) z[i] += v[i];
  }
  float sg[NPL], rv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    sg[i] = 1.0f / (1.0f + expf(-z[i]));
    float r = e < E ? sg[i] + bias[e] : -INFINITY;
    if (r != r) r = -INFINITY;  // a NaN score never wins
    rv[i] = r;
  }
  bool taken[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) taken[i] = (lane + 32 * i) >= E;
  float sum = 0.f, selv = 0.f;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bi = E;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {  // ascending expert ids: strict > keeps the lower id
      const int e = lane + 32 * i;
      if (!taken[i] && (rv[i] > best || (rv[i] == best && e < bi))) {
        best = rv[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    // the owner marks it and hands over its sigmoid
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i == bi) {
        taken[i] = true;
        mine = sg[i];
      }
    const float v = __shfl_sync(0xffffffffu, mine, bi & 31);
    if (lane == 0) topk_idx[(size_t)t * k + j] = bi;
    if (lane == j) selv = v;  // lane j keeps selection j (k <= 32)
    sum += v;                 // the same order as the one-warp kernel: j = 0, 1, ...
  }
  if (lane < k) {
    const float den = sum + 1e-20f;
    topk_w[(size_t)t * k + lane] = renorm ? __fdiv_rn(selv, den) : selv;
  }
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_workspace_size(int T, int H, int E) {
  if (T <= 0 || H <= 0 || E <= 0) return 256;
  if (T >= kRtTcMinTokens)  // split weights [3, E, H] bf16 + partials [T, splits, E] fp32
    return align_up((size_t)3 * E * H * sizeof(uint16_t), 256) +
           align_up((size_t)T * router_tc_splits(H) * E * sizeof(float), 256);
  if (T <= kRwMaxTokens)
    return align_up((size_t)((H + kRwK - 1) / kRwK) * T * E * sizeof(float), 256);
  const RouterSplit sp = router_split(T, H, E);
  return align_up((size_t)sp.splits * T * E * sizeof(float), 256);
}

int moe::route_with_terms(const uint16_t* x, const float* w_router, const uint16_t* w_terms,
                          const float* bias, int T, int H, int E, int k, int renorm,
                          int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                          cudaStream_t s) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (H % 64 != 0 || E > kMaxExperts || k > E || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID;
  if (ws_bytes < moe_route_workspace_size(T, H, E)) return MOE_ERR_WORKSPACE;
  if (w_terms && !aligned(w_terms, 16)) return MOE_ERR_INVALID;
  float* part;
  int S;
  size_t sp_stride, st_stride;
  if (T >= kRtTcMinTokens) {
    // tensor cores: partial logits per K slice, the three weight terms
    // accumulated together, [T, splits, E] fp32, summed in slice order
    const uint16_t* Ws = w_terms;
    part = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                    align_up((size_t)3 * E * H * sizeof(uint16_t), 256));
    if (!aligned(x, 16)) return MOE_ERR_INVALID;
    if (!Ws) {  // split the weight now (moe_router_prepare does it once ahead)
      uint16_t* Wt = static_cast<uint16_t*>(ws);
      const size_t n = (size_t)E * H;
      router_split_kernel<<<std::min<size_t>((n + 255) / 256, 4096), 256, 0, s>>>(w_router, n, Wt);
      MOE_LAUNCH_CHECK();
      Ws = Wt;
    }
    const int splits = router_tc_splits(H);
    const int rc = launch_linear_tc_f32_terms(x, Ws, 3, T, E, H, kRtTcKSlice, part, s);
    if (rc) return rc;
    S = splits;
    sp_stride = E;
    st_stride = (size_t)S * E;
  } else if (T <= kRwMaxTokens) {
    if (!aligned(x, 16) || !aligned(w_router, 16)) return MOE_ERR_INVALID;
    part = static_cast<float*>(ws);
    S = (H + kRwK - 1) / kRwK;
    MOE_TRY_CUDA(cudaFuncSetAttribute(router_logits_warp_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kRwSmem));
    dim3 grid((E + kRwExperts - 1) / kRwExperts, S);
    router_logits_warp_kernel<<<grid, 256, kRwSmem, s>>>(x, w_router, T, H, E, part);
    MOE_LAUNCH_CHECK();
    sp_stride = (size_t)T * E;
    st_stride = E;
  } else {
    const RouterSplit spl = router_split(T, H, E);
    part = static_cast<float*>(ws);
    dim3 grid((T + kRtTokens - 1) / kRtTokens, (E + kRtExperts - 1) / kRtExperts, spl.splits);
    router_logits_kernel<<<grid, 256, 0, s>>>(x, w_router, T, H, E, spl.kslice, part);
    MOE_LAUNCH_CHECK();
    S = spl.splits;
    sp_stride = (size_t)T * E;
    st_stride = E;
  }
  if (E <= 512 && T >= kTopkWarpMinTokens) {
    const int grid = (T + kTopkWarpTokens - 1) / kTopkWarpTokens, thr = 32 * kTopkWarpTokens;
    if (E <= 128)
      router_topk_warp_kernel<4><<<grid, thr, 0, s>>>(part, S, sp_stride, st_stride, bias, T, E, k,
                                                      renorm, topk_idx, topk_w);
    else if (E <= 256)
      router_topk_warp_kernel<8><<<grid, thr, 0, s>>>(part, S, sp_stride, st_stride, bias, T, E, k,
                                                      renorm, topk_idx, topk_w);
    else if (E <= 384)
      router_topk_warp_kernel<12><<<grid, thr, 0, s>>>(part, S, sp_stride, st_stride, bias, T, E,
                                                       k, renorm, topk_idx, topk_w);
    else
      router_topk_warp_kernel<16><<<grid, thr, 0, s>>>(part, S, sp_stride, st_stride, bias, T, E,
                                                       k, renorm, topk_idx, topk_w);
  } else {
    const size_t smem = (size_t)2 * E * sizeof(float);  // at most 16 KiB (E <= 2048)
    router_topk_kernel<<<T, kTopkThreads, smem, s>>>(part, S, sp_stride, st_stride, bias, T, E, k,
                                                     renorm, topk_idx, topk_w);
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_route(const uint16_t* x, const float* w_router, const float* bias, int T, int H,
                         int E, int k, int renorm, int32_t* topk_idx, float* topk_w, void* ws,
                         size_t ws_bytes, void* stream) {
  moe::Range range_("moe_route");
  return route_with_terms(x, w_router, nullptr, bias, T, H, E, k, renorm, topk_idx, topk_w, ws,
                          ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_router_prepare(const float* w_router, int E, int H, uint16_t* w_terms,
                                  void* stream) {
  moe::Range range_("moe_router_prepare");
  if (E <= 0 || H <= 0) return MOE_ERR_INVALID;
  if (!w_router || !w_terms || !aligned(w_router, 4) || !aligned(w_terms, 16))
    return MOE_ERR_INVALID;
  const size_t n = (size_t)E * H;
  router_split_kernel<<<std::min<size_t>((n + 255) / 256, 4096), 256, 0,
                        static_cast<cudaStream_t>(stream)>>>(w_router, n, w_terms);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
