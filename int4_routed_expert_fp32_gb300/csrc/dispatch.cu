// Dispatch: per-expert counts, exclusive scan, stable expert-major order and
// the gather of token rows, all on the device (Kimi K3 latent up-projection
// page, KimiSparseMoeBlock.moe_infer listing: one-hot counts, argsort, gather;
// Kimi K2.5 donor-reference equations "DeepSeek MoE.moe_infer: tokens per
// expert" and "... sorted tokens").  The argsort is read as stable: the rows
// of one expert ascend by token id.  In act_bits 8 mode each token row is
// quantised to int8 on the way (per-row symmetric, IEEE fp32 steps).
#include <cuda_fp16.h>
#include <math.h>


#include "common.cuh"
#include "dispatch.cuh"

namespace moe {

constexpr int kChunkTokens = 32;  // tokens per counting chunk (one warp)
constexpr int kCountWarps = 4;

// Per chunk of 32 tokens (one warp, lane = token): the chunk's expert
// histogram hist[c, :] and, for every (t, j), the number of earlier tokens of
// the chunk that chose the same expert (its rank inside the chunk).  A token
// lists an expert at most once, so each expert keeps a 32-bit mask of the
// chunk's tokens that chose it: count = popc(mask), rank = popc(mask & lower
// lanes).
__global__ void __launch_bounds__(kCountWarps * 32) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, int32_t* __restrict__ hist,
    int32_t* __restrict__ local_rank, int* status) {
  extern __shared__ uint32_t smc[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kCountWarps + warp;
  if (c * kChunkTokens >= T) return;
  uint32_t* mask = smc + warp * (E + kChunkTokens * kMaxTopK);
  int32_t* ids = reinterpret_cast<int32_t*>(mask + E) + lane * k;
  for (int e = lane; e < E; e += 32) mask[e] = 0u;
  __syncwarp();
  const int t = c * kChunkTokens + lane;
  const bool valid = t < T;
  if (valid) {
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= E) {
        record_status(status, MOE_ERR_INVALID);
        e = -1;
      }
      // an expert listed twice is an error; both slots then share one row,
      // which keeps every row below the total count
      for (int jj = 0; jj < j; ++jj)
        if (e >= 0 && ids[jj] == e) record_status(status, MOE_ERR_INVALID);
      ids[j] = e;
      if (e >= 0) atomicOr(&mask[e], 1u << lane);
    }
  }
  __syncwarp();
  if (valid) {
    const uint32_t lower = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = ids[j];
      if (e >= 0) local_rank[(size_t)t * k + j] = __popc(mask[e] & lower);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(size_t)c * E + e] = __popc(mask[e]);
}

// Exclusive scan of n <= 2048 ints held in shared memory, by 1024 threads.
__device__ void block_exclusive_scan_2048(int32_t* v, int n, int32_t* total) {
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid;
  const int a = i0 < n ? v[i0] : 0;
  const int b = i0 + 1 < n ? v[i0 + 1] : 0;
  int incl = a + b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int excl = incl - (a + b) + warp_tot[warp];
  if (i0 < n) v[i0] = excl;
  if (i0 + 1 < n) v[i0 + 1] = excl + a;
  __syncthreads();
}

// Column-wise exclusive scan of hist over chunks (per expert), then the
// exclusive scan of the expert totals.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int32_t* __restrict__ hist, int C,
                                                             int E, int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[kMaxExperts];
  __shared__ int32_t total;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    int c = 0;
    for (; c + 4 <= C; c += 4) {
      const int v0 = hist[(size_t)(c + 0) * E + e];
      const int v1 = hist[(size_t)(c + 1) * E + e];
      const int v2 = hist[(size_t)(c + 2) * E + e];
      const int v3 = hist[(size_t)(c + 3) * E + e];
      hist[(size_t)(c + 0) * E + e] = run;
      hist[(size_t)(c + 1) * E + e] = run + v0;
      hist[(size_t)(c + 2) * E + e] = run + v0 + v1;
      hist[(size_t)(c + 3) * E + e] = run + v0 + v1 + v2;
      run += v0 + v1 + v2 + v3;
    }
    for (; c < C; ++c) {
      const int v = hist[(size_t)c * E + e];
      hist[(size_t)c * E + e] = run;
      run += v;
    }
    tot[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan_2048(tot, E, &total);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = tot[e];
  if (threadIdx.x == 0) offsets[E] = total;
}

// Many chunks: the column scans run one warp per expert (32 experts per
// CTA).  Lane l takes 8 consecutive chunks of each 256-chunk segment (its 8
// loads in flight at once), and a warp scan of the lane sums joins them;
// segments follow one another with a carry.  counts[e] = the column total.
// The exclusive scan of the totals into offsets is dispatch_offsets_kernel.
constexpr int kScanPerLane = 8;

__global__ void __launch_bounds__(1024) dispatch_colscan_kernel(int32_t* __restrict__ hist, int C,
                                                                int E,
                                                                int32_t* __restrict__ counts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + warp;
  if (e >= E) return;
  int carry = 0;
  for (int c0 = 0; c0 < C; c0 += 32 * kScanPerLane) {
    const int cl = c0 + lane * kScanPerLane;
    int v[kScanPerLane];
#pragma unroll
    for (int i = 0; i < kScanPerLane; ++i) v[i] = cl + i < C ? hist[(size_t)(cl + i) * E + e] : 0;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kScanPerLane; ++i) sum += v[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = carry + incl - sum;  // exclusive prefix of this lane's first chunk
#pragma unroll
    for (int i = 0; i < kScanPerLane; ++i) {
      if (cl + i < C) hist[(size_t)(cl + i) * E + e] = run;
      run += v[i];
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) counts[e] = carry;
}

// offsets = exclusive scan of counts (E <= 2048), offsets[E] = the total.
__global__ void __launch_bounds__(1024) dispatch_offsets_kernel(const int32_t* __restrict__ counts,
                                                                int E,
                                                                int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[kMaxExperts];
  __shared__ int32_t total;
  for (int e = threadIdx.x; e < E; e += blockDim.x) tot[e] = counts[e];
  __syncthreads();
  block_exclusive_scan_2048(tot, E, &total);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = tot[e];
  if (threadIdx.x == 0) offsets[E] = total;
}

// Chunks from which the column scans run one warp per expert.
constexpr int kWarpScanMinChunks = 32;

// Quantise the 8 values of one 16-byte bf16 vector with a row scale: IEEE
// division, round half to even, clamp to [-127, 127]; packs 8 int8 in a uint2.
// F16: also the fp16 values of the eight codes (exact: |q| <= 127).
template <bool F16 = false>
__device__ __forceinline__ uint2 quant8(const uint4 v, float sc, uint4* f16 = nullptr) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0u, 0u};
  uint32_t h[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
    const float f = bf16_bits_to_f32(bits);
    float q = sc > 0.f ? rintf(__fdiv_rn(f, sc)) : 0.f;
    q = fminf(fmaxf(q, -127.f), 127.f);
    const uint32_t b = static_cast<uint32_t>(static_cast<int>(q)) & 0xffu;
    out[i >> 2] |= b << (8 * (i & 3));
    if (F16) h[i >> 1] |= static_cast<uint32_t>(__half_as_ushort(__float2half_rn(q))) << (16 * (i & 1));
  }
  if (F16) *f16 = make_uint4(h[0], h[1], h[2], h[3]);
  return make_uint2(out[0], out[1]);
}

__device__ __forceinline__ float amax8(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[i] & 0xffffu)));
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[i] >> 16)));
  }
  return m;
}

// Row scale of one warp's row: max|v| / 127 in IEEE fp32.
__device__ __forceinline__ float warp_row_scale(const uint4* row, int nv, int lane) {
  float m = 0.f;
  for (int v = lane; v < nv; v += 32) m = fmaxf(m, amax8(row[v]));
  m = warp_max(m);
  return __fdiv_rn(m, 127.0f);
}

// bf16 x8 (natural order) -> fp16 x8 in pair order (c0 c4 c1 c5 c2 c6 c3 c7);
// fin turns false for a value beyond the fp16 range.
__device__ __forceinline__ uint4 bf16x8_to_f16_pairs(const uint4 x, bool& fin) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    fin &= fabsf(f[j]) <= 65504.0f && fabsf(f[j + 4]) <= 65504.0f;
    const __half2 h = __floats2half2_rn(f[j], f[j + 4]);
    o[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One warp per token: place its k (token, slot) pairs, then copy (or quantise
// once and copy) the token row into each of its k expert-sorted rows.
// PAIR: the rows are written in the expert kernels' pair order, fp16 (bf16
// input beyond the fp16 range records MOE_ERR_UNSUPPORTED) or int8.
template <bool Q8, bool PAIR>
__global__ void __launch_bounds__(256) dispatch_place_kernel(
    const int32_t* __restrict__ idx, const uint16_t* __restrict__ x, int T, int D, int E, int k,
    const int32_t* __restrict__ hist, const int32_t* __restrict__ local_rank,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
    int32_t* __restrict__ row_slot, int32_t* __restrict__ inv_row, void* __restrict__ x_sorted,
    float* __restrict__ x_scale, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  // gridDim.y slices of the row's 16-byte vectors (few tokens: more CTAs);
  // slice 0 also writes the permutation
  const bool first = blockIdx.y == 0;
  int row = -1;
  if (lane < k) {
    const int e = idx[(size_t)t * k + lane];
    if (e >= 0 && e < E) {
      row = offsets[e] + hist[(size_t)(t / kChunkTokens) * E + e] + local_rank[(size_t)t * k + lane];
      if (first) {
        row_token[row] = t;
        row_slot[row] = lane;
      }
    }
    if (first) inv_row[(size_t)t * k + lane] = row;
  }
  const int nv = D / 8;
  const int per = (nv + gridDim.y - 1) / gridDim.y;
  const int v0 = blockIdx.y * per, v1 = min(nv, v0 + per);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * D);
  if (!Q8) {
    uint4* dst = static_cast<uint4*>(x_sorted);
    bool fin = true;
    for (int v = v0 + lane; v < v1; v += 32) {
      const uint4 val = PAIR ? bf16x8_to_f16_pairs(src[v], fin) : src[v];
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, row, j);
        if (r >= 0) dst[(size_t)r * nv + v] = val;
      }
    }
    if (PAIR && !fin) record_status(status, MOE_ERR_UNSUPPORTED);
  } else {
    const float sc = warp_row_scale(src, nv, lane);  // the whole row, in every slice
    uint2* dst = static_cast<uint2*>(x_sorted);
    for (int v = v0 + lane; v < v1; v += 32) {
      uint2 q = quant8(src[v], sc);
      if (PAIR) q = make_uint2(__byte_perm(q.x, q.y, 0x5140u), __byte_perm(q.x, q.y, 0x7362u));
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, row, j);
        if (r >= 0) dst[(size_t)r * nv + v] = q;
      }
    }
    if (first && lane < k && row >= 0) x_scale[row] = sc;
  }
}

// Per-row int8 quantisation of R rows of C bf16 values (one warp per row).
// Rows at or beyond *row_count (when given) are skipped.
// With q16 (F16) the kernel also writes the fp16 values of the codes, the
// operand copy the tensor-core kernels read.
template <bool F16>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ v, int R,
                                                            int C, const int32_t* row_count,
                                                            int8_t* __restrict__ q,
                                                            float* __restrict__ scale,
                                                            uint16_t* __restrict__ q16) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= R) return;
  if (row_count && r >= *row_count) return;
  const int nv = C / 8;
  const uint4* src = reinterpret_cast<const uint4*>(v + (size_t)r * C);
  const float sc = warp_row_scale(src, nv, lane);
  uint2* dst = reinterpret_cast<uint2*>(q + (size_t)r * C);
  uint4* d16 = F16 ? reinterpret_cast<uint4*>(q16 + (size_t)r * C) : nullptr;
  for (int i = lane; i < nv; i += 32) {
    if (F16)
      dst[i] = quant8<true>(src[i], sc, d16 + i);
    else
      dst[i] = quant8(src[i], sc);
  }
  if (lane == 0) scale[r] = sc;
}

int launch_quantize_rows(const uint16_t* v, int R, int C, const int32_t* row_count, int8_t* q,
                         float* scale, cudaStream_t s, uint16_t* q16) {
  if (R == 0) return MOE_OK;
  if (q16)
    quantize_rows_kernel<true><<<(R + 7) / 8, 256, 0, s>>>(v, R, C, row_count, q, scale, q16);
  else
    quantize_rows_kernel<false><<<(R + 7) / 8, 256, 0, s>>>(v, R, C, row_count, q, scale, nullptr);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

static size_t dispatch_chunks(int T) { return (size_t)(T + kChunkTokens - 1) / kChunkTokens; }

// Scratch of moe_dispatch_noalloc: the per-chunk expert histograms followed by
// the in-chunk ranks.  Every GPU that loads the library holds these 2 MiB
// until the process exits.  Host code must not use the symbol as a device
// address; noalloc_scratch() resolves the address on the current device.
constexpr size_t kNoAllocScratchInts = 512 * 1024;
static __device__ __align__(256) int32_t g_dispatch_scratch[kNoAllocScratchInts];

// Device address of g_dispatch_scratch in the current device's context,
// looked up on every call (so it stays right after a device reset or a new
// primary context).  On failure records the CUDA error for
// moe_last_cuda_error and returns null.
static int32_t* noalloc_scratch() {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return nullptr;
  }
  return static_cast<int32_t*>(p);
}

// Count, scan and place kernels of one dispatch (T > 0, arguments checked).
static int run_dispatch(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                        int act_bits, bool pair, int32_t* counts, int32_t* offsets,
                        int32_t* row_token, int32_t* row_slot, int32_t* inv_row, void* x_sorted,
                        float* x_scale, int32_t* hist, int32_t* local_rank, cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const int C = static_cast<int>(dispatch_chunks(T));
  const size_t smem = (size_t)kCountWarps * (E + kChunkTokens * kMaxTopK) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    MOE_TRY_CUDA(cudaFuncSetAttribute(dispatch_count_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  }
  dispatch_count_kernel<<<(C + kCountWarps - 1) / kCountWarps, kCountWarps * 32, smem, s>>>(
      topk_idx, T, E, k, hist, local_rank, status);
  MOE_LAUNCH_CHECK();
  if (C < kWarpScanMinChunks) {
    dispatch_scan_kernel<<<1, 1024, 0, s>>>(hist, C, E, counts, offsets);
    MOE_LAUNCH_CHECK();
  } else {
    dispatch_colscan_kernel<<<(E + 31) / 32, 1024, 0, s>>>(hist, C, E, counts);
    MOE_LAUNCH_CHECK();
    dispatch_offsets_kernel<<<1, 1024, 0, s>>>(counts, E, offsets);
    MOE_LAUNCH_CHECK();
  }
  auto place = act_bits == 16 ? (pair ? dispatch_place_kernel<false, true>
                                      : dispatch_place_kernel<false, false>)
                              : (pair ? dispatch_place_kernel<true, true>
                                      : dispatch_place_kernel<true, false>);
  // few tokens: split each row over CTAs so that about 4 CTAs per SM run
  const int blocks = (T + 7) / 8;
  const int max_slices = (D / 8 + 31) / 32;
  int slices = (4 * num_sms() + blocks - 1) / blocks;
  slices = slices < 1 ? 1 : (slices > max_slices ? max_slices : slices);
  place<<<dim3(blocks, slices), 256, 0, s>>>(topk_idx, x, T, D, E, k, hist, local_rank, offsets,
                                             row_token, row_slot, inv_row, x_sorted, x_scale,
                                             status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_dispatch_pairs(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                          int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                          int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                          void* ws, cudaStream_t s) {
  if (T == 0) {
    MOE_TRY_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_TRY_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
    return MOE_OK;
  }
  const size_t C = dispatch_chunks(T);
  int32_t* hist = static_cast<int32_t*>(ws);
  int32_t* local_rank =
      reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align_up(C * E * sizeof(int32_t), 256));
  return run_dispatch(topk_idx, x, T, D, E, k, act_bits, true, counts, offsets, row_token,
                      row_slot, inv_row, x_sorted, x_scale, hist, local_rank, s);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_dispatch_workspace_size(int T, int E, int k) {
  if (T <= 0 || E <= 0 || k <= 0) return 256;
  return align_up(dispatch_chunks(T) * E * sizeof(int32_t), 256) +
         align_up((size_t)T * k * sizeof(int32_t), 256);
}

extern "C" int moe_dispatch(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                            int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                            int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                            void* ws, size_t ws_bytes, void* stream) {
  moe::Range range_("moe_dispatch");
  if (T < 0 || D <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (D % 64 != 0 || E > kMaxExperts || k > E || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    MOE_TRY_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_TRY_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
    return MOE_OK;
  }
  if (!topk_idx || !x || !row_token || !row_slot || !inv_row || !x_sorted || !ws)
    return MOE_ERR_INVALID;
  if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(x_sorted, 16)) return MOE_ERR_INVALID;
  if (ws_bytes < moe_dispatch_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE;
  const size_t C = dispatch_chunks(T);
  int32_t* hist = static_cast<int32_t*>(ws);
  int32_t* local_rank =
      reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align_up(C * E * sizeof(int32_t), 256));
  return run_dispatch(topk_idx, x, T, D, E, k, act_bits, false, counts, offsets, row_token,
                      row_slot, inv_row, x_sorted, x_scale, hist, local_rank, s);
}

extern "C" int moe_dispatch_pairs(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E,
                                  int k, int act_bits, int32_t* counts, int32_t* offsets,
                                  int32_t* row_token, int32_t* row_slot, int32_t* inv_row,
                                  void* x_sorted, float* x_scale, void* ws, size_t ws_bytes,
                                  void* stream) {
  moe::Range range_("moe_dispatch_pairs");
  if (T < 0 || D <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (D % 64 != 0 || E > kMaxExperts || k > E || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID;
  if (T > 0) {
    if (!topk_idx || !x || !row_token || !row_slot || !inv_row || !x_sorted || !ws)
      return MOE_ERR_INVALID;
    if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(x_sorted, 16)) return MOE_ERR_INVALID;
    if (ws_bytes < moe_dispatch_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE;
  }
  return launch_dispatch_pairs(topk_idx, x, T, D, E, k, act_bits, counts, offsets, row_token,
                               row_slot, inv_row, x_sorted, x_scale, ws,
                               static_cast<cudaStream_t>(stream));
}

extern "C" int moe_quantize_rows(const uint16_t* v, int R, int C, int8_t* q, float* scale,
                                 void* stream) {
  moe::Range range_("moe_quantize_rows");
  if (R < 0 || C <= 0) return MOE_ERR_INVALID;
  if (C % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (R == 0) return MOE_OK;
  if (!v || !q || !scale || !aligned(v, 16) || !aligned(q, 8)) return MOE_ERR_INVALID;
  return launch_quantize_rows(v, R, C, nullptr, q, scale, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_dispatch_noalloc(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E,
                                    int k, int act_bits, int32_t* counts, int32_t* offsets,
                                    int32_t* row_token, int32_t* row_slot, int32_t* inv_row,
                                    void* x_sorted, float* x_scale, void* stream) {
  moe::Range range_("moe_dispatch_noalloc");
  if (T < 0 || D <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (D % 64 != 0 || E > kMaxExperts || k > E || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (act_bits != 16 && act_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID;
  if (T > 0) {
    if (!topk_idx || !x || !row_token || !row_slot || !inv_row || !x_sorted) return MOE_ERR_INVALID;
    if (act_bits == 8 && !x_scale) return MOE_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(x_sorted, 16)) return MOE_ERR_INVALID;
  }
  const size_t C = dispatch_chunks(T);
  const size_t hist_ints = align_up(C * E * sizeof(int32_t), 256) / sizeof(int32_t);
  if (hist_ints + (size_t)T * k > kNoAllocScratchInts) return MOE_ERR_WORKSPACE;
  int32_t* scratch = noalloc_scratch();
  if (!scratch) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    MOE_TRY_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_TRY_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
    return MOE_OK;
  }
  return run_dispatch(topk_idx, x, T, D, E, k, act_bits, false, counts, offsets, row_token,
                      row_slot, inv_row, x_sorted, x_scale, scratch, scratch + hist_ints, s);
}
