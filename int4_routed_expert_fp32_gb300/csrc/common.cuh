// Shared device helpers of the sm_103a kernels: status word, bounded
// mbarrier waits, bulk / tensor copies, bf16 conversions, tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#if defined(__has_include)
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define MOE_HAVE_NVTX 1
#endif
#endif

namespace moe {

constexpr int kGroup = 32;          // columns per weight scale
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 2048;
constexpr int64_t kDefaultWaitNs = 2000000000LL;  // 2 s per wait before giving up

// ------------------------------------------------------------------ host side

// Device address of the status word on the current device (null after a
// failed lookup, whose CUDA error is recorded for moe_last_cuda_error).
int* status_word();
// Number of SMs of the current device (cached).
int num_sms();
// Record the last CUDA error for moe_check_error diagnostics.
void note_cuda_error(cudaError_t e);
// Count one kernel launch of this library (read by moe_launch_count).
void count_launch();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Names a stretch of host code (one C-ABI call, or one stage of the layer) in
// a profiler's timeline: an NVTX range on the calling thread, open for the
// object's lifetime.  Without an attached tool NVTX calls return at once;
// without the NVTX headers this is empty.
class Range {
 public:
  explicit Range(const char* name) {
#ifdef MOE_HAVE_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~Range() {
#ifdef MOE_HAVE_NVTX
    nvtxRangePop();
#endif
  }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

// Pair order of the activation rows the expert kernels read and write: in
// every block of 8 columns, column j (j < 4) sits at position 2j and column
// j + 4 at 2j + 1 (c0 c4 c1 c5 c2 c6 c3 c7), the order in which a packed
// int32 word pairs its nibbles.
__host__ __device__ __forceinline__ int pair_pos(int c) {
  return (c & ~7) | ((c & 3) << 1) | ((c >> 2) & 1);
}
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Encode a tiled tensor map (driver entry point looked up through the runtime).
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);

#define MOE_TRY_CUDA(expr)                    \
  do {                                        \
    cudaError_t e__ = (expr);                 \
    if (e__ != cudaSuccess) {                 \
      ::moe::note_cuda_error(e__);            \
      return MOE_ERR_CUDA;                    \
    }                                         \
  } while (0)

// Follows every kernel launch of the library: counts it and checks it.
#define MOE_LAUNCH_CHECK()                    \
  do {                                        \
    ::moe::count_launch();                    \
    MOE_TRY_CUDA(cudaGetLastError());         \
  } while (0)

// ---------------------------------------------------------------- device side

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// SiLU(g) * u, with SiLU(g) = g / 2 + (g / 2) tanh(g / 2) (the logistic
// function through the hardware tanh approximation, relative error ~2^-11).
__device__ __forceinline__ float silu_mul(float g, float u) {
  float th;
  const float hg = 0.5f * g;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hg));
  return fmaf(hg, th, hg) * u;
}

// Two independent fp32 FMAs in one instruction: y0 = fma(s, p0, y0) and
// y1 = fma(s, p1, y1), each rounded as fmaf (the packed form halves the
// issue slots; the FMA pipe rate is the same).  s2 is s in both halves
// (pair_f32).
__device__ __forceinline__ uint64_t pair_f32(float s) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}

__device__ __forceinline__ void fma_f32x2(float& y0, float& y1, uint64_t s2, float p0, float p1) {
  asm("{\n .reg .b64 a, c;\n mov.b64 a, {%2, %3};\n mov.b64 c, {%0, %1};\n"
      " fma.rn.f32x2 c, %4, a, c;\n mov.b64 {%0, %1}, c;\n}"
      : "+f"(y0), "+f"(y1)
      : "f"(p0), "f"(p1), "l"(s2));
}

// ---- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to kSuspendNs while the phase
// is incomplete; the thread resumes as soon as the phase completes, so a
// waiting warp takes no issue slots from the working ones.
constexpr uint32_t kSuspendNs = 100000;

__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded waits.  Every wait on an mbarrier (or on another CTA's counter)
// is bounded by %globaltimer.  Each CTA keeps an abort flag in shared
// memory: a wait that runs out records MOE_ERR_TIMEOUT in the device status
// word and sets the flag, and every later wait of the same CTA then gives up
// at once, so a CTA whose pipeline stopped leaves after one time-out rather
// than one per wait.  Kernels only ever write the status word: an error that
// an earlier call recorded does not change what a later call computes.
struct Waiter {
  int* abort;        // the CTA's flag (shared memory)
  int* status;       // the device status word (written, never read)
  int64_t limit_ns;  // per wait
};

__device__ __forceinline__ bool aborted(const Waiter& w) {
  return *reinterpret_cast<const volatile int*>(w.abort) != 0;
}

__device__ __forceinline__ void give_up(const Waiter& w) {
  *reinterpret_cast<volatile int*>(w.abort) = 1;
  record_status(w.status, MOE_ERR_TIMEOUT);
}

// Wait for the phase with the given parity to complete, for at most
// w.limit_ns; gives up at once when the CTA has aborted.  Returns true when
// the phase completed.  backoff_ns > 0: sleep that long between rounds of
// polls (for waits that last long, so that the waiting warps leave the issue
// slots to others).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Waiter& w,
                                          uint32_t backoff_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  if (aborted(w)) return false;  // a shared-memory read: cheap on the fast path
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_suspend(bar, parity)) return true;
    if (backoff_ns) __nanosleep(backoff_ns);
    if (aborted(w)) return false;
    if (static_cast<int64_t>(global_timer_ns() - t0) > w.limit_ns) {
      give_up(w);
      return false;
    }
  }
}

// Time a CTA's exit path waits, per barrier, for work it issued itself
// (copies in flight, MMAs) before it leaves anyway.
constexpr int64_t kDrainNs = 100000000LL;

// Wait for a phase on the exit path: ignores the abort flag (the work it
// waits for was issued and completes by itself), bounded by kDrainNs.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<int64_t>(global_timer_ns() - t0) > kDrainNs) {
      record_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Let the last copies a producer issued into a `stages`-slot ring land:
// `issued` fills in total, fill i completing phase i / stages of barrier
// full[i % stages].  Called on every exit of a producer, so that no copy is
// still writing the CTA's shared memory when it leaves; on the normal path
// these phases have completed and the waits return at once.
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t issued, uint32_t stages,
                                          int* status) {
  const uint32_t first = issued >= stages ? issued - stages : 0;
  for (uint32_t i = first; i < issued; ++i) mbar_drain(&full[i % stages], (i / stages) & 1u, status);
}

// ---- asynchronous copies

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled tensor copy global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_g2s_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                           int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 4-byte asynchronous copy global -> shared (LDGSTS).
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Arrive on `bar` once all prior cp.async of this thread have landed; the
// barrier's expected count must include this arrival.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- warp reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace moe
