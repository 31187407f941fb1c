// Status word, device queries, tensor-map encoding, and the status /
// self-test entry points of the C ABI.
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {

__device__ int g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
std::atomic<uint64_t> g_launches{0};

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

// Looked up on every call, with the caller's device current: the address
// belongs to the current context, so it stays right after a device reset or
// a new primary context, which a cache keyed by device would not.
int* status_word() {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return nullptr;
  }
  return static_cast<int*>(p);
}

int num_sms() {
  int d = current_device();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_num_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
    g_num_sms[d] = n;
  }
  return g_num_sms[d];
}

void note_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim,
                        gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A barrier that nothing completes: the bounded wait must run out.
__global__ void wait_selftest_kernel(int64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int cta_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    cta_abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // The phase with parity 0 never completes (no arrival is ever made).
    mbar_wait(&bar, 0, Waiter{&cta_abort, status, limit_ns});
  }
  __syncthreads();
}

}  // namespace moe

extern "C" {

int moe_check_error(void* stream) {
  moe::Range range_("moe_check_error");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    moe::note_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  int* w = moe::status_word();
  if (!w) return MOE_ERR_CUDA;
  int host = 0;
  MOE_TRY_CUDA(cudaMemcpyAsync(&host, w, sizeof(int), cudaMemcpyDeviceToHost, s));
  MOE_TRY_CUDA(cudaMemsetAsync(w, 0, sizeof(int), s));
  MOE_TRY_CUDA(cudaStreamSynchronize(s));
  return host;
}

int moe_wait_selftest(int64_t limit_ns, void* stream) {
  moe::Range range_("moe_wait_selftest");
  if (limit_ns < 1000 || limit_ns > 5000000000LL) return MOE_ERR_INVALID;
  int* w = moe::status_word();
  if (!w) return MOE_ERR_CUDA;
  moe::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, w);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_cuda_error(void) { return cudaGetErrorName(moe::g_last_cuda_error); }

const char* moe_version(void) { return "int4-routed-moe sm_103a 0.1"; }

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
