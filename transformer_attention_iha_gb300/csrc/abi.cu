// Host-side plumbing of the C ABI: status strings, per-thread error detail,
// the device error words, SM count and tensor-map encoding.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"

namespace iha {

namespace {
thread_local char t_last_error[512] = "";
// One-shot failure-path test (iha_test_fail_next_wait): 0 = not armed.
thread_local uint64_t t_test_limit_ns = 0;
thread_local bool t_test_withhold = false;
std::mutex g_reader_mu;
dev_error_reader g_readers[16];
int g_n_readers = 0;
}  // namespace

iha_status fail(iha_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

iha_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(IHA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return IHA_OK;
}

uint64_t wait_limit_for_next_launch() {
  const uint64_t v = t_test_limit_ns;
  t_test_limit_ns = 0;
  return v ? v : kWaitLimitNs;
}

bool withhold_for_this_launch() {
  const bool v = t_test_withhold;
  t_test_withhold = false;
  return v;
}

int register_dev_error_reader(dev_error_reader r) {
  std::lock_guard<std::mutex> lk(g_reader_mu);
  if (g_n_readers < 16) g_readers[g_n_readers++] = r;
  return g_n_readers;
}

int sm_count() {
  // per-device cache, read and filled from any host thread (every writer
  // stores the same value, so relaxed ordering suffices)
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, rank, base, reinterpret_cast<const cuuint64_t*>(dims),
            reinterpret_cast<const cuuint64_t*>(strides_bytes),
            reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace iha

extern "C" {

const char* iha_status_string(iha_status s) {
  switch (s) {
    case IHA_OK: return "ok";
    case IHA_ERR_INVALID_ARG: return "invalid argument";
    case IHA_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case IHA_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case IHA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* iha_last_error(void) { return iha::t_last_error; }

iha_status iha_test_fail_next_wait(int limit_us) {
  if (limit_us < 1 || limit_us > 1000000)
    return iha::fail(IHA_ERR_INVALID_ARG, "iha_test_fail_next_wait: limit_us must be in [1, 1e6]");
  iha::t_test_limit_ns = (uint64_t)limit_us * 1000ull;
  iha::t_test_withhold = true;
  return IHA_OK;
}

int iha_device_error(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int n;
  {
    std::lock_guard<std::mutex> lk(iha::g_reader_mu);
    n = iha::g_n_readers;
  }
  int acc = 0;
  for (int i = 0; i < n; ++i) {
    int v = iha::g_readers[i](clear);
    if (v < 0) return -1;
    acc |= v;
  }
  return acc;
}

}  // extern "C"
