// Host runtime of libbiv: error strings, device error word, SM count, the
// timeout self-test, and the cached driver entry point for TMA descriptors.
#include <cstdlib>
#include <mutex>
#include <string>

#include "common.cuh"

namespace biv {

__device__ int g_error_word = 0;

int* device_error_word() {
  static int* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int*>(p);
  }
  return ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
  return fn;
}

static thread_local std::string t_last_error = "no error";

biv_status set_error(biv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

biv_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(BIV_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return BIV_OK;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("BIV_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// A CTA that waits on an mbarrier no one arrives on; the bounded wait gives up
// after limit_ns, sets the error word, and the kernel returns normally.
__global__ void selftest_timeout_kernel(uint64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, err, limit_ns);
}

}  // namespace biv

using namespace biv;

extern "C" {

int biv_version(void) { return 100; }

const char* biv_last_error(void) { return t_last_error.c_str(); }

int biv_device_sm_count(void) { return sm_count(); }

biv_status biv_poll_error(biv_stream_t stream, int* code) {
  int v = 0;
  if (cudaStreamSynchronize(as_cuda(stream)) != cudaSuccess)
    return set_error(BIV_ERR_CUDA, "biv_poll_error: stream sync failed: %s",
                     cudaGetErrorString(cudaGetLastError()));
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess)
    return set_error(BIV_ERR_CUDA, "biv_poll_error: read failed");
  int zero = 0;
  if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess)
    return set_error(BIV_ERR_CUDA, "biv_poll_error: clear failed");
  if (code) *code = v;
  if (v == kErrTimeout) return set_error(BIV_ERR_TIMEOUT, "a device-side wait timed out");
  if (v != 0) return set_error(BIV_ERR_INVALID, "device reported error code %d", v);
  return BIV_OK;
}

biv_status biv_selftest_timeout(uint64_t limit_ns, biv_stream_t stream) {
  BIV_REQUIRE(limit_ns <= 5000000000ull, "selftest_timeout: limit above 5 s");
  selftest_timeout_kernel<<<1, 32, 0, as_cuda(stream)>>>(limit_ns, device_error_word());
  return check_launch("selftest_timeout");
}

}  // extern "C"
