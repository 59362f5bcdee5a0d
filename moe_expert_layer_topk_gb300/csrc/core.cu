// Library core: error strings, the device status word, device queries.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace {

thread_local char g_err[512] = {0};

// Status word: OR of MOE_STATUS_* bits set by kernels.  One copy per device
// that loads the library; its address is looked up once per device.
__device__ int g_status_word = 0;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;

}  // namespace

namespace moe {

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_err[0] = 0; }

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return (d >= 0 && d < kMaxDevices) ? d : -1;
}

int* status_word() {
  int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

int sm_count() {
  int d = current_device();
  if (d < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    g_sms[d] = n;
  }
  return g_sms[d];
}

}  // namespace moe

extern "C" {

int moe_abi_version(void) { return 102; }

const char* moe_last_error_string(void) { return g_err; }

int moe_read_device_status(int* status, int reset, void* stream) {
  moe::clear_error();
  if (!status) return moe::fail(MOE_ERR_INVALID_ARG, "moe_read_device_status: status is NULL");
  int* p = moe::status_word();
  if (!p) return moe::fail(MOE_ERR_CUDA, "moe_read_device_status: no device status word");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, p, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && reset) {
    e = cudaMemsetAsync(p, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "moe_read_device_status: %s", cudaGetErrorString(e));
  *status = v;
  return MOE_OK;
}

}  // extern "C"
