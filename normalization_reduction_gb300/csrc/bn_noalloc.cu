// bn_noalloc.cu -- training-mode BatchNorm for callers that cannot allocate
// device memory.
//
// fnorm_batchnorm_train needs a caller-provided workspace for its per-CTA
// partial statistics. Some callers have no way to provide one: code that runs
// under a fixed memory budget carved out up front, plugins whose host owns the
// allocator and forbids allocation after start-up, and latency-critical loops
// where a cudaMalloc (which may synchronise the device) is not acceptable.
// fnorm_batchnorm_train_noalloc serves them with a scratch area that lives in
// this library: a file-scope __device__ array of kNoallocScratchBytes bytes.
// Every GPU that loads the library holds this array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fnorm.h"
#include "fnorm_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(2) << 20;   // 2 MiB per device

// The scratch itself. Host code must not pass this name to a kernel: on the
// host it is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bn_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_bn_scratch on the current device, looked up once per
// device (with that device current) and cached. nullptr on failure.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_bn_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" FNORM_API fnorm_status fnorm_batchnorm_train_noalloc(
    const float* x, float* y, const float* gamma, const float* beta, float scale,
    float* running_mean, float* running_var, float momentum, float eps, float* save_mean,
    float* save_rstd, int64_t N, int64_t C, int64_t S, fnorm_stream_t stream) {
  // The arguments are checked exactly as fnorm_batchnorm_train checks them
  // (same errors for the same mistakes); then shapes whose partial statistics
  // do not fit the static scratch are refused, before anything touches the GPU.
  int64_t total = 0;
  const fnorm_status st =
      fnorm::bn_train_check(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                            save_mean, save_rstd, N, C, S, &total);
  if (st != FNORM_OK || total == 0) return st;
  if (fnorm_batchnorm_workspace_size(N, C, S) > kNoallocScratchBytes)
    return FNORM_ERR_UNSUPPORTED;
  void* scratch = scratch_address();
  if (!scratch) return FNORM_ERR_CUDA;
  // The same validation and kernels as fnorm_batchnorm_train, with the static
  // scratch as the workspace. The workspace needs no clearing: each call
  // writes every partial before reading it.
  return fnorm_batchnorm_train(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                               save_mean, save_rstd, N, C, S, scratch, kNoallocScratchBytes,
                               stream);
}
