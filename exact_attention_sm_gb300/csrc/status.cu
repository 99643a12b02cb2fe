// Device status word shared by every kernel of the library, one per device,
// and the self-test of the bounded wait that every pipelined kernel uses.
#include "common.cuh"
#include "sm103_ptx.cuh"

namespace {
__device__ int g_attn_status = 0;

// One thread waits on an mbarrier that nothing ever arrives at, with the same
// bounded wait the attention kernels use, and records the timeout.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  sm103::mbar_init(&bar, 1);
  sm103::fence_mbar_init();
  if (!sm103::mbar_wait(&bar, 0, &abort_flag, limit_ns))
    attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
}
}  // namespace

namespace attn_host {

int* device_status_ptr() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cached[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace attn_host

extern "C" attn_status_t attn_get_device_status(attn_stream_t stream) {
  int* p = attn_host::device_status_ptr();
  if (p == nullptr) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return static_cast<attn_status_t>(value);
}

extern "C" attn_status_t attn_selftest_wait_timeout(int limit_ms, attn_stream_t stream) {
  if (limit_ms <= 0 || limit_ms > 10000) return ATTN_ERR_INVALID_ARG;
  int* p = attn_host::device_status_ptr();
  if (p == nullptr) return ATTN_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(limit_ms) * 1000000ull, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
