// attn_decode_paged_noalloc: split-KV paged decode whose workspace is a fixed
// array owned by the library, for callers that may not allocate device memory.
//
// The array below is a file-scope device variable.  Host code cannot use its
// name as a device address (on the host it only names a shadow object), so
// the entry point asks the runtime for the real address once per device and
// passes that pointer on.
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device; looked up on the
// first call for that device (with that device current) and cached.
attn_status_t scratch_for_current_device(void** out) {
  static void* cached[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  if (cached[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    cached[dev] = p;
  }
  *out = cached[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
    const int32_t* seq_lens, const int32_t* seq_lens_host, int page_size, int num_splits, void* o,
    float* lse, int B, int Hq, int Hkv, int d, int max_pages_per_seq, int num_pages, float scale,
    attn_dtype_t dtype, attn_stream_t stream) {
  // The planner needs the lengths on the host; without them attn_decode_paged
  // would make a host copy, which this entry point promises not to do.
  if (seq_lens_host == nullptr && num_splits != 1) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const attn_status_t s = scratch_for_current_device(&scratch);
  if (s != ATTN_OK) return s;
  // Same validation, planning and kernels as attn_decode_paged; the scratch
  // array stands in for the caller's workspace (ATTN_ERR_WORKSPACE if the
  // plan needs more than it holds).
  return attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, seq_lens_host, page_size,
                           num_splits, o, lse, B, Hq, Hkv, d, max_pages_per_seq, num_pages, scale,
                           scratch, kScratchBytes, dtype, stream);
}
