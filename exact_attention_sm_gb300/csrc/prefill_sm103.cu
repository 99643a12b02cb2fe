#include "common.cuh"
namespace attn_host {
attn_status_t launch_prefill_bf16(const void*, const void*, const void*, void*, float*, int, int,
                                  int, int, int, int, int, float, cudaStream_t) {
  return ATTN_ERR_UNSUPPORTED;
}
}  // namespace attn_host
