// Shared device/host helpers of libattn (no attention arithmetic here).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Records `code` in the library's device status word unless an earlier error
// is already there (the first error wins); the host reads and clears it with
// attn_get_device_status().
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

// Round-to-nearest-even pack of two floats into a bf16x2 word (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Streaming 16-byte load that bypasses L1 (each K/V byte is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace attn

// Host-side launchers (one per kernel family) used by api.cpp.
namespace attn_host {
// Index of the current device for per-device caches (kernel attributes,
// occupancy): -1 on error or for device numbers past 63.
inline int current_device_slot() {
  int d = 0;
  return (cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < 64) ? d : -1;
}

int* device_status_ptr();  // address of the status word on the current device (nullptr on error)
int num_sms();             // SM count of the current device (cached per device)
int decode_ctas_per_sm();  // resident decode CTAs per SM for the decode kernel

attn_status_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                 int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                 float scale, cudaStream_t stream);
// q_div > 1: output head h reads the Q rows of head h / q_div (several K/V
// ranges share one set of queries).
attn_status_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                  float scale, int q_div, cudaStream_t stream);
// Packed queries against a paged KV cache: a sequence's blocks are row b of
// block_table ([B, max_pages]) or, when kv_indptr is set, the block-sparse
// row indices[kv_indptr[b] .. kv_indptr[b + 1]) (block_table = indices, nnz
// entries); block_size is a power of two from 1 to 128.
attn_status_t launch_prefill_bf16_paged(const void* q, const void* k_pages, const void* v_pages,
                                        const int* block_table, const int* kv_indptr, int nnz,
                                        int block_size, const int* cu_q, const int* seq_lens_k,
                                        void* o, float* lse, int B, int max_q, int max_k,
                                        int total_q, int Hq, int Hkv, int d, int max_pages,
                                        int num_pages, int causal, float scale,
                                        cudaStream_t stream);
attn_status_t launch_prefill_bf16_varlen(const void* q, const void* k, const void* v, void* o,
                                         float* lse, const int* cu_q, const int* cu_k, int B,
                                         int max_q, int max_k, int total_q, int total_k, int Hq,
                                         int Hkv, int d, int causal, float scale,
                                         cudaStream_t stream);
attn_status_t launch_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* seq_lens, int page_size,
                                 int chunk, int max_splits, void* o, float* lse, float* part_o,
                                 float* part_lse, int B, int Hq, int Hkv, int d, int max_pages,
                                 int num_pages, float scale, const int32_t* lens_host,
                                 cudaStream_t stream);
attn_status_t launch_bwd_bf16(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                              float* dd, int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                              float scale, cudaStream_t stream);
int decode_balanced_ctas_per_sm();
attn_status_t launch_decode_balanced(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     const int32_t* cta_off, const int32_t* cta_units,
                                     const int32_t* unit, const int32_t* seg_off,
                                     const int32_t* seg_units, int num_ctas, int U, float* part_o,
                                     float* part_lse, void* o, float* lse, int B, int Hq, int Hkv,
                                     int d, int page_size, int max_pages, int num_pages,
                                     float scale, cudaStream_t stream);
attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int rows, int S, int d,
                           void* o_out, float* lse_out, attn_dtype_t out_dtype, cudaStream_t stream);
attn_status_t launch_cascade_gather_q(const void* q, void* q_stack, int B, int Hq, int Hkv, int d,
                                      cudaStream_t stream);
attn_status_t launch_cascade_merge(const void* o_pre, const float* lse_pre, int S_pre,
                                   const float* o_suf, const float* lse_suf, int S_suf, int B,
                                   int Hq, int Hkv, int d, void* o, float* lse, cudaStream_t stream);
}  // namespace attn_host
