// LSE merge of attention states.
//
// "10.3 FlashAttention: IO-aware algorithm design", 10.3.2 "LSE": segments
// with LSE_k combine as LSE = ln(sum_k e^LSE_k) and O = sum_k e^(LSE_k - LSE) O_k.
// "FlashAttention and inference operators" (CUDA handbook), split-K merge
// exercise: one row per worker, segments with no keys are skipped.
// Evaluated with M = max_k LSE_k as the shift, ascending k, no atomics, so the
// result is bitwise reproducible ("Lecture 4", sections 4.3 and 5.6).
//
// One warp per row; lane `l` owns dims 4l + 128c.  Every load is a 16-byte
// vector and a row's segments are read in order.
#include "common.cuh"

namespace {

template <int C, bool BF16_OUT>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int rows,
                                                    int S, int d, void* __restrict__ o_out,
                                                    float* __restrict__ lse_out) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lp = lse_parts + (size_t)row * S;

  float big = -INFINITY;
  for (int s = lane; s < S; s += 32) big = fmaxf(big, lp[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, off));

  float4 acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (big != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = lp[s];
      if (ls == -INFINITY) continue;  // empty segment: its O is never read
      const float w = expf(ls - big);
      wsum += w;
      const float* op = o_parts + ((size_t)row * S + s) * d;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const int j = 4 * lane + 128 * c;
        if (j < d) {
          const float4 x = *reinterpret_cast<const float4*>(op + j);
          acc[c].x = fmaf(w, x.x, acc[c].x);
          acc[c].y = fmaf(w, x.y, acc[c].y);
          acc[c].z = fmaf(w, x.z, acc[c].z);
          acc[c].w = fmaf(w, x.w, acc[c].w);
        }
      }
    }
  }
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int j = 4 * lane + 128 * c;
    if (j >= d) continue;
    const float4 r = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
    if (BF16_OUT) {
      uint2 packed = make_uint2(attn::pack_bf16x2(r.x, r.y), attn::pack_bf16x2(r.z, r.w));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + (size_t)row * d + j) = packed;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(o_out) + (size_t)row * d + j) = r;
    }
  }
  if (lane == 0 && lse_out != nullptr) lse_out[row] = empty ? -INFINITY : big + logf(wsum);
}

template <bool BF16_OUT>
void launch(const float* o_parts, const float* lse_parts, int rows, int S, int d, void* o_out,
            float* lse_out, cudaStream_t stream) {
  const int blocks = (rows + 3) / 4;
  const int c = (d + 127) / 128;
  if (c == 1)
    merge_kernel<1, BF16_OUT><<<blocks, 128, 0, stream>>>(o_parts, lse_parts, rows, S, d, o_out, lse_out);
  else if (c == 2)
    merge_kernel<2, BF16_OUT><<<blocks, 128, 0, stream>>>(o_parts, lse_parts, rows, S, d, o_out, lse_out);
  else
    merge_kernel<4, BF16_OUT><<<blocks, 128, 0, stream>>>(o_parts, lse_parts, rows, S, d, o_out, lse_out);
}

}  // namespace

namespace attn_host {

attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int rows, int S, int d,
                           void* o_out, float* lse_out, attn_dtype_t out_dtype, cudaStream_t stream) {
  if (out_dtype == ATTN_BF16)
    launch<true>(o_parts, lse_parts, rows, S, d, o_out, lse_out, stream);
  else
    launch<false>(o_parts, lse_parts, rows, S, d, o_out, lse_out, stream);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
