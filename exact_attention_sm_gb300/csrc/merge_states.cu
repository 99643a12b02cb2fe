// LSE merge of attention states.
//
// "10.3 FlashAttention: IO-aware algorithm design", 10.3.2 "LSE": segments
// with LSE_k combine as LSE = ln(sum_k e^LSE_k) and O = sum_k e^(LSE_k - LSE) O_k.
// "FlashAttention and inference operators" (CUDA handbook), split-K merge
// exercise: one row per worker, segments with no keys are skipped.
// Evaluated with M = max_k LSE_k as the shift, in an order fixed by the
// problem size alone and with no atomics, so the result is bitwise
// reproducible ("Lecture 4", sections 4.3 and 5.6).
//
// One CTA of NW warps per row, NW = 4, 8 or 16 from S (more warps when a
// row has many states, so that few rows still keep many loads in flight).
// The states of the row are dealt to the warps (warp w takes s = w, w + NW,
// ...), each warp keeps 4 states' loads in flight (the O loads do not wait
// for the weights) and lane l owns dims 4l + 128c; the NW warp partials are
// then added in warp order.  The summation order is fixed by (S, d) alone,
// so results are bitwise reproducible.
#include "common.cuh"

namespace {

constexpr int UNROLL = 4;

template <int NW, int C, bool BF16_OUT>
__global__ void __launch_bounds__(NW * 32) merge_kernel(const float* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts,
                                                        int S, int d, void* __restrict__ o_out,
                                                        float* __restrict__ lse_out) {
  __shared__ float red[NW];
  __shared__ __align__(16) float4 part_acc[NW][C * 32];
  __shared__ float part_w[NW];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* lp = lse_parts + static_cast<size_t>(row) * S;
  const float* op = o_parts + static_cast<size_t>(row) * S * d;

  float big = -INFINITY;
  for (int s = threadIdx.x; s < S; s += NW * 32) big = fmaxf(big, lp[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, off));
  if (lane == 0) red[warp] = big;
  __syncthreads();
  big = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) big = fmaxf(big, red[w]);

  float4 acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (big != -INFINITY) {
    for (int s0 = warp; s0 < S; s0 += NW * UNROLL) {
      float w[UNROLL];
      float4 x[UNROLL][C];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int s = s0 + u * NW;
        const float ls = s < S ? lp[s] : -INFINITY;
        w[u] = ls == -INFINITY ? 0.f : expf(ls - big);  // empty segment: weight 0
#pragma unroll
        for (int c = 0; c < C; ++c) {
          const int j = 4 * lane + 128 * c;
          x[u][c] = (s < S && j < d)
                        ? *reinterpret_cast<const float4*>(op + static_cast<size_t>(s) * d + j)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      // An empty segment's O may hold anything (it is not read by value):
      // its weight 0 selects zeros instead of multiplying.
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)
#pragma unroll
        for (int c = 0; c < C; ++c)
          if (!(w[u] > 0.f)) x[u][c] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        wsum += w[u];
#pragma unroll
        for (int c = 0; c < C; ++c) {
          acc[c].x = fmaf(w[u], x[u][c].x, acc[c].x);
          acc[c].y = fmaf(w[u], x[u][c].y, acc[c].y);
          acc[c].z = fmaf(w[u], x[u][c].z, acc[c].z);
          acc[c].w = fmaf(w[u], x[u][c].w, acc[c].w);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) part_acc[warp][c * 32 + lane] = acc[c];
  if (lane == 0) part_w[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;

  float total = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) total += part_w[w];
  const bool empty = !(total > 0.f);
  const float inv = empty ? 0.f : 1.f / total;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int j = 4 * lane + 128 * c;
    if (j >= d) continue;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float4 p = part_acc[w][c * 32 + lane];
      r.x += p.x;
      r.y += p.y;
      r.z += p.z;
      r.w += p.w;
    }
    r = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
    if (BF16_OUT) {
      uint2 packed = make_uint2(attn::pack_bf16x2(r.x, r.y), attn::pack_bf16x2(r.z, r.w));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + static_cast<size_t>(row) * d + j) = packed;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(o_out) + static_cast<size_t>(row) * d + j) = r;
    }
  }
  if (lane == 0 && lse_out != nullptr) lse_out[row] = empty ? -INFINITY : big + logf(total);
}

template <int NW, bool BF16_OUT>
void launch_nw(const float* o_parts, const float* lse_parts, int rows, int S, int d, void* o_out,
               float* lse_out, cudaStream_t stream) {
  const int c = (d + 127) / 128;
  if (c == 1)
    merge_kernel<NW, 1, BF16_OUT><<<rows, NW * 32, 0, stream>>>(o_parts, lse_parts, S, d, o_out,
                                                               lse_out);
  else if (c == 2)
    merge_kernel<NW, 2, BF16_OUT><<<rows, NW * 32, 0, stream>>>(o_parts, lse_parts, S, d, o_out,
                                                               lse_out);
  else
    merge_kernel<NW, 4, BF16_OUT><<<rows, NW * 32, 0, stream>>>(o_parts, lse_parts, S, d, o_out,
                                                               lse_out);
}

template <bool BF16_OUT>
void launch(const float* o_parts, const float* lse_parts, int rows, int S, int d, void* o_out,
            float* lse_out, cudaStream_t stream) {
  if (S <= 16)
    launch_nw<4, BF16_OUT>(o_parts, lse_parts, rows, S, d, o_out, lse_out, stream);
  else if (S <= 32)
    launch_nw<8, BF16_OUT>(o_parts, lse_parts, rows, S, d, o_out, lse_out, stream);
  else
    launch_nw<16, BF16_OUT>(o_parts, lse_parts, rows, S, d, o_out, lse_out, stream);
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
