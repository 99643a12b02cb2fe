// Cascade (shared-prefix) decode: the two small kernels around the prefix
// prefill and the suffix decode.
//
// "Lecture 4 - Efficient attention kernels", section 4.4 (cascade attention)
// and 5.3 (composable formats): the n requests' query rows of each KV head
// are stacked into one (n * g) x d matrix that attends to the shared prefix
// once, on the tensor cores; each request attends to its own suffix; the two
// attention states of every row are merged with the LSE operator
// ("10.3 FlashAttention", 10.3.2 "LSE").
//
//   cascade_gather_q: q [B, Hq, d] -> q_stack [Hkv, B * g, d], row b * g + i
//                     of KV head h = query head h * g + i of request b.
//   cascade_merge:    per output row, the S_pre prefix-chunk states (bf16 O
//                     normalised per chunk, fp32 LSE; from the prefill) and
//                     the S_suf suffix states (fp32 O, fp32 LSE; from the
//                     decode) are merged in a fixed order (prefix chunks
//                     ascending, then suffix segments ascending), no atomics.
#include "common.cuh"

namespace {

__global__ void cascade_gather_q_kernel(const uint4* __restrict__ q, uint4* __restrict__ q_stack,
                                        int B, int Hq, int Hkv, int chunks_per_group) {
  // One thread per 16-byte chunk of q_stack; a (KV head, request) pair owns
  // g consecutive query heads = chunks_per_group chunks, contiguous on both
  // sides.
  const long long total = static_cast<long long>(B) * Hkv * chunks_per_group;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int c = static_cast<int>(i % chunks_per_group);
  const long long hb = i / chunks_per_group;  // h * B + b
  const int b = static_cast<int>(hb % B);
  const int h = static_cast<int>(hb / B);
  const long long src = (static_cast<long long>(b) * Hkv + h) * chunks_per_group + c;
  q_stack[i] = q[src];
}

constexpr int kRowsPerBlock = 4;  // one warp per output row
constexpr unsigned kFull = 0xffffffffu;

// One warp per output row.  The row's S = S_pre + S_suf states are numbered
// prefix chunks first, then suffix segments; lane l holds the LSE (and later
// the weight) of states l, l + 32, ...  The max and the weight sum are
// butterfly reductions and the weighted sum of the O_s runs over s in
// ascending order, so the result depends on (S_pre, S_suf) alone.
__global__ void __launch_bounds__(kRowsPerBlock * 32)
    cascade_merge_kernel(const __nv_bfloat16* __restrict__ o_pre, const float* __restrict__ lse_pre,
                         int S_pre, const float* __restrict__ o_suf,
                         const float* __restrict__ lse_suf, int S_suf, int B, int Hq, int Hkv,
                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int D = 128;  // lane l owns dims 4l .. 4l+3
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerBlock + warp;
  if (r >= B * Hq) return;
  const int b = r / Hq, hq = r % Hq, g = Hq / Hkv;
  const int h = hq / g;
  const long long lq = static_cast<long long>(B) * g;  // stacked rows per KV head
  const long long prow = static_cast<long long>(b) * g + hq % g;
  const int S = S_pre + S_suf;
  auto state_lse = [&](int s) {
    return s < S_pre ? lse_pre[(static_cast<long long>(h) * S_pre + s) * lq + prow]
                     : lse_suf[static_cast<long long>(r) * S_suf + (s - S_pre)];
  };

  float big = -INFINITY;
  for (int s = lane; s < S; s += 32) big = fmaxf(big, state_lse(s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(kFull, big, off));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (big != -INFINITY) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int mine = s0 + lane;
      const float ls = mine < S ? state_lse(mine) : -INFINITY;
      const float wl = ls == -INFINITY ? 0.f : expf(ls - big);  // empty state: weight 0
      float part = wl;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
      wsum += part;
      const int n = min(32, S - s0);
      // Batches of 8 states: all loads first, then the FMAs in state order.
      // Empty states hold O = 0 (both producers write it), so their weight 0
      // needs no branch.
      for (int j0 = 0; j0 < n; j0 += 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int s = s0 + j0 + u;
          if (j0 + u >= n) {
            x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (s < S_pre) {
            const uint2 raw = *reinterpret_cast<const uint2*>(
                o_pre + ((static_cast<long long>(h) * S_pre + s) * lq + prow) * D + 4 * lane);
            x[u] = make_float4(attn::bf16_lo(raw.x), attn::bf16_hi(raw.x), attn::bf16_lo(raw.y),
                               attn::bf16_hi(raw.y));
          } else {
            x[u] = *reinterpret_cast<const float4*>(
                o_suf + (static_cast<long long>(r) * S_suf + (s - S_pre)) * D + 4 * lane);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = __shfl_sync(kFull, wl, (j0 + u) & 31);
          if (j0 + u >= n) break;
          acc.x = fmaf(w, x[u].x, acc.x);
          acc.y = fmaf(w, x[u].y, acc.y);
          acc.z = fmaf(w, x[u].z, acc.z);
          acc.w = fmaf(w, x[u].w, acc.w);
        }
      }
    }
  }
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
  const uint2 packed = make_uint2(attn::pack_bf16x2(acc.x * inv, acc.y * inv),
                                  attn::pack_bf16x2(acc.z * inv, acc.w * inv));
  *reinterpret_cast<uint2*>(o + static_cast<long long>(r) * D + 4 * lane) = packed;
  if (lane == 0 && lse != nullptr) lse[r] = empty ? -INFINITY : big + logf(wsum);
}

}  // namespace

namespace attn_host {

attn_status_t launch_cascade_gather_q(const void* q, void* q_stack, int B, int Hq, int Hkv, int d,
                                      cudaStream_t stream) {
  const int chunks_per_group = (Hq / Hkv) * d * 2 / 16;
  const long long total = static_cast<long long>(B) * Hkv * chunks_per_group;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;
  cascade_gather_q_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(q), static_cast<uint4*>(q_stack), B, Hq, Hkv, chunks_per_group);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_cascade_merge(const void* o_pre, const float* lse_pre, int S_pre,
                                   const float* o_suf, const float* lse_suf, int S_suf, int B,
                                   int Hq, int Hkv, int d, void* o, float* lse,
                                   cudaStream_t stream) {
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const int rows = B * Hq;
  cascade_merge_kernel<<<(rows + kRowsPerBlock - 1) / kRowsPerBlock, kRowsPerBlock * 32, 0,
                         stream>>>(static_cast<const __nv_bfloat16*>(o_pre), lse_pre, S_pre, o_suf,
                                   lse_suf, S_suf, B, Hq, Hkv, static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
