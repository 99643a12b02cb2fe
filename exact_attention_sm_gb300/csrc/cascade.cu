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
#include <type_traits>

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
constexpr int kBatch = 24;        // states whose O slices are in flight at once
constexpr unsigned kFull = 0xffffffffu;

// One warp per output row (lane l owns dims DL l .. DL l + DL - 1, DL = D /
// 32).  The row's S = S_pre + S_suf states are numbered prefix chunks first,
// then suffix segments.  The row is latency-bound (a few KB per row), so
// every load it needs is issued before any is used: the O slices of the
// first kBatch states and the LSEs of the first 32 go out together, and the
// max is reduced while they are in flight.  The weighted sum of the O_s and
// the weight sum run over s in ascending order, so the result depends on
// (S_pre, S_suf) alone.
template <int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
    cascade_merge_kernel(const __nv_bfloat16* __restrict__ o_pre, const float* __restrict__ lse_pre,
                         int S_pre, const float* __restrict__ o_suf,
                         const float* __restrict__ lse_suf, int S_suf, int B, int Hq, int Hkv,
                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int DL = D / 32;
  static_assert(DL == 2 || DL == 4, "d = 64 or 128");
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
  // The lane's DL dims of state s as raw words (bf16 pairs for a prefix
  // state, fp32 bits for a suffix state), converted only where they are
  // used, so that every load of a batch is in flight before the first use.
  using Raw = typename std::conditional<DL == 4, uint4, uint2>::type;
  auto load_o = [&](int s) {
    Raw x;
    if (s < S_pre) {
      const __nv_bfloat16* src =
          o_pre + ((static_cast<long long>(h) * S_pre + s) * lq + prow) * D + DL * lane;
      if constexpr (DL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        x = make_uint4(w.x, w.y, 0u, 0u);
      } else {
        x = make_uint2(*reinterpret_cast<const uint32_t*>(src), 0u);
      }
    } else {
      const float* src = o_suf + (static_cast<long long>(r) * S_suf + (s - S_pre)) * D + DL * lane;
      x = *reinterpret_cast<const Raw*>(src);
    }
    return x;
  };
  auto to_float = [&](int s, const Raw& x, float (&f)[DL]) {
    if constexpr (DL == 4) {
      if (s < S_pre) {
        f[0] = attn::bf16_lo(x.x); f[1] = attn::bf16_hi(x.x);
        f[2] = attn::bf16_lo(x.y); f[3] = attn::bf16_hi(x.y);
      } else {
        f[0] = __uint_as_float(x.x); f[1] = __uint_as_float(x.y);
        f[2] = __uint_as_float(x.z); f[3] = __uint_as_float(x.w);
      }
    } else {
      if (s < S_pre) {
        f[0] = attn::bf16_lo(x.x); f[1] = attn::bf16_hi(x.x);
      } else {
        f[0] = __uint_as_float(x.x); f[1] = __uint_as_float(x.y);
      }
    }
  };

  Raw x[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    if (u < S) x[u] = load_o(u);
  const float ls0 = lane < S ? state_lse(lane) : -INFINITY;
  float big = ls0;
  for (int s = lane + 32; s < S; s += 32) big = fmaxf(big, state_lse(s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(kFull, big, off));

  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (big != -INFINITY) {
    const float wl = ls0 == -INFINITY ? 0.f : expf(ls0 - big);  // weight of state `lane`
    for (int s0 = 0; s0 < S; s0 += kBatch) {
      if (s0 > 0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (s0 + u < S) x[u] = load_o(s0 + u);
      }
      // Empty states hold O = 0 (both producers write it) and weigh 0.
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int s = s0 + u;  // warp-uniform
        if (s >= S) break;
        float w;
        if (s < 32) {
          w = __shfl_sync(kFull, wl, s);
        } else {
          const float l = state_lse(s);
          w = l == -INFINITY ? 0.f : expf(l - big);
        }
        float v[DL];
        to_float(s, x[u], v);
        wsum += w;
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] = fmaf(w, v[e], acc[e]);
      }
    }
  }
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
  if constexpr (DL == 4) {
    *reinterpret_cast<uint2*>(o + static_cast<long long>(r) * D + DL * lane) =
        make_uint2(attn::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                   attn::pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(o + static_cast<long long>(r) * D + DL * lane) =
        attn::pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
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
  if (d != 128 && d != 64) return ATTN_ERR_UNSUPPORTED;
  const int rows = B * Hq;
  auto kernel = d == 64 ? cascade_merge_kernel<64> : cascade_merge_kernel<128>;
  kernel<<<(rows + kRowsPerBlock - 1) / kRowsPerBlock, kRowsPerBlock * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o_pre), lse_pre, S_pre, o_suf, lse_suf, S_suf, B, Hq, Hkv,
      static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
