// fp32 prefill attention on CUDA cores (no tensor cores: TF32's 10-bit
// mantissa cannot meet a 1e-4 bound on O).
//
// FlashAttention-2 loop order ("10.3 FlashAttention: IO-aware algorithm
// design", 10.3.2 tiled forward): a CTA owns BR query rows of one (b, h) and
// streams K/V tiles of BC keys through shared memory; each thread owns one
// query row and keeps its online-softmax state (m, l, O~) in registers
// ("FlashAttention tiling, online softmax and IO" blog, section 03).  Scores
// live in the base-2 domain: s2 = (q . k) * scale * log2(e), so that
// p = exp2(s2 - m2) and LSE = (m2 + log2 l) * ln 2.  Causal: K/V tiles past
// the CTA's last row are never loaded; the diagonal tile is masked per element
// (blog section 06).
#include "common.cuh"

namespace {

constexpr int BR = 64;  // query rows per CTA (one per thread)

template <int D, int BC>
__global__ void __launch_bounds__(BR) prefill_f32_kernel(const float* __restrict__ q,
                                                         const float* __restrict__ k,
                                                         const float* __restrict__ v,
                                                         float* __restrict__ o,
                                                         float* __restrict__ lse, int Hq, int Hkv,
                                                         int Lq, int Lk, int causal,
                                                         float scale_log2) {
  __shared__ __align__(16) float Ks[BC][D];
  __shared__ __align__(16) float Vs[BC][D];

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / (Hq / Hkv);
  const int row = tile * BR + threadIdx.x;
  const bool live_row = row < Lq;

  const float* qp = q + ((size_t)(b * Hq + h) * Lq + (live_row ? row : 0)) * D;
  const float* kp = k + (size_t)(b * Hkv + kvh) * Lk * D;
  const float* vp = v + (size_t)(b * Hkv + kvh) * Lk * D;

  float qr[D];
#pragma unroll
  for (int j = 0; j < D; j += 4) {
    float4 t = *reinterpret_cast<const float4*>(qp + j);
    qr[j] = t.x * scale_log2;
    qr[j + 1] = t.y * scale_log2;
    qr[j + 2] = t.z * scale_log2;
    qr[j + 3] = t.w * scale_log2;
  }
  float acc[D];
#pragma unroll
  for (int j = 0; j < D; ++j) acc[j] = 0.f;
  float m2 = -INFINITY, l = 0.f;

  // Keys this CTA can see: all of them, or up to its last row when causal.
  int kv_end = Lk;
  if (causal) kv_end = min(Lk, (tile + 1) * BR);

  for (int j0 = 0; j0 < kv_end; j0 += BC) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < BC * D / 4; idx += BR) {
      const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
      float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
      if (j0 + r < Lk) {
        kk = *reinterpret_cast<const float4*>(kp + (size_t)(j0 + r) * D + c);
        vv = *reinterpret_cast<const float4*>(vp + (size_t)(j0 + r) * D + c);
      }
      *reinterpret_cast<float4*>(&Ks[r][c]) = kk;
      *reinterpret_cast<float4*>(&Vs[r][c]) = vv;
    }
    __syncthreads();

    float s[BC];
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < BC; ++c) {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < D; j += 2) {
        acc0 = fmaf(qr[j], Ks[c][j], acc0);
        acc1 = fmaf(qr[j + 1], Ks[c][j + 1], acc1);
      }
      const int key = j0 + c;
      const bool visible = key < Lk && (!causal || key <= row);
      s[c] = visible ? acc0 + acc1 : -INFINITY;
      tmax = fmaxf(tmax, s[c]);
    }
    const float m_new = fmaxf(m2, tmax);
    if (m_new == -INFINITY) continue;  // nothing visible yet in this row
    const float corr = exp2f(m2 - m_new);  // exp2(-inf) = 0 on the first visible tile
    l *= corr;
#pragma unroll
    for (int j = 0; j < D; ++j) acc[j] *= corr;
#pragma unroll
    for (int c = 0; c < BC; ++c) {
      const float p = exp2f(s[c] - m_new);
      l += p;
#pragma unroll
      for (int j = 0; j < D; ++j) acc[j] = fmaf(p, Vs[c][j], acc[j]);
    }
    m2 = m_new;
  }

  if (!live_row) return;
  float* op = o + ((size_t)(b * Hq + h) * Lq + row) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int j = 0; j < D; j += 4) {
    *reinterpret_cast<float4*>(op + j) =
        make_float4(acc[j] * inv, acc[j + 1] * inv, acc[j + 2] * inv, acc[j + 3] * inv);
  }
  if (lse != nullptr) {
    lse[(size_t)(b * Hq + h) * Lq + row] =
        l > 0.f ? (m2 + log2f(l)) * attn::kLn2 : -INFINITY;
  }
}

}  // namespace

namespace attn_host {

attn_status_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                 int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                 float scale, cudaStream_t stream) {
  dim3 grid((Lq + BR - 1) / BR, Hq, B);
  const float sl2 = scale * attn::kLog2e;
  if (d == 64) {
    prefill_f32_kernel<64, 32><<<grid, BR, 0, stream>>>(q, k, v, o, lse, Hq, Hkv, Lq, Lk, causal, sl2);
  } else if (d == 128) {
    prefill_f32_kernel<128, 16><<<grid, BR, 0, stream>>>(q, k, v, o, lse, Hq, Hkv, Lq, Lk, causal, sl2);
  } else {
    return ATTN_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
