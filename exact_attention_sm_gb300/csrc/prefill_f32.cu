// fp32 exact attention on CUDA cores.  TF32 tensor cores (10-bit mantissa)
// cannot hold O to 1e-4, so every product here is a full fp32 FMA.
//
// What is computed ("10.3 FlashAttention: IO-aware algorithm design", 10.3.2;
// "FlashAttention tiling, online softmax and IO" blog, sections 03 and 06):
// per query row, S = q K^T * scale, the running max m and sum l of the online
// softmax over key blocks, O = sum_j e^(s_j - m) v_j / l and LSE = m + ln l.
// Scores are kept in base 2 (log2 e folded into the scale), so
// LSE = (m2 + log2 l) * ln 2.
//
// Work decomposition (warp-cooperative; designed for GB300's 32-wide warps):
//   * A CTA is 4 warps and owns 32 consecutive query rows of one (b, h):
//     8 rows per warp.  The rows' pre-scaled q vectors sit in shared memory
//     and are read as broadcasts.
//   * Keys stream in blocks of 32 through a two-stage shared-memory ring
//     filled with cp.async (16-byte copies, zero-filled past Lk).
//   * Score phase: lane i owns key i of the block and computes its 8 scores
//     (one per row of the warp) against its own K row (K rows are padded by
//     four floats so the 128-bit loads of 8 lanes hit 32 distinct banks).
//   * Block max: 5-step butterfly of warp shuffles per row.  The sum l is kept
//     per lane (the lane's keys only) and reduced once at the end.
//   * PV phase: lane c owns output columns [c D/32, (c+1) D/32); the block's
//     probabilities go through a per-warp shared array and are read back as
//     broadcasts while each lane walks the 32 V rows.
// Causal: key blocks past the CTA's last row are not loaded; a warp skips the
// blocks past its own last row and masks keys j > row element-wise.
#include "common.cuh"

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 8;
constexpr int kRows = kWarps * kRowsPerWarp;  // query rows per CTA
constexpr int kKeys = 32;                     // keys per block (one per lane)

template <int D>
struct F32Smem {
  static constexpr int KP = D + 4;  // padded K row (floats)
  static constexpr int Q_FLOATS = kRows * D;
  static constexpr int K_FLOATS = kKeys * KP;
  static constexpr int V_FLOATS = kKeys * D;
  static constexpr int P_FLOATS = kWarps * kRowsPerWarp * kKeys;
  static constexpr int BYTES = 4 * (Q_FLOATS + 2 * K_FLOATS + 2 * V_FLOATS + P_FLOATS);
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_le1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) prefill_f32_rows_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    float* __restrict__ o, float* __restrict__ lse, int Hq, int Hkv, int Lq, int Lk, int causal,
    float scale_log2) {
  using S = F32Smem<D>;
  constexpr int CPL = D / 32;  // output columns per lane
  constexpr int R = kRowsPerWarp;
  extern __shared__ __align__(16) float f32_smem[];
  float* qs = f32_smem;                   // [kRows][D]
  float* ks = qs + S::Q_FLOATS;           // [2][kKeys][KP]
  float* vs = ks + 2 * S::K_FLOATS;       // [2][kKeys][D]
  float* ps = vs + 2 * S::V_FLOATS;       // [kWarps][R][kKeys]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (Hq / Hkv);
  const int row0 = blockIdx.x * kRows;          // first row of the CTA
  const int wrow0 = row0 + warp * R;            // first row of this warp
  const size_t qh = static_cast<size_t>(b) * Hq + h;
  const float* kbase = k + (static_cast<size_t>(b) * Hkv + kvh) * Lk * D;
  const float* vbase = v + (static_cast<size_t>(b) * Hkv + kvh) * Lk * D;

  // Key blocks the CTA reads, and the last one this warp needs.
  const int cta_kend = causal ? min(Lk, row0 + kRows) : Lk;
  const int nblk = (cta_kend + kKeys - 1) / kKeys;
  const int warp_kend = causal ? min(Lk, wrow0 + R) : Lk;
  const int wblk = (warp_kend + kKeys - 1) / kKeys;

  auto load_block = [&](int blk) {
    float* kd = ks + (blk & 1) * S::K_FLOATS;
    float* vd = vs + (blk & 1) * S::V_FLOATS;
    constexpr int CHUNKS = kKeys * D / 4;  // 16-byte pieces per K (or V) block
    for (int c = threadIdx.x; c < CHUNKS; c += kWarps * 32) {
      const int r = c / (D / 4), col = (c % (D / 4)) * 4;
      const int key = blk * kKeys + r;
      const bool ok = key < Lk;
      const size_t off = static_cast<size_t>(ok ? key : 0) * D + col;
      cp_async16(kd + r * S::KP + col, kbase + off, ok);
      cp_async16(vd + r * D + col, vbase + off, ok);
    }
    cp_async_commit();
  };

  if (nblk > 0) load_block(0);
  // Pre-scaled query rows (rows past Lq read as zeros).
  for (int c = threadIdx.x; c < kRows * D / 4; c += kWarps * 32) {
    const int r = c / (D / 4), col = (c % (D / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < Lq) x = *reinterpret_cast<const float4*>(q + (qh * Lq + row0 + r) * D + col);
    x.x *= scale_log2;
    x.y *= scale_log2;
    x.z *= scale_log2;
    x.w *= scale_log2;
    *reinterpret_cast<float4*>(qs + r * D + col) = x;
  }

  float m[R], lpart[R], acc[R][CPL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    lpart[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[r][c] = 0.f;
  }
  const float* qw = qs + warp * R * D;
  float* pw = ps + warp * R * kKeys;

  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + 1 < nblk) {
      load_block(blk + 1);
      cp_async_wait_le1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();  // block blk (and the q rows) visible to every warp
    if (blk < wblk) {
      const float* kd = ks + (blk & 1) * S::K_FLOATS + lane * S::KP;
      const float* vd = vs + (blk & 1) * S::V_FLOATS;
      // Scores of key `lane` against the warp's R rows.
      float s[R];
#pragma unroll
      for (int r = 0; r < R; ++r) s[r] = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float kr[32];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 t = *reinterpret_cast<const float4*>(kd + c0 + c);
          kr[c] = t.x;
          kr[c + 1] = t.y;
          kr[c + 2] = t.z;
          kr[c + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(qw + r * D + c0 + c);
            s[r] = fmaf(qv.x, kr[c], s[r]);
            s[r] = fmaf(qv.y, kr[c + 1], s[r]);
            s[r] = fmaf(qv.z, kr[c + 2], s[r]);
            s[r] = fmaf(qv.w, kr[c + 3], s[r]);
          }
        }
      }
      const int key = blk * kKeys + lane;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool visible = key < Lk && (!causal || key <= wrow0 + r);
        const float sr = visible ? s[r] : -INFINITY;
        const float m_new = fmaxf(m[r], warp_max(sr));
        // A row with no visible key so far keeps m = -inf; its p are 0.
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m[r] - m_use);  // 1 when m is unchanged, 0 from -inf
        const float p = exp2f(sr - m_use);
        lpart[r] = lpart[r] * alpha + p;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[r][c] *= alpha;
        m[r] = m_new;
        pw[r * kKeys + lane] = p;
      }
      __syncwarp();
      // O += P V: lane owns columns [lane CPL, lane CPL + CPL).
#pragma unroll 4
      for (int j = 0; j < kKeys; j += 4) {
        float vr[4][CPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float* vrow = vd + (j + u) * D + lane * CPL;
          if constexpr (CPL == 4) {
            const float4 t = *reinterpret_cast<const float4*>(vrow);
            vr[u][0] = t.x;
            vr[u][1] = t.y;
            vr[u][2] = t.z;
            vr[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(vrow);
            vr[u][0] = t.x;
            vr[u][1] = t.y;
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 p4 = *reinterpret_cast<const float4*>(pw + r * kKeys + j);
          const float pj[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[r][c] = fmaf(pj[u], vr[u][c], acc[r][c]);
        }
      }
      __syncwarp();  // the next block's p overwrite pw only after every lane read it
    }
    __syncthreads();  // the ring slot of block blk may be refilled
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float l = warp_sum(lpart[r]);
    const int row = wrow0 + r;
    if (row >= Lq) continue;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* orow = o + (qh * Lq + row) * D + lane * CPL;
    if constexpr (CPL == 4) {
      *reinterpret_cast<float4*>(orow) =
          make_float4(acc[r][0] * inv, acc[r][1] * inv, acc[r][2] * inv, acc[r][3] * inv);
    } else {
      *reinterpret_cast<float2*>(orow) = make_float2(acc[r][0] * inv, acc[r][1] * inv);
    }
    if (lse != nullptr && lane == 0)
      lse[qh * Lq + row] = l > 0.f ? (m[r] + log2f(l)) * attn::kLn2 : -INFINITY;
  }
}

template <int D>
attn_status_t launch_rows(const float* q, const float* k, const float* v, float* o, float* lse,
                          int B, int Hq, int Hkv, int Lq, int Lk, int causal, float scale,
                          cudaStream_t stream) {
  constexpr int smem = F32Smem<D>::BYTES;
  static bool attr_set[64] = {};  // kernel attributes are per device
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return ATTN_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_f32_rows_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set[dev] = true;
  }
  const dim3 grid((Lq + kRows - 1) / kRows, Hq, B);
  prefill_f32_rows_kernel<D><<<grid, kWarps * 32, smem, stream>>>(
      q, k, v, o, lse, Hq, Hkv, Lq, Lk, causal, scale * attn::kLog2e);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

attn_status_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                 int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                 float scale, cudaStream_t stream) {
  if (d == 64) return launch_rows<64>(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, causal, scale, stream);
  if (d == 128) return launch_rows<128>(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, causal, scale, stream);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn_host
