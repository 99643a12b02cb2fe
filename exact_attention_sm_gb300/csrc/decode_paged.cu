// Paged grouped-query decode attention, bf16, head dim 128, on CUDA cores.
//
// Follows "FlashAttention and inference operators" (CUDA advanced handbook):
// "PagedAttention" (token t lives in page block_table[t / 16], slot t % 16),
// "Flash-Decoding and split-K" (each CTA owns one segment of the context and
// emits a normalised partial output plus its LSE), and the improvements that
// chapter lists for its teaching kernel: one CTA serves every query head that
// shares a KV head so each K/V byte is read once (the GQA exercise), 128-bit
// loads converted to fp32 in registers, and online softmax while scanning with
// no score buffer in shared memory.
//
// Work decomposition.  CTA = (segment s, KV head, request b), 4 warps.  The
// segment's pages are dealt round-robin to the warps; each warp keeps its own
// online-softmax state and the 4 states are merged at the end.  Inside a warp
// the two half-warps take the even / odd slots of a page and lane l (of 16)
// owns dims [8l, 8l+8): one 16-byte load per lane and token, a 256-byte
// contiguous row per half-warp.  The partial dot products of the 8 tokens x HG
// heads of a half-warp are reduced across its 16 lanes with a transposed
// butterfly (each step halves the values a lane carries), which needs far
// fewer shuffles than reducing each value separately; the probabilities are
// then gathered back to every lane for the P.V update.
#include "common.cuh"

namespace {

constexpr int D = 128;
constexpr int PAGE = 16;
constexpr int NW = 4;  // warps per CTA
constexpr unsigned FULL = 0xffffffffu;

template <int HG>
struct Lanes {
  static constexpr int NV = 8 * HG;                  // (token, head) values per half-warp per page
  static constexpr int NF = NV >= 16 ? NV / 16 : 1;  // values a lane holds after the reduction
};

// Transposed butterfly over the 16 lanes of a half-warp.  On return lane l16
// holds the full sums of value indices idx(l16, e), e < NF:
//   HG=4: idx = 2*l16 + e;  HG=2: idx = l16;  HG=1: idx = l16 >> 1.
template <int NV>
__device__ __forceinline__ void transposed_reduce(float (&v)[NV], int l16) {
  int n = NV;
#pragma unroll
  for (int bit = 3; bit >= 0; --bit) {
    const int off = 1 << bit;
    if (n >= 2) {
      const bool upper = (l16 >> bit) & 1;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? v[i] : v[i + n / 2];
          const float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(FULL, send, off);
        }
      }
      n /= 2;
    } else {
      v[0] += __shfl_xor_sync(FULL, v[0], off);
    }
  }
}

template <int HG>
__device__ __forceinline__ int value_index(int l16, int e) {
  if (HG == 4) return 2 * l16 + e;
  if (HG == 2) return l16;
  return l16 >> 1;
}

// Lane (within the half-warp) that holds value x after transposed_reduce, and
// which of its NF registers.
template <int HG>
__device__ __forceinline__ int owner_lane(int x) {
  if (HG == 4) return x >> 1;
  if (HG == 2) return x;
  return x << 1;
}

// Reduce over the lanes that hold the same head (and across both halves).
template <int HG, bool IS_MAX>
__device__ __forceinline__ float head_allreduce(float x) {
  constexpr int kBits = HG == 4 ? 2 : (HG == 2 ? 3 : 4);  // low lane bits that do not select the head
#pragma unroll
  for (int bit = 0; bit < kBits; ++bit) {
    const float y = __shfl_xor_sync(FULL, x, 1 << bit);
    x = IS_MAX ? fmaxf(x, y) : x + y;
  }
  const float y = __shfl_xor_sync(FULL, x, 16);
  return IS_MAX ? fmaxf(x, y) : x + y;
}

template <int HG>
__device__ __forceinline__ int lane_of_head(int h) {
  return HG == 4 ? 4 * h : (HG == 2 ? 8 * h : 0);
}

template <int HG>
__global__ void __launch_bounds__(NW * 32) decode_bf16_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_pages,
    const __nv_bfloat16* __restrict__ v_pages, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ seq_lens, int chunk, int max_splits,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, float* __restrict__ part_o,
    float* __restrict__ part_lse, int Hq, int Hkv, int max_pages, int num_pages,
    float scale_log2, int* status) {
  using L = Lanes<HG>;
  constexpr int NV = L::NV, NF = L::NF;
  __shared__ float sm_m[NW][HG];
  __shared__ float sm_l[NW][HG];
  __shared__ __align__(16) float sm_acc[NW][HG][D];

  const int s = blockIdx.x;
  const int group = Hq / Hkv;
  const int groups_per_kvh = group / HG;
  const int kvh = blockIdx.y / groups_per_kvh;
  const int h0 = kvh * group + (blockIdx.y % groups_per_kvh) * HG;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;

  const int len = seq_lens[b];
  const int t_begin = s * chunk;
  const int t_end = min(len, t_begin + chunk);

  float qf[HG][8];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const uint4 w = *reinterpret_cast<const uint4*>(q + ((size_t)b * Hq + h0 + h) * D + 8 * l16);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qf[h][2 * j] = attn::bf16_lo(ws[j]) * scale_log2;
      qf[h][2 * j + 1] = attn::bf16_hi(ws[j]) * scale_log2;
    }
  }

  float acc[HG][8];
  float m_run[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m_run[h] = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[h][j] = 0.f;
  }
  float l_own = 0.f;
  const int own_h = value_index<HG>(l16, 0) / 8;

  const size_t slot_stride = (size_t)Hkv * D;
  const int p_begin = t_begin / PAGE;
  const int p_end = t_end > t_begin ? (t_end + PAGE - 1) / PAGE : p_begin;

  for (int p = p_begin + warp; p < p_end; p += NW) {
    const int page = block_table[(size_t)b * max_pages + p];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
      continue;
    }
    const size_t base = ((size_t)page * PAGE * Hkv + kvh) * D + 8 * l16;
    uint4 kr[8], vr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) kr[i] = attn::ld_stream_v4(k_pages + base + (2 * i + half) * slot_stride);
#pragma unroll
    for (int i = 0; i < 8; ++i) vr[i] = attn::ld_stream_v4(v_pages + base + (2 * i + half) * slot_stride);

    float part[NV];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t ks[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
      float kf[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kf[2 * j] = attn::bf16_lo(ks[j]);
        kf[2 * j + 1] = attn::bf16_hi(ks[j]);
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaf(qf[h][j], kf[j], a);
        part[h * 8 + i] = a;
      }
    }
    transposed_reduce<NV>(part, l16);

    const int valid = t_end - p * PAGE;  // slots < valid hold tokens of this segment (>= 1)
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < NF; ++e) {
      const int slot = 2 * (value_index<HG>(l16, e) % 8) + half;
      if (slot >= valid) part[e] = -INFINITY;
      mx = fmaxf(mx, part[e]);
    }
    mx = head_allreduce<HG, true>(mx);

    float m_own = 0.f;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float pm = __shfl_sync(FULL, mx, lane_of_head<HG>(h));
      const float m_new = fmaxf(m_run[h], pm);
      const float alpha = exp2f(m_run[h] - m_new);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[h][j] *= alpha;
      if (h == own_h) {
        l_own *= alpha;
        m_own = m_new;
      }
      m_run[h] = m_new;
    }
    float pv[NF];
#pragma unroll
    for (int e = 0; e < NF; ++e) {
      pv[e] = exp2f(part[e] - m_own);
      if (HG > 1 || (l16 & 1) == 0) l_own += pv[e];
    }

    if (valid < PAGE) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (2 * i + half >= valid) vr[i] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t vs[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
      float vf[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        vf[2 * j] = attn::bf16_lo(vs[j]);
        vf[2 * j + 1] = attn::bf16_hi(vs[j]);
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const int x = h * 8 + i;
        const float pw = __shfl_sync(FULL, pv[NF > 1 ? (x & 1) : 0], (lane & 16) | owner_lane<HG>(x));
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[h][j] = fmaf(pw, vf[j], acc[h][j]);
      }
    }
  }

  // Combine the two half-warps (same dims, different slots), then the warps.
#pragma unroll
  for (int h = 0; h < HG; ++h)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[h][j] += __shfl_xor_sync(FULL, acc[h][j], 16);
  const float l_head = head_allreduce<HG, false>(l_own);
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const float lh = __shfl_sync(FULL, l_head, lane_of_head<HG>(h));
    if (lane == 0) {
      sm_m[warp][h] = m_run[h];
      sm_l[warp][h] = lh;
    }
    if (half == 0) {
      *reinterpret_cast<float4*>(&sm_acc[warp][h][8 * l16]) =
          make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      *reinterpret_cast<float4*>(&sm_acc[warp][h][8 * l16 + 4]) =
          make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
  }
  __syncthreads();

  const int t = threadIdx.x;  // output dim
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    float big = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) big = fmaxf(big, sm_m[w][h]);
    float lsum = 0.f, osum = 0.f;
    if (big != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float c = exp2f(sm_m[w][h] - big);
        lsum = fmaf(c, sm_l[w][h], lsum);
        osum = fmaf(c, sm_acc[w][h][t], osum);
      }
    }
    const bool empty = !(lsum > 0.f);
    const float out = empty ? 0.f : osum / lsum;
    const float row_lse = empty ? -INFINITY : (big + log2f(lsum)) * attn::kLn2;
    const size_t row = (size_t)b * Hq + h0 + h;
    if (max_splits == 1) {
      o[row * D + t] = __float2bfloat16_rn(out);
      if (t == 0 && lse != nullptr) lse[row] = row_lse;
    } else {
      part_o[(row * max_splits + s) * D + t] = out;
      if (t == 0) part_lse[row * max_splits + s] = row_lse;
    }
  }
}

}  // namespace

namespace attn_host {

int decode_ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel<4>, NW * 32, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

attn_status_t launch_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* seq_lens, int page_size,
                                 int chunk, int max_splits, void* o, float* lse, float* part_o,
                                 float* part_lse, int B, int Hq, int Hkv, int d, int max_pages,
                                 int num_pages, float scale, cudaStream_t stream) {
  if (d != D || page_size != PAGE) return ATTN_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  const int hg = group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1);
  dim3 grid(max_splits, Hkv * (group / hg), B);
  int* st = device_status_ptr();
  const float sl2 = scale * attn::kLog2e;
  auto args = [&](auto kern) {
    kern<<<grid, NW * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_pages),
        static_cast<const __nv_bfloat16*>(v_pages), block_table, seq_lens, chunk, max_splits,
        static_cast<__nv_bfloat16*>(o), lse, part_o, part_lse, Hq, Hkv, max_pages, num_pages, sl2,
        st);
  };
  if (hg == 4)
    args(decode_bf16_kernel<4>);
  else if (hg == 2)
    args(decode_bf16_kernel<2>);
  else
    args(decode_bf16_kernel<1>);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
