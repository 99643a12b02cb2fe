// Paged grouped-query decode attention, bf16, head dim 128 or 64.
//
// Follows "FlashAttention and inference operators" (CUDA advanced handbook):
// "PagedAttention" (token t lives in page block_table[t / 16], slot t % 16),
// "Flash-Decoding and split-K" (each CTA owns one segment of the context and
// emits a normalised partial output plus its LSE), and the improvements that
// chapter lists for its teaching kernel: one CTA serves every query head that
// shares a KV head so each K/V byte is read once (the GQA exercise), 128-bit
// bf16 reads with fp32 arithmetic, and online softmax while scanning with no
// score buffer.
//
// GB300 layout.  CTA = (segment, KV head [x head group], request) with one
// producer warp and 4 consumer warps:
//   * producer: walks the segment's block-table entries (read 32 at a time by
//     the warp) and, per page, issues two 4-D TMA copies (the page's 16 K rows
//     and 16 V rows of this KV head, 4 KB each) into an 8-stage shared-memory
//     ring guarded by mbarriers.  Up to 64 KB per CTA are in flight, which is
//     what keeps HBM busy; an out-of-range table entry is reported in the
//     device status word and its page is treated as empty (never read).
//   * consumers: page i of the segment goes to consumer warp i % 4.  Inside a
//     warp, 4 groups of 8 lanes each take one token at a time and lane l (of
//     8) owns dims [l d/8, (l+1) d/8): two 16-byte shared loads per row at
//     d = 128, one at d = 64 (whose ring has twice the stages, so the same
//     64 KB per CTA are in flight).  Scores
//     use the mixed-precision FMA (bf16 x bf16 + fp32), so neither q nor K is
//     converted; the 4 tokens x HG heads partial dot products of a group are
//     reduced over its 8 lanes with a transposed butterfly (each step halves
//     the values a lane carries), and the probabilities, rounded to bf16 like
//     the tensor-core path's P, come back with one shuffle per pair of tokens.
//   * online softmax in the base-2 domain with a conditional rescale: the
//     running max only moves when a page's max exceeds it by more than 8, so
//     the accumulators are rarely rescaled (the result is unchanged because
//     l and O share the same stale max).
//   * at the end the 4 consumer warps' states are merged in shared memory
//     (the LSE merge within the CTA) and the CTA writes the final O and LSE
//     (one segment) or its normalised partial state for the merge kernel.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace {

using namespace sm103;

constexpr int D = 128;                      // the balanced kernel's head dim
constexpr int PAGE = 16;
constexpr int NCW = 4;                      // consumer warps
constexpr int HG = 4;                       // query heads per CTA (padded when the group is smaller)
constexpr int NUM_THREADS = 32 * (NCW + 1);
constexpr int NST = 8;                      // ring stages (one page of K and V each)
constexpr int PAGE_BYTES = PAGE * D * 2;    // 4 KB: 16 rows of one KV head
constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;

// Head-dim dependent sizes of the plain decode kernel: DL dims per lane
// (two or one 16-byte loads of a row), ring stages so that 64 KB are in
// flight per CTA whatever d is.
template <int DD>
struct DecCfg {
  static constexpr int DL = DD / 8;
  static constexpr int WPL = DL / 2;                    // bf16 pairs per lane and row
  static constexpr int PAGE_BYTES = PAGE * DD * 2;
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int NST = 8 * 128 / DD;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;
};
static_assert(DecCfg<128>::SMEM_BYTES == SMEM_BYTES && DecCfg<64>::SMEM_BYTES == SMEM_BYTES,
              "the same ring bytes at both head dims");
constexpr unsigned FULL = 0xffffffffu;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// acc + lo/hi bf16 halves of a * lo/hi bf16 halves of b, fp32 accumulate.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
// p (the low / high bf16 half of pw) times both bf16 halves of v, fp32 accumulate.
__device__ __forceinline__ void fma_plo_v(uint32_t pw, uint32_t v, float& c0, float& c1) {
  asm("{\n\t.reg .b16 pl, ph, vl, vh;\n\tmov.b32 {pl, ph}, %2;\n\tmov.b32 {vl, vh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, pl, vl, %0;\n\tfma.rn.f32.bf16 %1, pl, vh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(pw), "r"(v));
}
__device__ __forceinline__ void fma_phi_v(uint32_t pw, uint32_t v, float& c0, float& c1) {
  asm("{\n\t.reg .b16 pl, ph, vl, vh;\n\tmov.b32 {pl, ph}, %2;\n\tmov.b32 {vl, vh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, ph, vl, %0;\n\tfma.rn.f32.bf16 %1, ph, vh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(pw), "r"(v));
}

// Compact grid of a split plan: request b owns the off[b + 1] - off[b]
// segment CTAs blockIdx.x = off[b] .. off[b + 1] - 1 (n = B), so requests
// shorter than the longest launch no empty CTAs.  n = 0: the plain grid
// (segment, KV head group, request).
constexpr int kSegMapMax = 512;
struct SegMap {
  int n;
  int off[kSegMapMax + 1];
};

// One page of K and V (16 tokens, the first `valid` of them live) against
// the query rows in qw: scores, online softmax in base 2 and P V into the
// lane's accumulators (lane layout as described at the top of the file).
template <int DD>
__device__ __forceinline__ void consume_page(const uint8_t* kst, const uint8_t* vst, int valid,
                                             const uint32_t (&qw)[HG][DecCfg<DD>::WPL],
                                             float (&acc)[HG][DecCfg<DD>::DL], float (&m_run)[HG],
                                             float& l_own, float scale_log2, int lane, int grp,
                                             int l8, int own_h) {
    constexpr int WPL = DecCfg<DD>::WPL, DL = DecCfg<DD>::DL, RS = DD * 2;  // RS: row bytes

    // Partial dots of this lane's DL dims: value index x = h * 4 + tt.
    float part[HG * 4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int slot = grp + 4 * tt;
      uint32_t kw[WPL];
#pragma unroll
      for (int c = 0; c < WPL / 4; ++c) {
        const uint4 k4 = *reinterpret_cast<const uint4*>(kst + slot * RS + 16 * c);
        kw[4 * c] = k4.x;
        kw[4 * c + 1] = k4.y;
        kw[4 * c + 2] = k4.z;
        kw[4 * c + 3] = k4.w;
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < WPL; ++w) {
          a0 = fma_bf16_lo(qw[h][w], kw[w], a0);
          a1 = fma_bf16_hi(qw[h][w], kw[w], a1);
        }
        part[h * 4 + tt] = a0 + a1;
      }
    }
    // Transposed butterfly over the 8 lanes of the group (bits 2, 1, 0).
    {
      int n = HG * 4;
#pragma unroll
      for (int bit = 2; bit >= 0; --bit) {
        const bool upper = (l8 >> bit) & 1;
#pragma unroll
        for (int x = 0; x < HG * 2; ++x) {
          if (x < n / 2) {
            const float send = upper ? part[x] : part[x + n / 2];
            const float keep = upper ? part[x + n / 2] : part[x];
            part[x] = keep + __shfl_xor_sync(FULL, send, 1 << bit);
          }
        }
        n /= 2;
      }
    }
    // Lane now holds x = 2 * l8 + e (e = 0, 1): head l8 / 2, tokens 2 (l8 & 1) + e.
    float sv[2];
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tt = 2 * (l8 & 1) + e;
      sv[e] = (grp + 4 * tt < valid) ? part[e] * scale_log2 : -INFINITY;
      mx = fmaxf(mx, sv[e]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
    float m_own = 0.f;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float pm = __shfl_sync(FULL, mx, 2 * h);
      if (pm > m_run[h] + kRescaleThreshold) {  // warp-uniform
        const float alpha = ex2(m_run[h] - pm);  // 0 on the first page (m_run = -inf)
#pragma unroll
        for (int j = 0; j < DL; ++j) acc[h][j] *= alpha;
        if (h == own_h) l_own *= alpha;
        m_run[h] = pm;
      }
      if (h == own_h) m_own = m_run[h];
    }
    const float p0 = ex2(sv[0] - m_own), p1 = ex2(sv[1] - m_own);
    l_own += p0 + p1;
    const uint32_t pw = attn::pack_bf16x2(p0, p1);

#pragma unroll
    for (int tp = 0; tp < 2; ++tp) {        // token pair (tokens 2tp, 2tp+1)
      uint32_t ph[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) ph[h] = __shfl_sync(FULL, pw, (lane & ~7) | (2 * h + tp));
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tt = 2 * tp + e;
        const int slot = grp + 4 * tt;
        uint32_t vw[WPL];
#pragma unroll
        for (int c = 0; c < WPL / 4; ++c) {
          uint4 v4 = *reinterpret_cast<const uint4*>(vst + slot * RS + 16 * c);
          if (slot >= valid) v4 = make_uint4(0u, 0u, 0u, 0u);  // rows past the segment may hold anything
          vw[4 * c] = v4.x;
          vw[4 * c + 1] = v4.y;
          vw[4 * c + 2] = v4.z;
          vw[4 * c + 3] = v4.w;
        }
#pragma unroll
        for (int h = 0; h < HG; ++h)
#pragma unroll
          for (int w = 0; w < WPL; ++w) {
            if (e == 0) fma_plo_v(ph[h], vw[w], acc[h][2 * w], acc[h][2 * w + 1]);
            else fma_phi_v(ph[h], vw[w], acc[h][2 * w], acc[h][2 * w + 1]);
          }
      }
    }
}

template <int DD>
__global__ void __launch_bounds__(NUM_THREADS, 3)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
                       const int32_t* __restrict__ seq_lens, int chunk, int max_splits,
                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                       float* __restrict__ part_o, float* __restrict__ part_lse, int Hq, int Hkv,
                       int max_pages, int num_pages, float scale_log2, int* status,
                       const __grid_constant__ SegMap map) {
  using DC = DecCfg<DD>;
  constexpr int NST = DC::NST, STAGE_BYTES = DC::STAGE_BYTES, PAGE_BYTES = DC::PAGE_BYTES;
  constexpr int DL = DC::DL, WPL = DC::WPL;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full[NST], empty[NST];
  __shared__ int skip[NST];
  __shared__ float sm_m[NCW][HG];
  __shared__ float sm_l[NCW][HG];
  __shared__ __align__(16) float sm_acc[NCW][HG][DD];
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  int s = blockIdx.x, b = blockIdx.z, n_segs = max_splits;
  if (map.n > 0) {  // the request whose segment range holds blockIdx.x
    int lo = 0, hi = map.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (map.off[mid] <= static_cast<int>(blockIdx.x)) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    s = blockIdx.x - map.off[b];
    n_segs = map.off[b + 1] - map.off[b];
  }
  const int group = Hq / Hkv;
  const int groups_per_kvh = (group + HG - 1) / HG;
  const int kvh = blockIdx.y / groups_per_kvh;
  const int gi = blockIdx.y % groups_per_kvh;
  const int h0 = kvh * group + gi * HG;
  const int nh = min(HG, group - gi * HG);  // real heads in this CTA (the rest is padding)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p_begin = s * chunk / PAGE;

  // The loads that start the CTA go out together, before the length is
  // known: the producer's first 32 block-table entries (inside the row,
  // used only below the page count), the consumers' query rows, the length.
  const int32_t* row = block_table + static_cast<size_t>(b) * max_pages + p_begin;
  int entry0 = 0;
  if (warp == 0 && lane < max_pages - p_begin) entry0 = row[lane];
  uint32_t qw[HG][WPL];
  if (warp != 0) {
    const int l8 = lane & 7;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const int hq = h0 + min(h, nh - 1);  // padded heads reuse a real head's q
      const uint4* qp =
          reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * Hq + hq) * DD + DL * l8);
#pragma unroll
      for (int c = 0; c < WPL / 4; ++c) {
        const uint4 a4 = qp[c];
        qw[h][4 * c] = a4.x;
        qw[h][4 * c + 1] = a4.y;
        qw[h][4 * c + 2] = a4.z;
        qw[h][4 * c + 3] = a4.w;
      }
    }
  }
  // A length past the table's capacity is reported and clamped, so the
  // block-table row is never read out of bounds.
  int len = seq_lens[b];
  if (len < 0 || len > max_pages * PAGE) {
    if (threadIdx.x == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
    len = len < 0 ? 0 : max_pages * PAGE;
  }
  const int t_begin = s * chunk;
  const int t_end = min(len, t_begin + chunk);
  const int n_pages = t_end > t_begin ? (t_end + PAGE - 1) / PAGE - p_begin : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    abort_flag_s = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    bool ok = true;
    int issued = 0;
    for (int i0 = 0; ok && i0 < n_pages; i0 += 32) {
      const int entry = i0 + lane < n_pages ? (i0 == 0 ? entry0 : row[i0 + lane]) : 0;
      const int cnt = min(32, n_pages - i0);
      for (int k = 0; k < cnt; ++k) {
        const int page = __shfl_sync(FULL, entry, k);
        const int i = i0 + k, st = i % NST;
        if (lane == 0) {
          if (i >= NST && !mbar_wait(&empty[st], ((i / NST) + 1) & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
          } else if (page < 0 || page >= num_pages) {
            attn::record_status(status, ATTN_ERR_BAD_INDEX);
            skip[st] = 1;
            mbar_arrive(&full[st]);  // an empty page: nothing is read
            issued = i + 1;
          } else {
            skip[st] = 0;
            uint8_t* dst = ring + st * STAGE_BYTES;
            mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
            tma_load_4d(dst, &tm_k, &full[st], 0, kvh, 0, page);
            tma_load_4d(dst + PAGE_BYTES, &tm_v, &full[st], 0, kvh, 0, page);
            issued = i + 1;
          }
        }
        ok = __shfl_sync(FULL, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0) {
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      int no_abort = 0;
      for (int i = issued > NST ? issued - NST : 0; i < issued; ++i)
        mbar_wait(&full[i % NST], (i / NST) & 1, &no_abort, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int grp = lane >> 3;       // token group within the warp
    const int l8 = lane & 7;         // owns dims [DL l8, DL l8 + DL)
    const int own_h = l8 >> 1;       // head of the values this lane holds after the reduction
    float acc[HG][DL];
    float m_run[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      m_run[h] = -INFINITY;
#pragma unroll
      for (int j = 0; j < DL; ++j) acc[h][j] = 0.f;
    }
    float l_own = 0.f;
    bool ok = true;

    for (int i = cw; i < n_pages; i += NCW) {
      const int st = i % NST;
      ok = __all_sync(FULL, mbar_wait(&full[st], (i / NST) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      if (!skip[st]) {
        const uint8_t* kst = ring + st * STAGE_BYTES + l8 * (DL * 2);
        consume_page<DD>(kst, kst + PAGE_BYTES, t_end - (p_begin + i) * PAGE, qw, acc, m_run,
                         l_own, scale_log2, lane, grp, l8, own_h);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }

    // Combine the 4 token groups of the warp, then the consumer warps.
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int j = 0; j < DL; ++j) {
        acc[h][j] += __shfl_xor_sync(FULL, acc[h][j], 8);
        acc[h][j] += __shfl_xor_sync(FULL, acc[h][j], 16);
      }
    float lsum = l_own;
    lsum += __shfl_xor_sync(FULL, lsum, 1);
    lsum += __shfl_xor_sync(FULL, lsum, 8);
    lsum += __shfl_xor_sync(FULL, lsum, 16);
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float lh = __shfl_sync(FULL, lsum, 2 * h);
      if (lane == 0) {
        sm_m[cw][h] = m_run[h];
        sm_l[cw][h] = lh;
      }
      if (grp == 0) {
        float4* dst = reinterpret_cast<float4*>(&sm_acc[cw][h][DL * l8]);
#pragma unroll
        for (int c = 0; c < DL / 4; ++c)
          dst[c] = make_float4(acc[h][4 * c], acc[h][4 * c + 1], acc[h][4 * c + 2], acc[h][4 * c + 3]);
      }
    }
    named_barrier(1, NCW * 32);

    const int t = threadIdx.x - 32;  // output dim (threads past d idle)
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      if (h >= nh || t >= DD) break;
      float big = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) big = fmaxf(big, sm_m[w][h]);
      float lw = 0.f, ow = 0.f;
      if (big != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float c = ex2(sm_m[w][h] - big);
          lw = fmaf(c, sm_l[w][h], lw);
          ow = fmaf(c, sm_acc[w][h][t], ow);
        }
      }
      const bool empty_row = !(lw > 0.f);
      const float out = empty_row ? 0.f : ow / lw;
      const float row_lse = empty_row ? -INFINITY : (big + log2f(lw)) * attn::kLn2;
      const size_t r = static_cast<size_t>(b) * Hq + h0 + h;
      if (part_o == nullptr) {  // one split: the final output
        o[r * DD + t] = __float2bfloat16_rn(out);
        if (t == 0 && lse != nullptr) lse[r] = row_lse;
      } else {
        part_o[(r * max_splits + s) * DD + t] = out;
        if (t == 0) part_lse[r * max_splits + s] = row_lse;
        // Compact grid: the request's last segment CTA also writes the empty
        // states (O = 0, LSE = -inf) of the slots past its segment count, so
        // the merge reads max_splits written states per row.
        if (s == n_segs - 1)
          for (int s2 = n_segs; s2 < max_splits; ++s2) {
            part_o[(r * max_splits + s2) * DD + t] = 0.f;
            if (t == 0) part_lse[r * max_splits + s2] = -INFINITY;
          }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Load-balanced decode with a fixed grid ("Lecture 4" section 5.6).  The host
// schedule (attn_decode_schedule) cuts every (request, KV-head group) into
// page-aligned segments of at most L_kv tokens and deals them to num_ctas
// CTAs, longest first; the plan sits in a device workspace, so the grid and
// every pointer stay the same from one decode step to the next and one
// captured CUDA graph can replay them all while the plan changes.  A CTA
// walks its segments with the ring position, the page counter and the
// barrier phases running on across segments (no pipeline drain between
// them) and writes every segment as a normalised partial state;
// decode_merge_kernel combines the segments of each output row in token
// order.
struct BalancedPlan {
  const int* cta_off;    // [num_ctas + 1]: the CTA's entries in cta_units
  const int* cta_units;  // unit ids, per CTA in the order they were assigned
  const int* unit;       // [units][4]: request, group, t_begin, t_end
  const int* seg_off;    // [B * G + 1]: the (request, group)'s entries in seg_units
  const int* seg_units;  // unit ids of each (request, group) in token order
};

__global__ void __launch_bounds__(NUM_THREADS, 3)
    decode_balanced_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __nv_bfloat16* __restrict__ q,
                           const int32_t* __restrict__ block_table,
                           const int32_t* __restrict__ seq_lens, const BalancedPlan plan,
                           float* __restrict__ part_o, float* __restrict__ part_lse, int B,
                           int Hq, int Hkv, int U, int max_pages, int num_pages, float scale_log2,
                           int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full[NST], empty[NST], st_ready, st_free;
  __shared__ int skip[NST];
  __shared__ float sm_m[NCW][HG];
  __shared__ float sm_l[NCW][HG];
  __shared__ __align__(16) float sm_acc[NCW][HG][D];
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int group = Hq / Hkv;
  const int gpk = (group + HG - 1) / HG;  // head groups per KV head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The plan is checked before use: an entry out of range is reported
  // (ATTN_ERR_BAD_INDEX) and skipped, so a damaged plan never reads or
  // writes outside the plan, the partial states or the block table.
  int k0 = plan.cta_off[blockIdx.x];
  int n_units = plan.cta_off[blockIdx.x + 1] - k0;
  if (k0 < 0 || n_units < 0 || k0 + n_units > U) {
    if (threadIdx.x == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
    k0 = 0;
    n_units = 0;
  }
  struct Seg {
    int u, b, grp, t_begin, t_end, p_begin, n_pages;  // u < 0: skipped
  };
  // Segment k of this CTA.  Its bounds are clamped to the request's device
  // length and to the block table's capacity (reported), so a stale plan
  // never reads past either.
  auto seg_at = [&](int k) {
    Seg sg;
    sg.u = plan.cta_units[k0 + k];
    sg.n_pages = 0;
    sg.t_begin = sg.t_end = sg.p_begin = 0;
    if (sg.u < 0 || sg.u >= U) {
      if (threadIdx.x == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
      sg.u = -1;
      return sg;
    }
    const int* e = plan.unit + 4 * sg.u;
    sg.b = e[0];
    sg.grp = e[1];
    if (sg.b < 0 || sg.b >= B || sg.grp < 0 || sg.grp >= Hkv * gpk || e[2] < 0 || e[3] < e[2]) {
      if (threadIdx.x == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
      sg.u = -1;
      return sg;
    }
    int len = seq_lens[sg.b];
    if (len < 0 || len > max_pages * PAGE) {
      if (threadIdx.x == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
      len = len < 0 ? 0 : max_pages * PAGE;
    }
    sg.t_begin = min(e[2], len);
    sg.t_end = min(e[3], len);
    sg.p_begin = sg.t_begin / PAGE;
    sg.n_pages = sg.t_end > sg.t_begin ? (sg.t_end + PAGE - 1) / PAGE - sg.p_begin : 0;
    return sg;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&st_ready, NCW);
    mbar_init(&st_free, NCW);
    abort_flag_s = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    bool ok = true;
    int gi = 0;  // pages issued over all segments (ring position)
    for (int k = 0; ok && k < n_units; ++k) {
      const Seg sg = seg_at(k);
      if (sg.u < 0) continue;
      const int kvh = sg.grp / gpk;
      const int32_t* row = block_table + static_cast<size_t>(sg.b) * max_pages + sg.p_begin;
      for (int i0 = 0; ok && i0 < sg.n_pages; i0 += 32) {
        const int entry = i0 + lane < sg.n_pages ? row[i0 + lane] : 0;
        const int cnt = min(32, sg.n_pages - i0);
        for (int kk = 0; kk < cnt; ++kk) {
          const int page = __shfl_sync(FULL, entry, kk);
          const int st = gi % NST;
          if (lane == 0) {
            if (gi >= NST && !mbar_wait(&empty[st], ((gi / NST) + 1) & 1, abort_flag, kWaitLimitNs)) {
              ok = false;
            } else if (page < 0 || page >= num_pages) {
              attn::record_status(status, ATTN_ERR_BAD_INDEX);
              skip[st] = 1;
              mbar_arrive(&full[st]);  // an empty page: nothing is read
            } else {
              skip[st] = 0;
              uint8_t* dst = ring + st * STAGE_BYTES;
              mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
              tma_load_4d(dst, &tm_k, &full[st], 0, kvh, 0, page);
              tma_load_4d(dst + PAGE_BYTES, &tm_v, &full[st], 0, kvh, 0, page);
            }
          }
          ok = __shfl_sync(FULL, ok, 0);
          if (!ok) break;
          ++gi;
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      int no_abort = 0;
      for (int i = gi > NST ? gi - NST : 0; i < gi; ++i)
        mbar_wait(&full[i % NST], (i / NST) & 1, &no_abort, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int grp_l = lane >> 3;     // token group within the warp
    const int l8 = lane & 7;         // owns dims [16 l8, 16 l8 + 16)
    const int own_h = l8 >> 1;       // head of the values this lane holds after the reduction
    const int t = threadIdx.x - 32;  // output dim in the combine step
    bool ok = true;
    int gbase = 0;                   // ring position of the segment's first page
    int kc = 0;                      // segments combined so far (barrier phases)
    for (int k = 0; ok && k < n_units; ++k) {
      const Seg sg = seg_at(k);
      if (sg.u < 0) continue;
      const int kvh = sg.grp / gpk, gi_h = sg.grp % gpk;
      const int h0 = kvh * group + gi_h * HG;
      const int nh = min(HG, group - gi_h * HG);
      uint32_t qw[HG][8];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const int hq = h0 + min(h, nh - 1);  // padded heads reuse a real head's q
        const uint4* qp =
            reinterpret_cast<const uint4*>(q + (static_cast<size_t>(sg.b) * Hq + hq) * D + 16 * l8);
        const uint4 a = qp[0], c = qp[1];
        qw[h][0] = a.x; qw[h][1] = a.y; qw[h][2] = a.z; qw[h][3] = a.w;
        qw[h][4] = c.x; qw[h][5] = c.y; qw[h][6] = c.z; qw[h][7] = c.w;
      }
      float acc[HG][16];
      float m_run[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[h][j] = 0.f;
      }
      float l_own = 0.f;
      // Page i of the segment is ring entry gbase + i, taken by consumer
      // warp (gbase + i) % NCW.
      for (int i = ((cw - gbase) % NCW + NCW) % NCW; i < sg.n_pages; i += NCW) {
        const int gi = gbase + i, st = gi % NST;
        ok = __all_sync(FULL, mbar_wait(&full[st], (gi / NST) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        if (!skip[st]) {
          const uint8_t* kst = ring + st * STAGE_BYTES + l8 * 32;
          consume_page<D>(kst, kst + PAGE_BYTES, sg.t_end - (sg.p_begin + i) * PAGE, qw, acc, m_run,
                       l_own, scale_log2, lane, grp_l, l8, own_h);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      if (!ok) break;
      gbase += sg.n_pages;
      // Combine the 4 token groups of the warp, then the consumer warps
      // (shared memory, reused once every warp has read the previous
      // segment's values: st_free; all written: st_ready).
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          acc[h][j] += __shfl_xor_sync(FULL, acc[h][j], 8);
          acc[h][j] += __shfl_xor_sync(FULL, acc[h][j], 16);
        }
      float lsum = l_own;
      lsum += __shfl_xor_sync(FULL, lsum, 1);
      lsum += __shfl_xor_sync(FULL, lsum, 8);
      lsum += __shfl_xor_sync(FULL, lsum, 16);
      if (kc > 0) {
        ok = __all_sync(FULL, mbar_wait(&st_free, (kc - 1) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float lh = __shfl_sync(FULL, lsum, 2 * h);
        if (lane == 0) {
          sm_m[cw][h] = m_run[h];
          sm_l[cw][h] = lh;
        }
        if (grp_l == 0) {
          float4* dst = reinterpret_cast<float4*>(&sm_acc[cw][h][16 * l8]);
          dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
          dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
          dst[2] = make_float4(acc[h][8], acc[h][9], acc[h][10], acc[h][11]);
          dst[3] = make_float4(acc[h][12], acc[h][13], acc[h][14], acc[h][15]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&st_ready);
      ok = __all_sync(FULL, mbar_wait(&st_ready, kc & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ++kc;
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        if (h >= nh) break;
        float big = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) big = fmaxf(big, sm_m[w][h]);
        float lw = 0.f, ow = 0.f;
        if (big != -INFINITY) {
#pragma unroll
          for (int w = 0; w < NCW; ++w) {
            const float c = ex2(sm_m[w][h] - big);
            lw = fmaf(c, sm_l[w][h], lw);
            ow = fmaf(c, sm_acc[w][h][t], ow);
          }
        }
        const bool empty_row = !(lw > 0.f);
        const size_t slot = static_cast<size_t>(sg.u) * HG + h;
        part_o[slot * D + t] = empty_row ? 0.f : ow / lw;
        if (t == 0) part_lse[slot] = empty_row ? -INFINITY : (big + log2f(lw)) * attn::kLn2;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&st_free);
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }
}

// Output row r = (request b, query head hq): the partial states of its
// (request, group) segments, merged in token order (one warp per row, lane
// l owns dims 4l .. 4l+3; sums in a fixed order, no atomics).
__global__ void __launch_bounds__(128)
    decode_merge_kernel(const BalancedPlan plan, const float* __restrict__ part_o,
                        const float* __restrict__ part_lse, int B, int Hq, int Hkv, int U,
                        __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int* status) {
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= B * Hq) return;
  const int group = Hq / Hkv, gpk = (group + HG - 1) / HG;
  const int b = r / Hq, hq = r % Hq;
  const int kvh = hq / group, hin = hq % group;
  const int grp = kvh * gpk + hin / HG, h = hin % HG;
  int s0 = plan.seg_off[b * Hkv * gpk + grp], s1 = plan.seg_off[b * Hkv * gpk + grp + 1];
  if (s0 < 0 || s1 < s0 || s1 > U) {  // a damaged plan: reported, the row left empty
    if (lane == 0) attn::record_status(status, ATTN_ERR_BAD_INDEX);
    s0 = s1 = 0;
  }
  auto unit_of = [&](int s) {
    const int u = plan.seg_units[s];
    return (u >= 0 && u < U) ? u : -1;
  };
  // The row is latency-bound (a few KB over many segments), so loads go out
  // together: lane l holds the unit and LSE of segments s0 + l, s0 + l + 32,
  // ... (the first 32 kept in registers), and the O slices are read in
  // batches of 8 segments, all 8 loads issued before the first is used.
  const int n = s1 - s0;
  const int u_first = lane < n ? unit_of(s0 + lane) : -1;
  const float ls_first = u_first >= 0 ? part_lse[static_cast<size_t>(u_first) * HG + h] : -INFINITY;
  float big = ls_first;
  for (int i = lane + 32; i < n; i += 32) {
    const int u = unit_of(s0 + i);
    if (u >= 0) big = fmaxf(big, part_lse[static_cast<size_t>(u) * HG + h]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(FULL, big, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (big != -INFINITY) {
    for (int base = 0; base < n; base += 32) {
      int u_l = u_first;
      float ls_l = ls_first;
      if (base > 0) {
        u_l = base + lane < n ? unit_of(s0 + base + lane) : -1;
        ls_l = u_l >= 0 ? part_lse[static_cast<size_t>(u_l) * HG + h] : -INFINITY;
      }
      // An empty segment (LSE = -inf) weighs 0 and its O is not read.
      const float w_l = (u_l >= 0 && ls_l != -INFINITY) ? expf(ls_l - big) : 0.f;
      const int cnt = min(32, n - base);
      for (int j0 = 0; j0 < cnt; j0 += 8) {
        float4 x[8];
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int j = j0 + k;  // warp-uniform
          const int u = __shfl_sync(FULL, u_l, j & 31);
          w[k] = __shfl_sync(FULL, w_l, j & 31);
          if (j >= cnt) w[k] = 0.f;
          x[k] = w[k] > 0.f ? *reinterpret_cast<const float4*>(
                                  part_o + (static_cast<size_t>(u) * HG + h) * D + 4 * lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (j0 + k >= cnt) break;
          if (!(w[k] > 0.f)) continue;
          wsum += w[k];
          acc.x = fmaf(w[k], x[k].x, acc.x);
          acc.y = fmaf(w[k], x[k].y, acc.y);
          acc.z = fmaf(w[k], x[k].z, acc.z);
          acc.w = fmaf(w[k], x[k].w, acc.w);
        }
      }
    }
  }
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
  *reinterpret_cast<uint2*>(o + static_cast<size_t>(r) * D + 4 * lane) =
      make_uint2(attn::pack_bf16x2(acc.x * inv, acc.y * inv), attn::pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0 && lse != nullptr) lse[r] = empty ? -INFINITY : big + logf(wsum);
}

// k_pages / v_pages [num_pages, 16, Hkv, d] bf16 as a 4-D tensor
// {d, Hkv, 16, num_pages}; box {d, 1, 16, 1} = one page of one KV head.
bool make_page_map(CUtensorMap* m, const void* base, int Hkv, int num_pages, int dd = D) {
  attn_host::EncodeTiledFn enc = attn_host::encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(dd), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(PAGE), static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(dd) * 2,
                                 static_cast<cuuint64_t>(Hkv) * dd * 2,
                                 static_cast<cuuint64_t>(PAGE) * Hkv * dd * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(dd), 1, PAGE, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool set_smem_attr() {
  static bool done[64] = {};  // per device: kernel attributes are per device
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(decode_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(decode_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

bool set_balanced_smem_attr() {
  static bool done[64] = {};
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(decode_balanced_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

}  // namespace

namespace attn_host {

int decode_balanced_ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (!set_balanced_smem_attr() ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_balanced_kernel, NUM_THREADS,
                                                      SMEM_BYTES) != cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

attn_status_t launch_decode_balanced(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     const int32_t* cta_off, const int32_t* cta_units,
                                     const int32_t* unit, const int32_t* seg_off,
                                     const int32_t* seg_units, int num_ctas, int U, float* part_o,
                                     float* part_lse, void* o, float* lse, int B, int Hq, int Hkv,
                                     int d, int page_size, int max_pages, int num_pages,
                                     float scale, cudaStream_t stream) {
  if (d != D || page_size != PAGE) return ATTN_ERR_UNSUPPORTED;
  if (!set_balanced_smem_attr()) return ATTN_ERR_CUDA;
  CUtensorMap mk, mv;
  if (!make_page_map(&mk, k_pages, Hkv, num_pages) || !make_page_map(&mv, v_pages, Hkv, num_pages))
    return ATTN_ERR_CUDA;
  const BalancedPlan plan{cta_off, cta_units, unit, seg_off, seg_units};
  decode_balanced_kernel<<<num_ctas, NUM_THREADS, SMEM_BYTES, stream>>>(
      mk, mv, static_cast<const __nv_bfloat16*>(q), block_table, seq_lens, plan, part_o, part_lse,
      B, Hq, Hkv, U, max_pages, num_pages, scale * attn::kLog2e, device_status_ptr());
  const int rows = B * Hq;
  decode_merge_kernel<<<(rows + 3) / 4, 128, 0, stream>>>(
      plan, part_o, part_lse, B, Hq, Hkv, U, static_cast<__nv_bfloat16*>(o), lse,
      device_status_ptr());
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int decode_ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (!set_smem_attr() ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel<128>, NUM_THREADS,
                                                      SMEM_BYTES) != cudaSuccess ||
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
                                 int num_pages, float scale, const int32_t* lens_host,
                                 cudaStream_t stream) {
  if ((d != 128 && d != 64) || page_size != PAGE) return ATTN_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (!set_smem_attr()) return ATTN_ERR_CUDA;
  CUtensorMap mk, mv;
  if (!make_page_map(&mk, k_pages, Hkv, num_pages, d) ||
      !make_page_map(&mv, v_pages, Hkv, num_pages, d))
    return ATTN_ERR_CUDA;
  const int groups = Hkv * ((group + HG - 1) / HG);
  dim3 grid(max_splits, groups, B);
  SegMap map;
  map.n = 0;
  if (max_splits > 1 && lens_host != nullptr && B <= kSegMapMax) {
    // One CTA per non-empty segment (at least one per request): a plan that
    // fits the resident CTAs runs as one wave with no empty CTAs in it.
    map.n = B;
    map.off[0] = 0;
    for (int i = 0; i < B; ++i) {
      const int len = lens_host[i] < 0 ? 0 : lens_host[i];
      const int n = std::min(max_splits, std::max(1, (len + chunk - 1) / chunk));
      map.off[i + 1] = map.off[i] + n;
    }
    grid = dim3(map.off[B], groups, 1);
  }
  auto kernel = d == 64 ? decode_bf16_kernel<64> : decode_bf16_kernel<128>;
  kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
      mk, mv, static_cast<const __nv_bfloat16*>(q), block_table, seq_lens, chunk, max_splits,
      static_cast<__nv_bfloat16*>(o), lse, part_o, part_lse, Hq, Hkv, max_pages, num_pages,
      scale * attn::kLog2e, device_status_ptr(), map);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
