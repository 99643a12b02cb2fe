// C ABI entry points: host-side validation, split planning and launch
// selection.  Every check happens before anything is enqueued, so an invalid
// call touches no memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "attn.h"

namespace attn_host {
int* device_status_ptr();
int num_sms();
int decode_ctas_per_sm();
attn_status_t launch_prefill_f32(const float*, const float*, const float*, float*, float*, int, int,
                                 int, int, int, int, int, float, cudaStream_t);
attn_status_t launch_prefill_bf16(const void*, const void*, const void*, void*, float*, int, int,
                                  int, int, int, int, int, float, int, cudaStream_t);
attn_status_t launch_prefill_bf16_paged(const void*, const void*, const void*, const int*,
                                        const int*, int, int, const int*, const int*, void*, float*,
                                        int, int, int, int, int, int, int, int, int, int, float,
                                        cudaStream_t);
attn_status_t launch_prefill_bf16_varlen(const void*, const void*, const void*, void*, float*,
                                         const int*, const int*, int, int, int, int, int, int, int,
                                         int, int, float, cudaStream_t);
attn_status_t launch_decode_bf16(const void*, const void*, const void*, const int32_t*,
                                 const int32_t*, int, int, int, void*, float*, float*, float*, int,
                                 int, int, int, int, int, float, const int32_t*, cudaStream_t);
attn_status_t launch_bwd_bf16(const void*, const void*, const void*, const void*, const float*,
                              const void*, void*, void*, void*, float*, int, int, int, int, int,
                              int, int, float, cudaStream_t);
int decode_balanced_ctas_per_sm();
attn_status_t launch_decode_balanced(const void*, const void*, const void*, const int32_t*,
                                     const int32_t*, const int32_t*, const int32_t*,
                                     const int32_t*, const int32_t*, const int32_t*, int, int, float*,
                                     float*, void*, float*, int, int, int, int, int, int, int,
                                     float, cudaStream_t);
attn_status_t launch_merge(const float*, const float*, int, int, int, void*, float*, attn_dtype_t,
                           cudaStream_t);
attn_status_t launch_cascade_gather_q(const void*, void*, int, int, int, int, cudaStream_t);
attn_status_t launch_cascade_merge(const void*, const float*, int, const float*, const float*, int,
                                   int, int, int, int, void*, float*, cudaStream_t);
}  // namespace attn_host

namespace {

constexpr size_t kAlign = 256;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Non-empty work units (request, KV head, segment) for chunk length C.
int64_t plan_units(const int32_t* lens, int B, int Hkv, int64_t chunk) {
  int64_t n = 0;
  for (int b = 0; b < B; ++b) n += cdiv(std::max<int32_t>(lens[b], 0), chunk);
  return n * Hkv;
}

// Split planner ("Lecture 4" section 4.2 and exercise 6; the reading is
// spelled out in attn.h): the shortest page-multiple chunk C whose units fit
// in one round of `slots` workers, or no split when even whole requests do
// not fit.  Returns C and the largest per-request segment count.
void plan(const int32_t* lens, int B, int Hkv, int page, int num_splits, int slots, int32_t* chunk,
          int32_t* max_splits) {
  int64_t longest = 1;
  for (int b = 0; b < B; ++b) longest = std::max<int64_t>(longest, lens[b]);
  const int64_t full = std::max<int64_t>(page, cdiv(longest, page) * page);
  int64_t best_c = full;
  if (num_splits > 0) {
    best_c = std::max<int64_t>(page, cdiv(cdiv(longest, num_splits), page) * page);
  } else if (plan_units(lens, B, Hkv, full) <= slots) {
    int64_t lo = 1, hi = full / page;  // in pages; hi fits
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (plan_units(lens, B, Hkv, mid * page) <= slots)
        hi = mid;
      else
        lo = mid + 1;
    }
    best_c = hi * page;
  }
  int64_t smax = 1;
  for (int b = 0; b < B; ++b) smax = std::max<int64_t>(smax, cdiv(lens[b], best_c));
  *chunk = static_cast<int32_t>(best_c);
  *max_splits = static_cast<int32_t>(smax);
}

// The last plan of this thread, reused when the next call has the same
// lengths and parameters (every layer of one decode step does).
struct PlanCache {
  std::vector<int32_t> lens;
  int Hkv = -1, page = -1, num_splits = -1, slots = -1;
  int32_t chunk = 0, max_splits = 0;
};

void plan_cached(const int32_t* lens, int B, int Hkv, int page, int num_splits, int slots,
                 int32_t* chunk, int32_t* max_splits) {
  thread_local PlanCache cache;
  if (cache.Hkv == Hkv && cache.page == page && cache.num_splits == num_splits &&
      cache.slots == slots && cache.lens.size() == static_cast<size_t>(B) &&
      std::equal(cache.lens.begin(), cache.lens.end(), lens)) {
    *chunk = cache.chunk;
    *max_splits = cache.max_splits;
    return;
  }
  plan(lens, B, Hkv, page, num_splits, slots, chunk, max_splits);
  cache.lens.assign(lens, lens + B);
  cache.Hkv = Hkv;
  cache.page = page;
  cache.num_splits = num_splits;
  cache.slots = slots;
  cache.chunk = *chunk;
  cache.max_splits = *max_splits;
}

// ---------------------------------------------------------------------------
// Load-balanced decode schedule ("Lecture 4" section 5.6; the reading is in
// attn.h).  Plan layout in the workspace (int32, then the fp32 partials):
//   [0] number of units
//   cta_off[num_ctas + 1], cta_units[U], unit[U][4] (request, group, t_begin,
//   t_end), seg_off[B * G + 1], seg_units[U]
// with G = Hkv * ceil((Hq / Hkv) / 4) head groups and U = num_ctas + B * G,
// the most units any lengths can produce, so the layout (and a captured
// graph) only depends on (B, Hq, Hkv, num_ctas).
constexpr int kHeadsPerCta = 4;

struct BalancedLayout {
  int G, U;
  size_t cta_off, cta_units, unit, seg_off, seg_units, ints;  // int32 offsets
  size_t part_o, part_lse, total;                           // byte offsets
};

BalancedLayout balanced_layout(int B, int Hq, int Hkv, int d, int num_ctas) {
  BalancedLayout L;
  L.G = Hkv * ((Hq / Hkv + kHeadsPerCta - 1) / kHeadsPerCta);
  L.U = num_ctas + B * L.G;
  L.cta_off = 1;
  L.cta_units = L.cta_off + num_ctas + 1;
  L.unit = L.cta_units + L.U;
  L.seg_off = L.unit + 4 * static_cast<size_t>(L.U);
  L.seg_units = L.seg_off + static_cast<size_t>(B) * L.G + 1;
  L.ints = L.seg_units + L.U;
  L.part_o = round_up(L.ints * sizeof(int32_t), kAlign);
  L.part_lse = L.part_o + round_up(static_cast<size_t>(L.U) * kHeadsPerCta * d * sizeof(float), kAlign);
  L.total = L.part_lse + round_up(static_cast<size_t>(L.U) * kHeadsPerCta * sizeof(float), kAlign);
  return L;
}

// Steps 2-5 of the section: L_kv from the total work, page-aligned segments
// of at most L_kv tokens per (request, group) (an empty request keeps one
// empty unit), units sorted by token count from large to small (ties in
// list order) and each given to the least-loaded CTA (lowest index on ties).
void plan_balanced(const int32_t* lens, int B, int G, int num_ctas, int page,
                   const BalancedLayout& L, int32_t* out) {
  int64_t total = 0;
  for (int b = 0; b < B; ++b) total += std::max<int32_t>(lens[b], 0);
  total *= G;
  int64_t lkv = std::max<int64_t>(1, cdiv(total, num_ctas));
  lkv = cdiv(lkv, page) * page;
  struct U4 {
    int32_t b, g, t0, t1;
  };
  std::vector<U4> units;
  std::vector<int32_t> seg_off(static_cast<size_t>(B) * G + 1, 0);
  for (int b = 0; b < B; ++b) {
    const int64_t n = std::max<int32_t>(lens[b], 0);
    for (int g = 0; g < G; ++g) {
      if (n == 0) units.push_back({b, g, 0, 0});
      for (int64_t t0 = 0; t0 < n; t0 += lkv)
        units.push_back({b, g, static_cast<int32_t>(t0), static_cast<int32_t>(std::min(n, t0 + lkv))});
      seg_off[static_cast<size_t>(b) * G + g + 1] = static_cast<int32_t>(units.size());
    }
  }
  const int nu = static_cast<int>(units.size());
  std::vector<int32_t> order(nu);
  for (int u = 0; u < nu; ++u) order[u] = u;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t c) {
    return units[a].t1 - units[a].t0 > units[c].t1 - units[c].t0;
  });
  std::priority_queue<std::pair<int64_t, int>, std::vector<std::pair<int64_t, int>>,
                      std::greater<std::pair<int64_t, int>>>
      heap;
  for (int c = 0; c < num_ctas; ++c) heap.push({0, c});
  std::vector<std::vector<int32_t>> per(num_ctas);
  for (int32_t u : order) {
    const auto top = heap.top();
    heap.pop();
    per[top.second].push_back(u);
    heap.push({top.first + (units[u].t1 - units[u].t0), top.second});
  }
  out[0] = nu;
  int32_t k = 0;
  for (int c = 0; c < num_ctas; ++c) {
    out[L.cta_off + c] = k;
    for (int32_t u : per[c]) out[L.cta_units + k++] = u;
  }
  out[L.cta_off + num_ctas] = k;
  for (int u = 0; u < nu; ++u) {
    out[L.unit + 4 * u + 0] = units[u].b;
    out[L.unit + 4 * u + 1] = units[u].g;
    out[L.unit + 4 * u + 2] = units[u].t0;
    out[L.unit + 4 * u + 3] = units[u].t1;
  }
  for (size_t i = 0; i < seg_off.size(); ++i) out[L.seg_off + i] = seg_off[i];
  for (int u = 0; u < nu; ++u) out[L.seg_units + u] = u;  // list order is token order
}

int balanced_ctas(int num_ctas) {
  if (num_ctas > 0) return num_ctas;
  const int sms = attn_host::num_sms();
  return sms <= 0 ? -1 : sms * attn_host::decode_balanced_ctas_per_sm();
}

}  // namespace

extern "C" {

int attn_version(void) { return 100; }

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_BAD_INDEX: return "ATTN_ERR_BAD_INDEX";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                       attn_dtype_t dtype, attn_stream_t stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32)
    return attn_host::launch_prefill_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                         static_cast<const float*>(v), static_cast<float*>(o), lse,
                                         B, Hq, Hkv, Lq, Lk, d, causal ? 1 : 0, scale, st);
  return attn_host::launch_prefill_bf16(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal ? 1 : 0,
                                        scale, 1, st);
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                              int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                              int Hkv, int d, int causal, float scale, attn_dtype_t dtype,
                              attn_stream_t stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 ||
      total_q < 0 || total_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (total_q == 0) return ATTN_OK;  // no query rows: nothing to write
  if (!q || !o || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * Hq > (1 << 24) || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (total_k == 0) {
    // No sequence has keys, so every row sees none (O = 0, LSE = -inf) and
    // no K/V tile is ever loaded; q stands in for the unread K/V buffers so
    // that their tensor maps are still encodable.
    k = v = q;  // Hkv <= Hq rows of q are a valid stand-in
    total_k = 1;
    max_seqlen_k = 1;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  return attn_host::launch_prefill_bf16_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B,
                                               max_seqlen_q, max_seqlen_k, total_q, total_k, Hq,
                                               Hkv, d, causal ? 1 : 0, scale,
                                               reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens_k, void* o, float* lse, int B,
                                 int max_seqlen_q, int max_seqlen_k, int total_q, int Hq, int Hkv,
                                 int d, int page_size, int max_pages_per_seq, int num_pages,
                                 int causal, float scale, attn_dtype_t dtype, attn_stream_t stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen_q <= 0 || max_seqlen_k < 0 ||
      total_q < 0 || max_pages_per_seq <= 0 || num_pages <= 0 || page_size <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (total_q == 0) return ATTN_OK;  // no query rows: nothing to write
  if (!q || !k_pages || !v_pages || !block_table || !cu_seqlens_q || !seq_lens_k || !o)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (page_size > 128 || (page_size & (page_size - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)max_seqlen_k > (int64_t)max_pages_per_seq * page_size) return ATTN_ERR_INVALID_ARG;
  if ((int64_t)B * max_pages_per_seq > 0x7fffffffLL || num_pages == 0x7fffffff ||
      (int64_t)num_pages * page_size > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * Hq > (1 << 24) || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens_k) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  return attn_host::launch_prefill_bf16_paged(
      q, k_pages, v_pages, block_table, nullptr, 0, page_size, cu_seqlens_q, seq_lens_k, o, lse,
      B, max_seqlen_q, std::max(max_seqlen_k, 1), total_q, Hq, Hkv, d, max_pages_per_seq,
      num_pages, causal ? 1 : 0, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_prefill_bsr(const void* q, const void* k_blocks, const void* v_blocks,
                               const int32_t* kv_indptr, const int32_t* kv_indices, int nnz,
                               const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o,
                               float* lse, int B, int max_seqlen_q, int max_seqlen_k, int total_q,
                               int Hq, int Hkv, int d, int block_size, int num_blocks, int causal,
                               float scale, attn_dtype_t dtype, attn_stream_t stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen_q <= 0 || max_seqlen_k < 0 ||
      total_q < 0 || nnz < 0 || num_blocks <= 0 || block_size <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (total_q == 0) return ATTN_OK;  // no query rows: nothing to write
  if (!q || !k_blocks || !v_blocks || !kv_indptr || !cu_seqlens_q || !seq_lens_k || !o ||
      (nnz > 0 && !kv_indices))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (block_size > 128 || (block_size & (block_size - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
  if (num_blocks == 0x7fffffff || (int64_t)num_blocks * block_size > 0x7fffffffLL ||
      (int64_t)max_seqlen_k > (int64_t)nnz * block_size)
    return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * Hq > (1 << 24) || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_blocks) || !aligned16(v_blocks) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(kv_indptr) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(kv_indices) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens_k) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  // With no blocks at all (nnz = 0) kv_indptr stands in for the unread indices.
  return attn_host::launch_prefill_bf16_paged(
      q, k_blocks, v_blocks, nnz > 0 ? kv_indices : kv_indptr, kv_indptr, nnz, block_size,
      cu_seqlens_q, seq_lens_k, o, lse, B, max_seqlen_q, std::max(max_seqlen_k, 1), total_q, Hq,
      Hkv, d, 0, num_blocks, causal ? 1 : 0, scale, reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_decode_sched_workspace_bytes(int B, int Hq, int Hkv, int d, int num_ctas) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 0;
  const int ctas = balanced_ctas(num_ctas);
  if (ctas <= 0) return 0;
  return balanced_layout(B, Hq, Hkv, d, ctas).total;
}

attn_status_t attn_decode_schedule_host(const int32_t* seq_lens_host, int B, int Hq, int Hkv,
                                        int page_size, int num_ctas, int32_t* plan_out,
                                        size_t plan_ints) {
  if (!seq_lens_host || !plan_out || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 ||
      page_size <= 0 || num_ctas <= 0)
    return ATTN_ERR_INVALID_ARG;
  const BalancedLayout L = balanced_layout(B, Hq, Hkv, 128, num_ctas);
  if (plan_ints < L.ints) return ATTN_ERR_WORKSPACE;
  plan_balanced(seq_lens_host, B, L.G, num_ctas, page_size, L, plan_out);
  return ATTN_OK;
}

attn_status_t attn_decode_schedule(const int32_t* seq_lens_host, int B, int Hq, int Hkv,
                                   int page_size, int num_ctas, void* workspace,
                                   size_t workspace_bytes, attn_stream_t stream) {
  if (!seq_lens_host || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0)
    return ATTN_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens_host[b] < 0) return ATTN_ERR_INVALID_ARG;
  const int ctas = balanced_ctas(num_ctas);
  if (ctas <= 0) return ATTN_ERR_CUDA;
  const BalancedLayout L = balanced_layout(B, Hq, Hkv, 128, ctas);
  if (workspace == nullptr || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return ATTN_ERR_WORKSPACE;
  thread_local std::vector<int32_t> host;
  host.assign(L.ints, 0);
  plan_balanced(seq_lens_host, B, L.G, ctas, page_size, L, host.data());
  // From pageable memory: the copy is staged before the call returns, so the
  // host vector may be reused right away.
  return cudaMemcpyAsync(workspace, host.data(), L.ints * sizeof(int32_t), cudaMemcpyHostToDevice,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

attn_status_t attn_decode_paged_balanced(const void* q, const void* k_pages, const void* v_pages,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int page_size, void* o, float* lse, int B, int Hq,
                                         int Hkv, int d, int max_pages_per_seq, int num_pages,
                                         float scale, int num_ctas, void* workspace,
                                         size_t workspace_bytes, attn_dtype_t dtype,
                                         attn_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages_per_seq <= 0 || num_pages <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 128 || page_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  const int ctas = balanced_ctas(num_ctas);
  if (ctas <= 0) return ATTN_ERR_CUDA;
  const BalancedLayout L = balanced_layout(B, Hq, Hkv, d, ctas);
  if (workspace == nullptr || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return ATTN_ERR_WORKSPACE;
  const int32_t* plan = static_cast<const int32_t*>(workspace);
  char* ws = static_cast<char*>(workspace);
  return attn_host::launch_decode_balanced(
      q, k_pages, v_pages, block_table, seq_lens, plan + L.cta_off, plan + L.cta_units,
      plan + L.unit, plan + L.seg_off, plan + L.seg_units, ctas, L.U,
      reinterpret_cast<float*>(ws + L.part_o), reinterpret_cast<float*>(ws + L.part_lse), o, lse, B,
      Hq, Hkv, d, page_size, max_pages_per_seq, num_pages, scale,
      reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Lq) {
  if (B <= 0 || Hq <= 0 || Lq <= 0) return 0;
  // -LSE log2e and -D (one float per query row, rows padded to whole
  // 128-row tiles), then the kernels' two work counters.
  const size_t rows_pad = static_cast<size_t>(B) * Hq * ((static_cast<size_t>(Lq) + 127) / 128) * 128;
  return 2 * round_up(rows_pad * sizeof(float), kAlign) + kAlign;
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* d_o, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                       void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                       attn_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(d_o) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_bwd_workspace_bytes(B, Hq, Lq);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return ATTN_ERR_WORKSPACE;
  return attn_host::launch_bwd_bf16(q, k, v, o, lse, d_o, dq, dk, dv,
                                    static_cast<float*>(workspace), B, Hq, Hkv, Lq, Lk, d,
                                    causal ? 1 : 0, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_decode_plan(const int32_t* seq_lens_host, int B, int Hkv, int page_size,
                               int num_splits, int slots, int32_t* chunk_out,
                               int32_t* max_splits_out) {
  if (!seq_lens_host || !chunk_out || !max_splits_out) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || page_size <= 0 || num_splits < 0) return ATTN_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens_host[b] < 0) return ATTN_ERR_INVALID_ARG;
  if (slots <= 0) {
    const int sms = attn_host::num_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    slots = sms * attn_host::decode_ctas_per_sm();
  }
  plan_cached(seq_lens_host, B, Hkv, page_size, num_splits, slots, chunk_out, max_splits_out);
  return ATTN_OK;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || max_splits <= 1) return 0;
  const size_t states = (size_t)B * Hq * max_splits;
  return round_up(states * d * sizeof(float), kAlign) + round_up(states * sizeof(float), kAlign);
}

attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const int32_t* seq_lens_host, int page_size, int num_splits,
                                void* o, float* lse, int B, int Hq, int Hkv, int d,
                                int max_pages_per_seq, int num_pages, float scale,
                                void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                                attn_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages_per_seq <= 0 || num_pages <= 0 ||
      num_splits < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if ((d != 64 && d != 128) || page_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  int32_t chunk = max_pages_per_seq * page_size, smax = 1;
  std::vector<int32_t> host_lens;
  const int32_t* lens = seq_lens_host;
  if (num_splits != 1) {
    if (lens == nullptr) {
      host_lens.resize(B);
      if (cudaMemcpyAsync(host_lens.data(), seq_lens, sizeof(int32_t) * B, cudaMemcpyDeviceToHost,
                          st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        return ATTN_ERR_CUDA;
      lens = host_lens.data();
    }
    for (int b = 0; b < B; ++b)
      if (lens[b] < 0 || (int64_t)lens[b] > (int64_t)max_pages_per_seq * page_size)
        return ATTN_ERR_INVALID_ARG;
    int slots = 1;
    if (num_splits == 0) {
      const int sms = attn_host::num_sms();
      if (sms <= 0) return ATTN_ERR_CUDA;
      slots = sms * attn_host::decode_ctas_per_sm();
    }
    plan_cached(lens, B, Hkv, page_size, num_splits, slots, &chunk, &smax);
  }
  if (smax > 65535) return ATTN_ERR_UNSUPPORTED;
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (smax > 1) {
    const size_t need = attn_decode_workspace_bytes(B, Hq, d, smax);
    if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return ATTN_ERR_WORKSPACE;
    part_o = static_cast<float*>(workspace);
    part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        round_up((size_t)B * Hq * smax * d * sizeof(float), kAlign));
  }
  attn_status_t s = attn_host::launch_decode_bf16(q, k_pages, v_pages, block_table, seq_lens,
                                                  page_size, chunk, smax, o, lse, part_o, part_lse,
                                                  B, Hq, Hkv, d, max_pages_per_seq, num_pages,
                                                  scale, lens, st);
  if (s != ATTN_OK || smax == 1) return s;
  return attn_host::launch_merge(part_o, part_lse, B * Hq, smax, d, o, lse, dtype, st);
}

attn_status_t attn_merge_states(const float* o_parts, const float* lse_parts, int rows, int S,
                                int d, void* o_out, float* lse_out, attn_dtype_t out_dtype,
                                attn_stream_t stream) {
  if (!o_parts || !lse_parts || !o_out) return ATTN_ERR_INVALID_ARG;
  if (rows <= 0 || S <= 0 || d <= 0 || d % 4 != 0) return ATTN_ERR_INVALID_ARG;
  if (d > 512) return ATTN_ERR_UNSUPPORTED;
  if (out_dtype != ATTN_F32 && out_dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o_out)) return ATTN_ERR_INVALID_ARG;
  if (rows > 0x7fffffff / 2) return ATTN_ERR_UNSUPPORTED;
  return attn_host::launch_merge(o_parts, lse_parts, rows, S, d, o_out, lse_out, out_dtype,
                                 reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---------------------------------------------------------------- cascade decode

namespace {

// Prefix chunks for the cascade prefix pass ("Lecture 4", section 4.4: the
// stacked query rows attend to the prefix once; splitting the prefix into
// chunks merged by the LSE operator only adds parallelism).  The prefill
// kernel at d = 128 runs one item (two 128-row Q tiles of one head, one
// chunk) per SM at a time, so a plan costs
//   waves x (kItemOverheadTiles + K/V tiles per chunk),
// waves = ceil(Hkv x tile pairs x chunks / slots).  Chunks are divisors of
// the prefix of at least 128 tokens (one chunk if the prefix is shorter);
// the cheapest plan wins, ties to fewer chunks.
constexpr int64_t kItemOverheadTiles = 2;

int cascade_prefix_chunks(int prefix_len, int rows_per_kvh, int Hkv, int slots) {
  const int64_t pairs = cdiv(rows_per_kvh, 256);
  int best = 1;
  int64_t best_cost = -1;
  for (int c = 1; c == 1 || (int64_t)c * 128 <= prefix_len; ++c) {
    if (prefix_len % c != 0) continue;
    const int64_t waves = cdiv((int64_t)Hkv * pairs * c, slots);
    const int64_t cost = waves * (kItemOverheadTiles + cdiv(prefix_len / c, 128));
    if (best_cost < 0 || cost < best_cost) {
      best = c;
      best_cost = cost;
    }
  }
  return best;
}

// The prefix pass runs beside the suffix decode, whose CTAs need the SMs the
// prefill leaves free (a d = 128 prefill CTA takes a whole SM's shared
// memory), so the chunk plan is made for half the SMs.
int cascade_prefix_slots(int sms) { return sms / 2 > 0 ? sms / 2 : 1; }

// One side stream and its fork / join events per device, created on first
// use and kept for the process.  Concurrent callers share them: the side
// stream then runs their suffix passes one after another, and a join event
// re-recorded by another call only makes a caller wait longer, never less.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream() {
  static std::mutex mu;
  static SideStream per_device[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  SideStream& s = per_device[dev];
  if (s.stream == nullptr) {
    if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
      s.stream = nullptr;
      return nullptr;
    }
  }
  return &s;
}

struct CascadeLayout {
  size_t q_stack, o_pre, lse_pre, o_suf, lse_suf, total;
};

CascadeLayout cascade_layout(int B, int Hq, int d, int prefix_chunks, int suffix_splits) {
  CascadeLayout L;
  const size_t rows = (size_t)B * Hq;
  size_t off = 0;
  L.q_stack = off;
  off += round_up(rows * d * 2, kAlign);
  L.o_pre = off;
  off += round_up(rows * prefix_chunks * d * 2, kAlign);
  L.lse_pre = off;
  off += round_up(rows * prefix_chunks * sizeof(float), kAlign);
  L.o_suf = off;
  off += round_up(rows * suffix_splits * d * sizeof(float), kAlign);
  L.lse_suf = off;
  off += round_up(rows * suffix_splits * sizeof(float), kAlign);
  L.total = off;
  return L;
}

}  // namespace

attn_status_t attn_cascade_plan(int B, int Hq, int Hkv, int prefix_len,
                                const int32_t* suffix_lens_host, int page_size, int num_splits,
                                int prefix_slots, int suffix_slots, int32_t* prefix_chunks_out,
                                int32_t* suffix_chunk_out, int32_t* suffix_splits_out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || prefix_len <= 0 || page_size <= 0 ||
      num_splits < 0 || suffix_lens_host == nullptr || prefix_chunks_out == nullptr ||
      suffix_chunk_out == nullptr || suffix_splits_out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (prefix_slots <= 0) {
    const int sms = attn_host::num_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    prefix_slots = cascade_prefix_slots(sms);
  }
  *prefix_chunks_out = cascade_prefix_chunks(prefix_len, B * (Hq / Hkv), Hkv, prefix_slots);
  return attn_decode_plan(suffix_lens_host, B, Hkv, page_size, num_splits, suffix_slots,
                          suffix_chunk_out, suffix_splits_out);
}

size_t attn_cascade_workspace_bytes(int B, int Hq, int d, int prefix_chunks, int suffix_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || prefix_chunks <= 0 || suffix_splits <= 0) return 0;
  return cascade_layout(B, Hq, d, prefix_chunks, suffix_splits).total;
}

attn_status_t attn_decode_cascade(const void* q, const void* prefix_k, const void* prefix_v,
                                  int prefix_len, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const int32_t* seq_lens_host, int page_size, int num_splits,
                                  void* o, float* lse, int B, int Hq, int Hkv, int d,
                                  int max_pages_per_seq, int num_pages, float scale,
                                  void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                                  attn_stream_t stream) {
  if (!q || !prefix_k || !prefix_v || !k_pages || !v_pages || !block_table || !seq_lens || !o ||
      !seq_lens_host)
    return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || prefix_len <= 0 ||
      max_pages_per_seq <= 0 || num_pages <= 0 || num_splits < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if ((d != 128 && d != 64) || page_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535 || (int64_t)B * Hq > (1 << 24)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(prefix_k) || !aligned16(prefix_v) || !aligned16(k_pages) ||
      !aligned16(v_pages) || !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens_host[b] < 0 || (int64_t)seq_lens_host[b] > (int64_t)max_pages_per_seq * page_size)
      return ATTN_ERR_INVALID_ARG;
  const int sms = attn_host::num_sms();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int prefix_chunks =
      cascade_prefix_chunks(prefix_len, B * (Hq / Hkv), Hkv, cascade_prefix_slots(sms));
  int32_t chunk = max_pages_per_seq * page_size, smax = 1;
  if (num_splits != 1)
    plan_cached(seq_lens_host, B, Hkv, page_size, num_splits,
                num_splits == 0 ? sms * attn_host::decode_ctas_per_sm() : 1, &chunk, &smax);
  if (smax > 65535) return ATTN_ERR_UNSUPPORTED;
  const CascadeLayout L = cascade_layout(B, Hq, d, prefix_chunks, smax);
  if (workspace == nullptr || workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return ATTN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  void* q_stack = ws + L.q_stack;
  void* o_pre = ws + L.o_pre;
  float* lse_pre = reinterpret_cast<float*>(ws + L.lse_pre);
  float* o_suf = reinterpret_cast<float*>(ws + L.o_suf);
  float* lse_suf = reinterpret_cast<float*>(ws + L.lse_suf);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The suffix decode does not depend on the prefix pass: it runs on a side
  // stream forked from (and joined back into) the caller's stream, so its
  // CTAs fill the SMs the prefix prefill leaves free.
  SideStream* side = side_stream();
  if (side == nullptr) return ATTN_ERR_CUDA;
  if (cudaEventRecord(side->fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // 3. (side stream) each request's own suffix, as partial states;
  attn_status_t s = attn_host::launch_decode_bf16(q, k_pages, v_pages, block_table, seq_lens,
                                                  page_size, chunk, smax, o, lse, o_suf, lse_suf,
                                                  B, Hq, Hkv, d, max_pages_per_seq, num_pages,
                                                  scale, seq_lens_host, side->stream);
  if (cudaEventRecord(side->join, side->stream) != cudaSuccess) return ATTN_ERR_CUDA;

  // 1. the query rows of each KV head, stacked over the requests;
  if (s == ATTN_OK) s = attn_host::launch_cascade_gather_q(q, q_stack, B, Hq, Hkv, d, st);
  // 2. those rows against the prefix, once, in prefix_chunks chunks: the
  //    prefix [Hkv, P, d] is the same memory as [Hkv * chunks, P / chunks, d],
  //    and output head h * chunks + c reads the Q rows of KV head h;
  if (s == ATTN_OK)
    s = attn_host::launch_prefill_bf16(q_stack, prefix_k, prefix_v, o_pre, lse_pre, 1,
                                       Hkv * prefix_chunks, Hkv * prefix_chunks, B * (Hq / Hkv),
                                       prefix_len / prefix_chunks, d, 0, scale, prefix_chunks, st);
  // 4. prefix and suffix states merged per row, once the side stream is done.
  if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return ATTN_ERR_CUDA;
  if (s == ATTN_OK)
    s = attn_host::launch_cascade_merge(o_pre, lse_pre, prefix_chunks, o_suf, lse_suf, smax, B, Hq,
                                        Hkv, d, o, lse, st);
  return s;
}
