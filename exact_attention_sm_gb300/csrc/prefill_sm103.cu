// Fused exact-attention prefill for sm_103a: persistent, warp-specialised,
// TMA-fed, tcgen05 MMAs accumulating in tensor memory (TMEM).
//
// The method ("10.3 FlashAttention: IO-aware algorithm design", 10.3.2 tiled
// forward in FlashAttention-2 order; "FlashAttention tiling, online softmax
// and IO" blog, sections 03 and 06): a 128-row Q tile of one (batch, head)
// streams 128-key K/V tiles; per tile
//   S = Q K^T (scaled), m_new = max(m, rowmax S), P = exp(S - m_new),
//   l = l e^(m - m_new) + rowsum P,  O~ = O~ e^(m - m_new) + P V,
// and finally O = O~ / l, LSE = m + ln l.  S and P never leave the SM.
//
// GB300 mapping (the pages' FlashAttention-4 notes, 10.3.6, name the
// primitives; this arrangement is ours).  Two kernels share the method:
// prefill_bf16_kernel (d = 128, below) and prefill_bf16_d64_kernel (d = 64,
// further down: two CTAs per SM, one Q tile each).  For d = 128:
//   * One persistent CTA per SM walks a static list of work items; an item is
//     a pair of consecutive Q tiles (A = rows 256i.., B = rows 256i+128..) of
//     one (batch, head), heaviest items first.  Both tiles consume the same
//     K/V stream, so every K/V tile is loaded once for 256 query rows.
//   * warp 0: TMA producer.  Q_A, Q_B (prefetched for the next item as soon as
//     the current item's last QK^T has read them) and an NS-stage ring of
//     128-byte-swizzled K/V tiles, mbarrier full/empty pairs.
//   * warp 1: MMA issuer (one thread).  TMEM holds S_A, S_B (128 columns
//     each) and O_A, O_B (d columns each).  For K/V tile j it issues
//       PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//     so the tensor core works for one tile while the other tile's softmax
//     runs (ping-pong).  QK^T is SS (Q, K in shared memory); PV is TS: P is
//     read from TMEM, V from shared memory as an MN-major operand.
//   * warps 4-7 / 8-11: softmax of tile A / B; thread r owns query row r
//     (TMEM lane r).  It loads S with tcgen05.ld, masks, keeps (m, l) in
//     registers, writes P as bf16 over S's own TMEM columns, rescales O in
//     TMEM when needed, and at the end of the item writes O / l and the LSE.
// Warps 2-3 only help fill warpgroup 0, which gives registers back
// (setmaxnreg) to the two softmax warpgroups.  Scores stay in the base-2
// domain: log2(e) is folded into the scale and the exponentials run on the
// MUFU ex2 unit.
//
// Conditional rescale (the lecture's FlashAttention-4 notes; the threshold is
// not given there): the running max m used for the exponentials is only
// raised when a tile's max exceeds it by more than 8 (base 2).  Otherwise the
// stale m is kept, P <= 2^8, and because l and O~ share that m the results
// O~ / l and LSE = m + log2 l are unchanged.
//
// Causal: Q tile i reads K/V tiles 0..i only (tiles above the diagonal are
// skipped); the diagonal tile is masked element-wise; keys past Lk are
// masked in the last tile.
//
// Every wait is bounded: after ~2 s the waiting role records
// ATTN_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort flag, drains its own
// in-flight copies / MMAs and the CTA frees its TMEM and exits.  CTAs that
// start while the device status word holds a timeout return at once.
#include <cuda.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace {

using namespace sm103;

constexpr int BM = 128;                // query rows per Q tile (MMA M)
constexpr int BN = 128;                // keys per K/V tile
constexpr int NUM_THREADS = 384;       // 12 warps = 3 warpgroups
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned FULL = 0xffffffffu;

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;             // 128-byte swizzle column blocks per row
  static constexpr int BLOCK_BYTES = BM * 128;  // one 128-row x 128-byte column block
  static constexpr int TILE_BYTES = BM * D * 2; // a Q, K or V tile
  static constexpr int NS = D == 64 ? 5 : 2;    // V pipeline stages
  static constexpr int NSK = D == 64 ? 5 : 3;   // K pipeline stages (K runs further ahead)
  static constexpr int OFF_Q = 0;               // Q_A, Q_B
  static constexpr int OFF_K = 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_LIST = OFF_BAR + 512;           // packed layouts: the item list
  static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t O_COL = 2 * BN;     // S_X at X * 128, O_X at O_COL + X * D
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// s if column c <= kv (visible), else -inf: one compare and one select.
__device__ __forceinline__ float mask_col(float s, int c, int kv) {
  float r;
  asm("{\n\t.reg .pred q;\n\tsetp.gt.s32 q, %2, %3;\n\tselp.f32 %0, 0fFF800000, %1, q;\n\t}"
      : "=f"(r)
      : "f"(s), "r"(c), "r"(kv));
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed two-lane fp32 FMA / add (one instruction for two lanes of work).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Row geometry.  Dense: every (batch, head) has Lq query rows and Lk keys,
// stored head by head ([B * H, L, d]).  Packed ("10.3 FlashAttention",
// 10.3.8, variable-length batching): sequence b owns rows cu_q[b] ..
// cu_q[b+1]-1 of q [total_q, Hq, d] and keys cu_k[b] .. of k, v
// [total_k, Hkv, d]; Lq and Lk are then bounds on the lengths.
// Paged K/V ([LLM book] 10.3.7 block-table addressing; "Lecture 4" 5.2):
// the queries are packed as above, sequence b's keys are tokens 0 ..
// seq_k[b]-1 of the cache [num_pages, block, Hkv, d], token t in block
// row[t / block], slot t % block, where row is the sequence's list of
// physical blocks: table + b * max_pages (a block table), or, in the
// block-sparse-row form of "Lecture 4" 5.2, indices + indptr[b] with
// indptr[b + 1] - indptr[b] entries (table = indices, nnz entries).
struct Geo {
  const int* cu_q;  // nullptr: dense
  const int* cu_k;
  int Lq, Lk, total_q, total_k;
  const int* seq_k;  // paged layouts only
  const int* table;
  int max_pages, num_pages;
  const int* indptr;  // block-sparse-row form (else nullptr: a [B, max_pages] table)
  int nnz;            // entries of indices (block-sparse-row form)
  int block_shift;    // tokens per block = 1 << block_shift
  const void* k_raw;  // gathered layouts: the caches as plain pointers
  const void* v_raw;
};

// Tensor layouts of one launch: dense [B, H, L, d]; packed sequences
// (cu_seqlens); packed queries with K/V in a paged cache, 16-token pages
// fetched by one TMA box each (kPagedLayout) or blocks of any other size
// gathered row by row by the producer warp (kGatherLayout).
constexpr int kDenseLayout = 0, kPackedLayout = 1, kPagedLayout = 2, kGatherLayout = 3;

struct Seq {
  int q_off, lq, k_off, lk;
};

// One sequence's rows; a packed entry outside its bounds is reported and the
// sequence treated as empty (nothing is read or written for it).
template <int kLayout>
__device__ __forceinline__ Seq seq_of(const Geo& g, int b, int* status) {
  if constexpr (kLayout == kDenseLayout) {
    return Seq{0, g.Lq, 0, g.Lk};
  } else if constexpr (kLayout == kPackedLayout) {
    const int q0 = g.cu_q[b], q1 = g.cu_q[b + 1], k0 = g.cu_k[b], k1 = g.cu_k[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > g.total_q || q1 - q0 > g.Lq || k0 < 0 || k1 < k0 ||
        k1 > g.total_k || k1 - k0 > g.Lk) {
      attn::record_status(status, ATTN_ERR_BAD_INDEX);
      return Seq{0, 0, 0, 0};
    }
    return Seq{q0, q1 - q0, k0, k1 - k0};
  } else {
    const int q0 = g.cu_q[b], q1 = g.cu_q[b + 1], lk = g.seq_k[b];
    // Blocks the sequence owns (block-sparse rows: checked against nnz).
    long long nblk = g.max_pages;
    if (g.indptr != nullptr) {
      const int p0 = g.indptr[b], p1 = g.indptr[b + 1];
      nblk = (p0 < 0 || p1 < p0 || p1 > g.nnz) ? -1 : p1 - p0;
    }
    if (q0 < 0 || q1 < q0 || q1 > g.total_q || q1 - q0 > g.Lq || lk < 0 || lk > g.Lk ||
        nblk < 0 || lk > (nblk << g.block_shift)) {
      attn::record_status(status, ATTN_ERR_BAD_INDEX);
      return Seq{0, 0, 0, 0};
    }
    return Seq{q0, q1 - q0, 0, lk};
  }
}

// K/V tiles a 128-row Q tile reads: -1 if the tile has no rows, 0 if its rows
// see no key.  Causal is aligned bottom-right: row r of a sequence sees keys
// j <= r + (lk - lq) (the square rule when lq == lk); tiles past the last
// visible key of the tile's last row are skipped.
__device__ __forceinline__ int kv_tiles(const Seq& sq, int qt, int causal) {
  if (qt * BM >= sq.lq) return -1;
  if (!causal) return (sq.lk + BN - 1) / BN;
  const int last_row = min(sq.lq, (qt + 1) * BM) - 1;
  const int kmax = min(sq.lk - 1, last_row + sq.lk - sq.lq);
  return kmax < 0 ? 0 : kmax / BN + 1;
}

// Last visible key of a row (grow = row within its sequence), and whether K/V
// tile j needs the element-wise mask for any row of Q tile qt.
__device__ __forceinline__ int row_kmax(const Seq& sq, int grow, int causal) {
  return causal ? min(sq.lk - 1, grow + sq.lk - sq.lq) : sq.lk - 1;
}
__device__ __forceinline__ bool tile_needs_mask(const Seq& sq, int qt, int j, int causal) {
  return j * BN + BN - 1 > row_kmax(sq, qt * BM, causal);
}

// The row of physical blocks of sequence b.
__device__ __forceinline__ const int* block_row(const Geo& g, int b) {
  return g.indptr != nullptr ? g.table + g.indptr[b] : g.table + static_cast<size_t>(b) * g.max_pages;
}

// Physical pages of one sequence's K/V tiles (16-token pages), looked up
// one tile ahead: the entries of tile j + 1 are requested when tile j is
// taken, so their latency overlaps the wait for a free ring slot (the ids
// are only used a tile later: the producer is a single thread on the
// critical path of every K/V tile).  Pages past the sequence's length are
// not looked up; they, and entries outside [0, num_pages) (reported as
// ATTN_ERR_BAD_INDEX), take the page coordinate num_pages, which lies
// outside the tensor: TMA writes zeros there and reads nothing, and the
// complete-tx count is the full tile either way.  Other block sizes take
// the gathered layout below.
constexpr int kPage = 16;  // tokens per TMA page
struct PageCursor {
  static constexpr int NP = BN / kPage;  // pages per K/V tile
  const int* row;                        // the sequence's pages
  int lk, j;                             // length; tile whose entries `next` holds
  int next[NP];

  __device__ __forceinline__ void fetch(const Geo& g) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int p = j * NP + i;
      next[i] = p * kPage < lk ? row[p] : g.num_pages;
    }
  }
  __device__ __forceinline__ void begin(const Geo& g, int b, int len) {
    row = block_row(g, b);
    lk = len;
    j = 0;
    fetch(g);
  }
  // Pages of tile j (tiles are taken in order 0, 1, ...).
  __device__ __forceinline__ void take(int (&pg)[NP], const Geo& g, int* status) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const bool needed = (j * NP + i) * kPage < lk;
      pg[i] = next[i];
      if (needed && (pg[i] < 0 || pg[i] >= g.num_pages)) {
        attn::record_status(status, ATTN_ERR_BAD_INDEX);
        pg[i] = g.num_pages;
      }
    }
    ++j;
    fetch(g);
  }
};

// One K or V tile from the paged cache: a 4-D TMA copy {64 columns, KV head,
// 16 slots, page} per page and 64-column block, into the same swizzled rows
// a dense tile occupies (each page is 16 rows, 2 KB per block, so the
// 1024-byte swizzle atoms line up).
template <int KB, int BLOCK_BYTES>
__device__ __forceinline__ void tma_load_pages(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                               const int (&pg)[PageCursor::NP], int kvh) {
#pragma unroll
  for (int i = 0; i < PageCursor::NP; ++i)
#pragma unroll
    for (int kb = 0; kb < KB; ++kb)
      tma_load_4d(dst + kb * BLOCK_BYTES + i * kPage * 128, map, bar, kb * 64, kvh, 0, pg[i]);
}

// Blocks of other sizes ("Lecture 4" 5.2's block size 4, the radix tree's
// 1, or 32 to 128) are gathered row by row.  GatherCursor holds the block ids of
// one sequence's next 128-token tile, np = 128 / block of them, entry
// k * 32 + lane in register ids[k] of that lane; they are loaded one tile
// ahead (coalesced), so their latency overlaps the current tile's copies.
// Ids past the sequence's length are -1.
struct GatherCursor {
  const int* row;  // the sequence's blocks
  int lk, j, shift, np;
  int ids[4];      // tile j's block ids (np <= 128 = 4 x 32)

  __device__ __forceinline__ void fetch(int lane) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = k * 32 + lane, p = j * np + e;
      ids[k] = e < np && (p << shift) < lk ? row[p] : -1;
    }
  }
  __device__ __forceinline__ void begin(const Geo& g, int b, int len, int lane) {
    row = block_row(g, b);
    lk = len;
    j = 0;
    shift = g.block_shift;
    np = BN >> shift;
    fetch(lane);
  }
  __device__ __forceinline__ void advance(int lane) {
    ++j;
    fetch(lane);
  }
};

// One 128-row tile of K or V (tile c.j of the cursor's sequence) gathered
// with 16-byte cp.async copies by the 32 lanes of the producer warp: 8 lanes
// per row and 4 rows per instruction, so each instruction reads whole
// 128-byte rows; rows go straight into the tile's 128-byte swizzle (chunk c
// of row r at c ^ (r % 8)).  Row r's block id comes from lane (r / block) %
// 32 by a shuffle (for a given instruction every lane wants the same ids
// register).  Rows past the sequence's length, and rows whose block is
// outside [0, num_pages) (reported), are zero-filled.  The copies form one
// cp.async group; GatherRetire publishes the tile once they have landed.
template <int KB>
__device__ __forceinline__ void gather_tile(uint8_t* dst, const __nv_bfloat16* base,
                                            const Geo& g, const GatherCursor& c, int kvh, int Hkv,
                                            int lane, int* status) {
  constexpr int D = KB * 64;
  const int chunk = lane & 7;
  const uint32_t sdst = smem_u32(dst);
#pragma unroll 8
  for (int i = 0; i < BN / 4; ++i) {
    const int r = 4 * i + (lane >> 3);
    const int idx = r >> c.shift;  // entry of the tile's ids
    const int k = (4 * i >> c.shift) >> 5;  // the same for every lane
    const int src_reg = k == 0 ? c.ids[0] : k == 1 ? c.ids[1] : k == 2 ? c.ids[2] : c.ids[3];
    int blk = __shfl_sync(0xffffffffu, src_reg, idx & 31);
    const int t = c.j * BN + r;
    if (t < c.lk && (blk < 0 || blk >= g.num_pages)) {
      attn::record_status(status, ATTN_ERR_BAD_INDEX);
      blk = -1;
    }
    const bool ok = t < c.lk && blk >= 0;
    const size_t src =
        ok ? ((static_cast<size_t>(blk) << c.shift) + (t & ((1 << c.shift) - 1))) *
                     static_cast<size_t>(Hkv) * D +
                 static_cast<size_t>(kvh) * D
           : 0;
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const uint32_t d_addr = sdst + kb * (BM * 128) + r * 128 + ((chunk ^ (r & 7)) << 4);
      const __nv_bfloat16* s_ptr = base + src + kb * 64 + chunk * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d_addr), "l"(s_ptr),
                   "r"(ok ? 16 : 0)
                   : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Publishes gathered tiles to the tensor core one tile late: after tile t's
// group is committed, tile t - 1's copies are waited for (wait_group 1),
// made visible to the async proxy (fence.proxy.async by every writing lane)
// and its full barrier arrived on (count 1).  flush() publishes the last
// one; the producer calls it before any wait that is not already satisfied,
// so a consumer never waits on a tile the producer is holding back.
struct GatherRetire {
  uint64_t* pend = nullptr;
  __device__ __forceinline__ void publish(int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(pend);
  }
  __device__ __forceinline__ void committed(uint64_t* full, int lane) {
    if (pend != nullptr) {
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      publish(lane);
    }
    pend = full;
  }
  __device__ __forceinline__ void flush(int lane) {
    if (pend != nullptr) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      publish(lane);
      pend = nullptr;
    }
  }
};

// Paged cache: the slots of a sequence's last block past its length may hold
// anything, and P = 0 times a NaN there would still reach O through the PV
// MMA.  Before P of the tile holding the last key is handed over, the softmax
// thread of each such row clears it in the landed V tile (tile rows
// [lk - j BN, round_up(lk, block) - j BN)); blocks wholly past the length
// were zero-filled by TMA.  (Gathered tiles are zero-filled past the length.)
template <int KB, int BLOCK_BYTES>
__device__ __forceinline__ void clear_v_tail(uint8_t* vtile, int row, int lk, int j, int shift) {
  const int lo = lk - j * BN;
  const int hi = min(BN, ((((lk - 1) >> shift) + 1) << shift) - j * BN);
  if (row >= lo && row < hi) {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      uint4* r = reinterpret_cast<uint4*>(vtile + kb * BLOCK_BYTES + row * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) r[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();  // the generic stores, then the tensor core's reads
}

// Whether tile j of a sequence of lk keys holds its last key inside a
// partial block (the case clear_v_tail handles).
__device__ __forceinline__ bool has_v_tail(int lk, int j, int shift) {
  return (lk & ((1 << shift) - 1)) != 0 && (lk - 1) / BN == j;
}

struct Item {
  int bh, qt[2], n[2];  // n[x] == 0: tile x has no K/V work
  bool zero[2];         // tile x has rows that see no key: O = 0, LSE = -inf
  Seq sq;
};

// Work-item order and assignment.
//  * Long causal rows (more than kGroupedMaxPairs pairs per head): items are
//    listed heaviest pair first across all heads and dealt round-robin to the
//    persistent CTAs, odd rounds in reverse CTA order (the d = 128 kernel,
//    through build_item_list), which keeps them balanced when the work per
//    item varies.
//  * Packed (variable-length) batches: each CTA works through its list from
//    build_item_list (units sorted by decreasing cost, dealt round-robin with
//    odd rounds reversed); batches too large for the list fall back to the
//    round-robin order of long causal rows.
//  * Short rows or non-causal: items are listed head by head and every CTA
//    takes one contiguous run of them, so the pairs of a head run back to back
//    on the same SM and re-read that head's K/V from L2; each run spans whole
//    heads (up to its ends), so every CTA gets a similar mix of pair weights.
constexpr int kGroupedMaxPairs = 16;

struct Schedule {
  bool grouped;
  int first, last, step;  // items first, first+step, ... < last
};

__device__ __forceinline__ Schedule make_schedule(int num_items, int num_pairs, int causal,
                                                  bool packed) {
  Schedule sc;
  sc.grouped = !packed && (!causal || num_pairs <= kGroupedMaxPairs);
  if (sc.grouped) {
    sc.first = static_cast<int>(static_cast<long long>(num_items) * blockIdx.x / gridDim.x);
    sc.last = static_cast<int>(static_cast<long long>(num_items) * (blockIdx.x + 1) / gridDim.x);
    sc.step = 1;
  } else {
    sc.first = blockIdx.x;
    sc.last = num_items;
    sc.step = gridDim.x;
  }
  return sc;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// The item slot of this CTA's round-robin position it = r * gridDim.x +
// blockIdx.x: even rounds deal slots in CTA order, odd rounds in reverse.
__device__ __forceinline__ int dealt_slot(int it) {
  const int G = gridDim.x, r = it / G;
  return (r & 1) ? r * G + (G - 1 - static_cast<int>(blockIdx.x)) : it;
}

// Each CTA's list of work items, built once in the prologue (packed batches,
// and the d = 128 kernel's long causal rows of the dense layout, whose equal
// rows already come heaviest first: their list skips the sort).
// Unit u is Q-tile position num_pos - 1 - u / B of sequence u % B (u counts
// heaviest position first, as the natural order does); a position is one Q
// tile, or a pair of Q tiles (kTiles = 2).  A unit's cost is the K/V tiles its
// Q tiles read plus one per Q tile present (its Q load and output write).
// Every CTA sorts the units by decreasing cost with the same deterministic,
// stable counting sort, lists the items (unit, head) in that order, and takes
// the items of its round-robin positions, odd rounds dealt in reverse CTA
// order: each CTA's sum of costs comes out close to the mean (a static form
// of longest-processing-time-first).  An entry is bh | position << 20, or
// ~0u for a position without work.  Batches with more than kMaxSortUnits
// units or kMaxListItems positions per CTA keep the natural order.
constexpr int kMaxSortUnits = 4096;
constexpr int kCostBins = 2048;  // higher costs share the top bin
constexpr int kMaxListItems = 256;  // 1 KB: what the d = 128 kernel's three K stages leave
constexpr int kListBytes = kMaxListItems * 4;
// cost[kMaxSortUnits], start[kCostBins] (int), order[kMaxSortUnits] (uint16)
constexpr int kSortScratchBytes = (kMaxSortUnits + kCostBins) * 4 + kMaxSortUnits * 2;

template <int kLayout, int kTiles>
__device__ __forceinline__ int unit_cost(const Geo& geo, int u, int B, int num_pos, int causal,
                                         int* status) {
  const int pos = num_pos - 1 - u / B;
  const Seq sq = seq_of<kLayout>(geo, u % B, status);
  int c = 0;
#pragma unroll
  for (int x = 0; x < kTiles; ++x) {
    const int kv = kv_tiles(sq, kTiles * pos + x, causal);
    if (kv >= 0) c += kv + 1;
  }
  return min(c, kCostBins - 1);
}

// Called by every thread of the CTA (it holds block-wide barriers); scratch
// is kSortScratchBytes of shared memory, free until the list is built.
// Returns the list length (this CTA's positions up to its last item with
// work), or -1 for a batch that keeps the natural order.
template <int kLayout, int kTiles>
__device__ int build_item_list(uint32_t* list, uint8_t* scratch, int BH, int Hq, int num_pos,
                               const Geo& geo, int causal, int* status) {
  const int B = BH / Hq, U = B * num_pos, G = gridDim.x;
  const long long num_items = static_cast<long long>(BH) * num_pos;
  const long long npos = (num_items + G - 1) / G;
  if (npos > kMaxListItems || BH >= (1 << 20) || num_pos >= (1 << 12)) return -1;
  if constexpr (kLayout == kDenseLayout) {
    // Equal rows: the natural order (position-major) is already heaviest
    // first and every unit has work; only the dealing changes.
    for (int k = threadIdx.x; k < npos; k += blockDim.x) {
      const int slot = dealt_slot(k * G + static_cast<int>(blockIdx.x));
      list[k] = slot < num_items ? static_cast<uint32_t>(slot % BH) |
                                       static_cast<uint32_t>(num_pos - 1 - slot / BH) << 20
                                 : ~0u;
    }
    __syncthreads();
    return static_cast<int>(npos);
  }
  if (U > kMaxSortUnits) return -1;
  int* cost = reinterpret_cast<int*>(scratch);
  int* start = cost + kMaxSortUnits;  // per cost: count, then first position
  uint16_t* order = reinterpret_cast<uint16_t*>(start + kCostBins);
  const int nbins = min(kCostBins, kTiles * ((geo.Lk + BN - 1) / BN + 1) + 1);
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) start[i] = 0;
  for (int u = threadIdx.x; u < U; u += blockDim.x)
    cost[u] = unit_cost<kLayout, kTiles>(geo, u, B, num_pos, causal, status);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned below = (1u << lane) - 1u;
    // Counts: 32 units at a time; the lowest lane of each group of equal
    // costs adds the group's size.
    for (int base = 0; base < U; base += 32) {
      const int c = base + lane < U ? cost[base + lane] : -1;
      const unsigned same = __match_any_sync(FULL, c);
      if (c >= 0 && (same & below) == 0) start[c] += __popc(same);
      __syncwarp();
    }
    // First position of each cost in decreasing cost order: lane L sums the
    // bins at descending positions [L S, (L + 1) S), a warp scan gives each
    // lane its offset, and the lane rewrites its bins as running offsets.
    const int S = (nbins + 31) / 32, p0 = lane * S, p1 = min(nbins, p0 + S);
    int sum = 0;
    for (int p = p0; p < p1; ++p) sum += start[nbins - 1 - p];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - sum;
    for (int p = p0; p < p1; ++p) {
      const int cnt = start[nbins - 1 - p];
      start[nbins - 1 - p] = run;
      run += cnt;
    }
    __syncwarp();
    // Stable scatter, 32 units at a time in order of u.
    for (int base = 0; base < U; base += 32) {
      const int c = base + lane < U ? cost[base + lane] : -1;
      const unsigned same = __match_any_sync(FULL, c);
      if (c >= 0) order[start[c] + __popc(same & below)] = static_cast<uint16_t>(base + lane);
      __syncwarp();
      if (c >= 0 && (same & below) == 0) start[c] += __popc(same);
      __syncwarp();
    }
    if (lane == 0) start[0] = 0;  // from here on: the list length
  }
  __syncthreads();
  for (int k = threadIdx.x; k < npos; k += blockDim.x) {
    const int slot = dealt_slot(k * G + static_cast<int>(blockIdx.x));
    uint32_t e = ~0u;
    if (slot < num_items) {
      const int u = order[slot / Hq];
      if (cost[u] > 0) {
        e = static_cast<uint32_t>((u % B) * Hq + slot % Hq) |
            static_cast<uint32_t>(num_pos - 1 - u / B) << 20;
        atomicMax(&start[0], k + 1);
      }
    }
    list[k] = e;
  }
  __syncthreads();
  return start[0];
}

// With an item list (`list`: its shared-memory address, 0 for none): item
// `it` is the list's entry it.
template <int kLayout>
__device__ __forceinline__ Item decode_item(int it, bool grouped, int BH, int Hq, int num_pairs,
                                            const Geo& geo, int causal, int* status,
                                            uint32_t list) {
  Item w;
  int pair;
  if (list != 0) {
    const uint32_t e = ld_shared_u32(list + 4u * it);
    if (e == ~0u) {  // a position without work
      w.bh = 0;
      w.sq = Seq{0, 0, 0, 0};
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        w.qt[x] = x;
        w.n[x] = 0;
        w.zero[x] = false;
      }
      return w;
    }
    w.bh = static_cast<int>(e & 0xFFFFFu);
    pair = static_cast<int>(e >> 20);
  } else if (grouped) {
    w.bh = it / num_pairs;
    pair = num_pairs - 1 - it % num_pairs;
  } else {
    pair = num_pairs - 1 - it / BH;
    w.bh = it % BH;
  }
  w.sq = seq_of<kLayout>(geo, w.bh / Hq, status);
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    w.qt[x] = 2 * pair + x;
    const int kv = kv_tiles(w.sq, w.qt[x], causal);
    w.n[x] = kv > 0 ? kv : 0;
    w.zero[x] = kv == 0;
  }
  return w;
}

template <int D, int kLayout>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
                        float* __restrict__ lse, int BH, int Hq, int Hkv, const Geo geo,
                        int causal, float scale_log2, int q_div, int* status) {
  using C = Cfg<D>;
  constexpr int NS = C::NS, NSK = C::NSK;
  constexpr bool kPacked = kLayout != kDenseLayout;
  constexpr bool kPaged = kLayout == kPagedLayout;
  constexpr bool kGather = kLayout == kGatherLayout;  // K/V rows gathered by warp 0
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;            // [2]
  uint64_t* q_empty = q_full + 2;     // [2]
  uint64_t* k_full = q_empty + 2;     // [NSK]
  uint64_t* v_full = k_full + NSK;    // [NS]
  uint64_t* k_empty = v_full + NS;    // [NSK] the slot's last QK^T done
  uint64_t* v_empty = k_empty + NSK;  // [NS] the slot's last PV done
  uint64_t* s_full = v_empty + NS;    // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* o_done = p_full + 2;      // [2]
  uint64_t* o_free = o_done + 2;      // [2]
  uint64_t* drain = o_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_qt = (geo.Lq + BM - 1) / BM;
  const int num_pairs = (num_qt + 1) / 2;
  const int num_items = BH * num_pairs;
  constexpr bool packed = kPacked;
  const int group = Hq / Hkv;
  Schedule sched = make_schedule(num_items, num_pairs, causal, kPacked);

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_free[x], 128);
    }
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = (status != nullptr &&
                   *reinterpret_cast<volatile int*>(status) == ATTN_ERR_DEVICE_TIMEOUT) ? 2 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (*abort_flag == 2) return;
  // Packed batches and long causal rows: this CTA's item list (the K ring,
  // not yet in use, is the sort's scratch); `list` is its shared-memory
  // address, 0 if the batch keeps the natural order.
  uint32_t list = 0;
  if (!sched.grouped) {
    static_assert(kSortScratchBytes <= NSK * C::TILE_BYTES, "sort scratch fits the K ring");
    const int n = build_item_list<kLayout, 2>(reinterpret_cast<uint32_t*>(smem + C::OFF_LIST),
                                              smem + C::OFF_K, BH, Hq, num_pairs, geo, causal,
                                              status);
    if (n >= 0) {
      list = sbase + C::OFF_LIST;
      sched.first = 0;
      sched.last = n;
      sched.step = 1;
    }
  }
  auto item_of = [&](int it) {
    return decode_item<kLayout>(it, sched.grouped, BH, Hq, num_pairs, geo, causal, status, list);
  };
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // (gathered layouts: the whole warp copies K/V rows; lane 0 alone issues
    // the Q copies and the barrier bookkeeping of TMA)
    if (kGather || lane == 0) {
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        if constexpr (!kGather) {
          prefetch_tmap(&tm_k);
          prefetch_tmap(&tm_v);
        }
      }
      // A wait every lane takes (the lanes of a gathering warp stay together;
      // a gathered tile held back is published before the warp blocks).
      GatherRetire retire;
      auto pwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if constexpr (kGather) {
          if (__all_sync(FULL, mbar_test_wait(bar, parity))) return true;
          retire.flush(lane);
          return __all_sync(FULL, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
        } else {
          return mbar_wait(bar, parity, abort_flag, kWaitLimitNs);
        }
      };
      int g = 0;                // K/V tiles issued (ring position)
      int nq[2] = {0, 0};       // Q tiles issued per slot
      bool ok = true;
      for (int it = sched.first; ok && it < sched.last; it += sched.step) {
        const Item w = item_of(it);
        const int nmax = max(w.n[0], w.n[1]);
        if (nmax == 0) continue;
        const int h = w.bh % Hq;
        // TMA coordinates (rows, heads): dense tensors are [heads, rows],
        // packed ones [rows, heads].
        const int kv_c1 = packed ? h / group : 0;
        const int kv_c2 = packed ? w.sq.k_off : (w.bh / Hq) * Hkv + h / group;
        PageCursor pages;
        if constexpr (kPaged) pages.begin(geo, w.bh / Hq, w.sq.lk);
        GatherCursor gc;  // gathered layouts: the item's block ids, one tile ahead
        if constexpr (kGather) gc.begin(geo, w.bh / Hq, w.sq.lk, lane);
        // K/V tile j of this item into the next ring slot.  The K and V halves
        // of a slot free separately: K after the slot's last QK^T, which the
        // MMA issuer commits one K/V tile before the slot's last PV, so K(j)
        // goes out as soon as V(j - 1) has (the two frees come together).
        auto issue_kv = [&](int j) -> bool {
          const int sk = g % NSK, st = g % NS;  // K slot, V slot
          const uint32_t phk = ((g / NSK) + 1) & 1, ph = ((g / NS) + 1) & 1;
          // Giving up between the K and V copies: K(j) lands before the
          // producer moves on (the drain below covers whole tiles only).
          auto drain_k = [&](int slot) {
            int no_abort = 0;
            mbar_wait(&k_full[slot], (g / NSK) & 1, &no_abort, kWaitLimitNs);
            return false;
          };
          uint8_t* kdst = smem + C::OFF_K + sk * C::TILE_BYTES;
          uint8_t* vdst = smem + C::OFF_V + st * C::TILE_BYTES;
          if (g >= NSK && !pwait(&k_empty[sk], phk)) return false;
          if constexpr (kGather) {  // tile j of the item (the cursor's tile); V: warp 3
            gather_tile<C::KB>(kdst, static_cast<const __nv_bfloat16*>(geo.k_raw), geo, gc, kv_c1,
                               Hkv, lane, status);
            retire.committed(&k_full[sk], lane);
            gc.advance(lane);
            (void)vdst;
            (void)ph;
          } else if constexpr (kPaged) {
            int pg[PageCursor::NP];
            pages.take(pg, geo, status);  // tile j (tiles are issued in order)
            mbar_arrive_expect_tx(&k_full[sk], C::TILE_BYTES);
            tma_load_pages<C::KB, C::BLOCK_BYTES>(kdst, &tm_k, &k_full[sk], pg, kv_c1);
            if (g >= NS && !mbar_wait(&v_empty[st], ph, abort_flag, kWaitLimitNs))
              return drain_k(sk);
            mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
            tma_load_pages<C::KB, C::BLOCK_BYTES>(vdst, &tm_v, &v_full[st], pg, kv_c1);
          } else {
            mbar_arrive_expect_tx(&k_full[sk], C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_3d(kdst + kb * C::BLOCK_BYTES, &tm_k, &k_full[sk], kb * 64,
                          packed ? kv_c1 : j * BN, packed ? kv_c2 + j * BN : kv_c2);
            if (g >= NS && !mbar_wait(&v_empty[st], ph, abort_flag, kWaitLimitNs))
              return drain_k(sk);
            mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_3d(vdst + kb * C::BLOCK_BYTES, &tm_v, &v_full[st], kb * 64,
                          packed ? kv_c1 : j * BN, packed ? kv_c2 + j * BN : kv_c2);
          }
          ++g;
          return true;
        };
        // The first K/V tile goes out before the Q tiles: its slot frees while
        // the previous item is still finishing, and Q waits for that item's
        // last QK^T.
        ok = issue_kv(0);
        for (int x = 0; x < 2 && ok; ++x) {
          if (w.n[x] == 0) continue;
          if (nq[x] > 0 && !pwait(&q_empty[x], (nq[x] - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&q_full[x], C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_3d(smem + C::OFF_Q + x * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tm_q,
                          &q_full[x], kb * 64, packed ? h : w.qt[x] * BM,
                          packed ? w.sq.q_off + w.qt[x] * BM : w.bh / q_div);
          }
          ++nq[x];
        }
        for (int j = 1; ok && j < nmax; ++j) ok = issue_kv(j);
      }
      if (!ok && lane == 0) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: every issued copy has landed before the CTA may exit (these
      // waits ignore the abort flag; TMA copies always complete).
      if constexpr (kGather) retire.flush(lane);
      int no_abort = 0;
      for (int x = 0; x < 2; ++x)
        if (nq[x] > 0) mbar_wait(&q_full[x], (nq[x] - 1) & 1, &no_abort, kWaitLimitNs);
      for (int t = g > NSK ? g - NSK : 0; t < g; ++t)
        mbar_wait(&k_full[t % NSK], (t / NSK) & 1, &no_abort, kWaitLimitNs);
      if constexpr (!kGather)
        for (int t = g > NS ? g - NS : 0; t < g; ++t)
          mbar_wait(&v_full[t % NS], (t / NS) & 1, &no_abort, kWaitLimitNs);
    }
  } else if (kGather && warp == 3) {
    // ------------------------------------------------------------ V gatherer
    // Gathered layouts: this warp copies the V rows, warp 0 the K rows (one
    // warp's 16-byte copies per tile are what limits a gathered stream).
    GatherRetire retire;
    auto pwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (__all_sync(FULL, mbar_test_wait(bar, parity))) return true;
      retire.flush(lane);
      return __all_sync(FULL, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
    };
    int g = 0;  // V tiles issued (ring position, as warp 0 counts K/V tiles)
    bool ok = true;
    for (int it = sched.first; ok && it < sched.last; it += sched.step) {
      const Item w = item_of(it);
      const int nmax = max(w.n[0], w.n[1]);
      if (nmax == 0) continue;
      const int kv_c1 = (w.bh % Hq) / group;
      GatherCursor gc;
      gc.begin(geo, w.bh / Hq, w.sq.lk, lane);
      for (int j = 0; j < nmax; ++j, ++g) {
        const int st = g % NS;
        if (g >= NS && !pwait(&v_empty[st], ((g / NS) + 1) & 1)) {
          ok = false;
          break;
        }
        gather_tile<C::KB>(smem + C::OFF_V + st * C::TILE_BYTES,
                           static_cast<const __nv_bfloat16*>(geo.v_raw), geo, gc, kv_c1, Hkv, lane,
                           status);
        retire.committed(&v_full[st], lane);
        gc.advance(lane);
      }
    }
    if (!ok && lane == 0) {
      attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
    retire.flush(lane);
    int no_abort = 0;
    for (int t = g > NS ? g - NS : 0; t < g; ++t)
      mbar_wait(&v_full[t % NS], (t / NS) & 1, &no_abort, kWaitLimitNs);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      int g = 0;                  // K/V tiles consumed (ring position)
      int nitem[2] = {0, 0};      // items started per tile slot
      int np[2] = {0, 0};         // P tiles consumed per slot
      bool ok = true;

      // S_x = Q_x K^T for the K tile in ring slot st.
      // Descriptors are built once; a K step or a ring slot only moves the
      // start-address field (bits 0-13, address >> 4), so each MMA costs one
      // 64-bit add of a constant.  Shared addresses stay below 256 KB, so the
      // field never carries into the neighbouring bits.
      const uint64_t q_desc0 = smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(sbase + C::OFF_V, C::BLOCK_BYTES, 1024);
      constexpr uint64_t kTileStep = C::TILE_BYTES >> 4;
      auto issue_qk = [&](int x, int st, bool last) {
        const uint64_t qd = q_desc0 + static_cast<uint64_t>(x) * kTileStep;
        const uint64_t kd = k_desc0 + static_cast<uint64_t>(st) * kTileStep;
        const uint32_t d_tmem = tmem + x * BN;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          constexpr uint32_t kBlk = C::BLOCK_BYTES >> 4;
          const uint64_t off = (k >> 2) * kBlk + (k & 3) * 2;  // (k>>2) blocks + (k&3)*32 bytes
          mma_bf16_ss(d_tmem, qd + off, kd + off, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[x]);
        if (last) mma_commit(&q_empty[x]);  // Q_x may be refilled for the next item
      };
      // O_x (+)= P_x V for the V tile in ring slot st; P_x sits in S_x's columns.
      // B = V, MN-major: 16 keys = two 8-row groups of 128 bytes (2048 bytes
      // per K step); LBO steps to the next 64-column block of d.
      auto issue_pv = [&](int x, int st, bool accumulate) {
        const uint64_t vd = v_desc0 + static_cast<uint64_t>(st) * kTileStep;
        const uint32_t d_tmem = tmem + C::O_COL + x * D;
        const uint32_t a_tmem = tmem + x * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ts(d_tmem, a_tmem + k * 8, vd + static_cast<uint64_t>(k) * 128, idesc_pv,
                      (accumulate || k > 0) ? 1u : 0u);
      };

      for (int it = sched.first; ok && it < sched.last; it += sched.step) {
        const Item w = item_of(it);
        const int nmax = max(w.n[0], w.n[1]);
        if (nmax == 0) continue;
        // First QK^T of each present tile.
        if (!mbar_wait(&k_full[g % NSK], (g / NSK) & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
        for (int x = 0; x < 2 && ok; ++x) {
          if (w.n[x] == 0) continue;
          if (!mbar_wait(&q_full[x], nitem[x] & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
          tc_fence_after();
          issue_qk(x, g % NSK, w.n[x] == 1);
        }
        if (ok) mma_commit(&k_empty[g % NSK]);  // K(0) of the item is read
        for (int j = 0; ok && j < nmax; ++j) {
          const int st = (g + j) % NS, ph = ((g + j) / NS) & 1;
          const int st1 = (g + j + 1) % NSK, ph1 = ((g + j + 1) / NSK) & 1;  // K slot
          bool v_ready = false, k_ready = false;  // each K/V tile is waited for once
          for (int x = 0; x < 2; ++x) {
            if (j >= w.n[x]) continue;
            if (!mbar_wait(&p_full[x], np[x] & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
            ++np[x];
            if (j == 0 && nitem[x] > 0 &&
                !mbar_wait(&o_free[x], (nitem[x] - 1) & 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            if (!v_ready && !mbar_wait(&v_full[st], ph, abort_flag, kWaitLimitNs)) { ok = false; break; }
            v_ready = true;
            tc_fence_after();
            issue_pv(x, st, j > 0);
            if (j + 1 < w.n[x]) {
              if (!k_ready && !mbar_wait(&k_full[st1], ph1, abort_flag, kWaitLimitNs)) { ok = false; break; }
              k_ready = true;
              tc_fence_after();
              issue_qk(x, st1, j + 2 == w.n[x]);
            } else {
              mma_commit(&o_done[x]);
            }
          }
          if (ok) {
            if (j + 1 < nmax) mma_commit(&k_empty[st1]);  // K(j + 1) is read
            mma_commit(&v_empty[st]);
          }
        }
        g += nmax;
        for (int x = 0; x < 2; ++x)
          if (w.n[x] > 0) ++nitem[x];
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: all MMAs issued by this thread are complete before teardown.
      int no_abort = 0;
      mma_commit(drain);
      mbar_wait(drain, 0, &no_abort, kWaitLimitNs);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------------------ softmax warps
    const int x = (warp - 4) >> 2;     // 0: tile A (warps 4-7), 1: tile B (warps 8-11)
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;  // row within the Q tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + x * BN;
    const uint32_t o_addr = tmem + lane_off + C::O_COL + x * D;
    int ns = 0, nitem = 0;
    int g0 = 0;  // K/V tiles of the items before this one (the producer's ring count)
    bool ok = true;
    for (int it = sched.first; ok && it < sched.last; it += sched.step) {
      const Item w = item_of(it);
      const int n = w.n[x];
      const int g_item = g0;
      g0 += max(w.n[0], w.n[1]);
      const int grow = w.qt[x] * BM + row;
      const int h = w.bh % Hq;
      // Output row: dense [heads, rows], packed [rows, heads].
      const size_t orow_index = packed ? static_cast<size_t>(w.sq.q_off + grow) * Hq + h
                                       : static_cast<size_t>(w.bh) * geo.Lq + grow;
      if (n == 0) {
        if constexpr (kPacked) {
          if (w.zero[x] && grow < w.sq.lq) {  // rows that see no key
            uint4* op = reinterpret_cast<uint4*>(o + orow_index * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr) lse[orow_index] = -INFINITY;
          }
        }
        continue;
      }
      float m_s = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        ok = __all_sync(FULL, mbar_wait(&s_full[x], ns & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        ++ns;
        tc_fence_after();
        // S and, from the load itself, the maximum of each 32-column chunk.
        float sr[4][32], cmax[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(s_addr + c * 32, sr[c], cmax[c]);
        tmem_ld_wait();
        float* s = &sr[0][0];

        const bool need_mask = kPacked ? tile_needs_mask(w.sq, w.qt[x], j, causal)
                                       : (j == n - 1) && (causal || (geo.Lk % BN) != 0);
        if (need_mask) {
          // Element mask by compare-and-select (straight-line, no branches).
          const int kv = row_kmax(w.sq, grow, causal) - j * BN;  // last visible column
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = mask_col(s[c], c, kv);
        }
        // Row max: an unmasked tile takes it from the load; a masked one
        // reduces the masked scores as 8 independent chains.
        float mt = fmaxf(fmaxf(cmax[0], cmax[1]), fmaxf(cmax[2], cmax[3]));
        if (need_mask) {
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int c = 16; c < BN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
          mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        }
        const float mt_s = mt * scale_log2;
        float alpha = 1.f;
        if (mt_s > m_s + kRescaleThreshold) {
          alpha = ex2(m_s - mt_s);  // 0 on the first tile (m_s = -inf)
          m_s = mt_s;
        }
        // p = 2^(s * scale * log2e - m): paired FMAs, MUFU ex2, paired adds
        // into 4 independent row-sum chains; P goes to TMEM in 16-column
        // chunks (8 bf16x2 words) over S's own columns as soon as a chunk is
        // packed, which keeps few registers live next to S.
        // A row that sees no key yet (every score -inf, possible when causal
        // is aligned bottom-right with lq > lk) keeps m = -inf: subtract 0
        // instead so that its p are exp(-inf) = 0, not NaN.
        const float m_sub = kPacked && m_s == -INFINITY ? 0.f : m_s;
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_sub, -m_sub);
        float2 rs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < BN / 16; ++ch) {
          uint32_t pk[8];
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            float2 t = ffma2(make_float2(s[ch * 16 + c], s[ch * 16 + c + 1]), sc2, nm2);
            t.x = ex2(t.x);
            t.y = ex2(t.y);
            rs[(c >> 1) & 3] = fadd2(rs[(c >> 1) & 3], t);
            pk[c >> 1] = attn::pack_bf16x2(t.x, t.y);
          }
          tmem_st8(s_addr + ch * 8, pk);
        }
        const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
        const float2 r = fadd2(r01, r23);
        l = l * alpha + (r.x + r.y);
        if (j > 0 && __any_sync(FULL, alpha != 1.f)) {
          // O <- alpha O before PV of this tile is issued; PV of the previous
          // tile completed before S of this one (issue order).
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o32[32];
            tmem_ld32(o_addr + c * 32, o32);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
            tmem_st32(o_addr + c * 32, o32);
          }
        }
        if constexpr (kPaged) {
          if (has_v_tail(w.sq.lk, j, geo.block_shift)) {
            const int gt = g_item + j;  // this K/V tile's ring position
            ok = __all_sync(FULL, mbar_wait(&v_full[gt % NS], (gt / NS) & 1, abort_flag,
                                            kWaitLimitNs));
            clear_v_tail<C::KB, C::BLOCK_BYTES>(smem + C::OFF_V + (gt % NS) * C::TILE_BYTES, row,
                                                w.sq.lk, j, geo.block_shift);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
      }
      if (ok) ok = __all_sync(FULL, mbar_wait(&o_done[x], nitem & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool live = grow < w.sq.lq;
      __nv_bfloat16* orow = o + (live ? orow_index : 0) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(o_addr + c * 32, r);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            uint4 q4;
            q4.x = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 0]) * inv, __uint_as_float(r[v8 * 8 + 1]) * inv);
            q4.y = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 2]) * inv, __uint_as_float(r[v8 * 8 + 3]) * inv);
            q4.z = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 4]) * inv, __uint_as_float(r[v8 * 8 + 5]) * inv);
            q4.w = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 6]) * inv, __uint_as_float(r[v8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + v8 * 8) = q4;
          }
        }
      }
      if (live && lse != nullptr)
        lse[orow_index] =
            l > 0.f ? (m_s + log2f(l)) * attn::kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&o_free[x]);
      ++nitem;
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// d = 64: two CTAs per SM, each streaming K/V for ONE 128-row Q tile.
//
// A d = 64 tile step is short on the tensor core (QK^T 4 MMAs, PV 8), so a
// CTA that interleaves two Q tiles spends most of a step on barrier tests
// and on one tile waiting for the other.  Here each CTA owns 256 TMEM
// columns and runs one independent pipeline; the two CTAs on an SM fill each
// other's gaps on the tensor core and on the MUFU.
//   TMEM columns (per CTA): S 0..127, P 128..191 (bf16 pairs), O 192..255.
// P has its own columns, so S(t+1) is written while the softmax still works
// on P(t).  Two threads issue the MMAs: one the QK^T groups, one the PV
// groups.  tcgen05.mma issue blocks while the tensor pipe is busy (its queue
// holds about one MMA), so with a single issuer S(t+1) waited behind the
// eight MMAs of PV(t-1); with two, each group goes out as soon as its inputs
// are ready and the pipe interleaves them.
//   QK issuer: S(t) once K(t) has landed (k_full) and the softmax has read
//              S(t-1) (s_read); commits s_full and k_done.
//   PV issuer: PV(t) once V(t) has landed (v_full) and the softmax wrote P(t)
//              (p_ready); commits pv_done (V slot free, P and O may be
//              rewritten; after an item's last PV, its O is final).
// Epilogue (dense layout): the softmax threads write O / l as bf16 rows into
// the item's Q buffer (its last QK^T is done) in the tensor map's 128-byte
// swizzle, and the Q producer stores the tile with one TMA copy before it
// refills that buffer; rows past L are clipped by the map.  Packed and paged
// layouts store rows directly (a tile may reach into the next sequence).
// Work items are single Q tiles.
struct Cfg64 {
  static constexpr int D = 64;
  static constexpr int THREADS = 256;            // 8 warps; two CTAs per SM
  static constexpr int TILE_BYTES = BM * D * 2;  // 16 KB: one 128 x 128-byte swizzled block
  static constexpr int NS = 2;                   // K/V pipeline stages
  static constexpr int NQ = 2;                   // Q buffers
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NQ * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_LIST = OFF_BAR + 256;  // packed layouts: the item list
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr uint32_t COLS = 256;
  static constexpr uint32_t P_COL = BN;
  static constexpr uint32_t O_COL = BN + BN / 2;
  static constexpr uint32_t kSoftmaxWarps = 4;
};

struct Item1 {
  int bh, qt, n;  // n == 0: no K/V work
  bool zero;      // rows that see no key: O = 0, LSE = -inf
  Seq sq;
};

// The last sequence a thread looked up: consecutive items mostly belong to
// the same sequence, so its cu_seqlens entries are read from memory once.
struct SeqCache {
  int b = -1;
  Seq sq;
};

template <int kLayout>
__device__ __forceinline__ Item1 decode_item1(int it, bool grouped, int BH, int Hq, int num_qt,
                                              const Geo& geo, int causal, int* status,
                                              SeqCache& cache, uint32_t list) {
  constexpr bool kPacked = kLayout != kDenseLayout;
  Item1 w;
  if (kPacked && list != 0) {  // the CTA's item list (packed batches)
    const uint32_t e = ld_shared_u32(list + 4u * it);
    if (e == ~0u) {  // a position without work
      w.bh = 0;
      w.qt = 0;
      w.n = 0;
      w.zero = false;
      w.sq = Seq{0, 0, 0, 0};
      return w;
    }
    w.bh = static_cast<int>(e & 0xFFFFFu);
    w.qt = static_cast<int>(e >> 20);
  } else if (grouped) {
    w.bh = it / num_qt;
    w.qt = num_qt - 1 - it % num_qt;
  } else {
    w.qt = num_qt - 1 - it / BH;
    w.bh = it % BH;
  }
  if constexpr (kPacked) {
    const int b = w.bh / Hq;
    if (b != cache.b) {
      cache.sq = seq_of<kLayout>(geo, b, status);
      cache.b = b;
    }
    w.sq = cache.sq;
  } else {
    w.sq = seq_of<kLayout>(geo, w.bh / Hq, status);
  }
  const int kv = kv_tiles(w.sq, w.qt, causal);
  w.n = kv > 0 ? kv : 0;
  w.zero = kv == 0;
  return w;
}

// The epilogue of one d = 64 row: O / l as bf16 and the LSE.  Dense layout:
// the row goes into the item's Q buffer `stage` (its QK^T MMAs are
// complete), 16-byte chunk c at position c ^ (row % 8) of the 128-byte row
// (the O map's swizzle; rows past L are clipped by the TMA store, so every
// row is written) and each warp arrives on st_ready.  Other layouts store
// the row directly.
template <bool kTmaStore>
__device__ __forceinline__ void finish_row(const uint32_t (&r)[2][32], float l, float m_s,
                                           bool live, size_t orow, __nv_bfloat16* o, float* lse,
                                           uint8_t* stage, int row, int lane, uint64_t* st_ready) {
  constexpr int D = Cfg64::D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint4 q4[8];
#pragma unroll
  for (int v8 = 0; v8 < 8; ++v8) {
    const uint32_t* rv = &r[v8 >> 2][(v8 & 3) * 8];
    q4[v8].x = attn::pack_bf16x2(__uint_as_float(rv[0]) * inv, __uint_as_float(rv[1]) * inv);
    q4[v8].y = attn::pack_bf16x2(__uint_as_float(rv[2]) * inv, __uint_as_float(rv[3]) * inv);
    q4[v8].z = attn::pack_bf16x2(__uint_as_float(rv[4]) * inv, __uint_as_float(rv[5]) * inv);
    q4[v8].w = attn::pack_bf16x2(__uint_as_float(rv[6]) * inv, __uint_as_float(rv[7]) * inv);
  }
  if constexpr (kTmaStore) {
    uint8_t* buf = stage + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(buf + ((c ^ (row & 7)) << 4)) = q4[c];
    fence_proxy_async_smem();  // visible to the TMA store
    __syncwarp();
    if (lane == 0) mbar_arrive(st_ready);
  } else if (live) {
    uint4* orow_p = reinterpret_cast<uint4*>(o + orow * D);
#pragma unroll
    for (int v8 = 0; v8 < 8; ++v8) orow_p[v8] = q4[v8];
  }
  if (live && lse != nullptr) lse[orow] = l > 0.f ? (m_s + log2f(l)) * attn::kLn2 : -INFINITY;
}

template <int kLayout>
__global__ void __launch_bounds__(Cfg64::THREADS, 2)
    prefill_bf16_d64_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_o,
                            __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int BH, int Hq,
                            int Hkv, const Geo geo, int causal, float scale_log2, int q_div,
                            int* status) {
  using C = Cfg64;
  constexpr int D = C::D, NS = C::NS, NQ = C::NQ;
  constexpr bool kPacked = kLayout != kDenseLayout;
  constexpr bool kPaged = kLayout == kPagedLayout;
  constexpr bool kGather = kLayout == kGatherLayout;   // K/V rows gathered by warp 0
  constexpr bool kTmaStore = kLayout == kDenseLayout;  // O tile through the Q buffer
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;                 // [NQ]
  uint64_t* q_empty = q_full + NQ;         // [NQ] packed / paged: the item's last QK^T done
  uint64_t* k_full = q_empty + NQ;         // [NS] TMA
  uint64_t* v_full = k_full + NS;          // [NS] TMA
  uint64_t* k_done = v_full + NS;          // [NS] QK^T of the slot's tile done (K slot free)
  uint64_t* pv_done = k_done + NS;         // [NS] PV of the slot's tile done (V slot free)
  uint64_t* s_full = pv_done + NS;         // S(t) written
  uint64_t* s_read = s_full + 1;           // the softmax has read S(t) (one arrival per warp)
  uint64_t* p_ready = s_read + 1;          // the softmax wrote P(t) (one arrival per warp)
  uint64_t* o_done = p_ready + 1;
  uint64_t* o_free = o_done + 1;
  uint64_t* st_ready = o_free + 1;         // dense: the item's O rows are staged (per warp)
  uint64_t* drain = st_ready + 1;          // both issuers' MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert(8 * (6 * 2 + 7) + 8 <= 256, "d = 64 barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_qt = (geo.Lq + BM - 1) / BM;
  const int num_items = BH * num_qt;
  constexpr bool packed = kPacked;
  const int group = Hq / Hkv;
  // Dense short rows (or no mask): each CTA takes a contiguous run of items,
  // head by head, so a head's K/V is re-read from L2.  Long causal rows:
  // items heaviest first (Q tile index descending over all heads), dealt
  // round-robin, which balances the CTAs when the work per item varies.
  // Packed batches: the item list of build_item_list (units sorted by cost),
  // else the round-robin order.
  Schedule sched;
  sched.grouped = !kPacked && (!causal || num_qt <= 2 * kGroupedMaxPairs);
  if (sched.grouped) {
    sched.first = static_cast<int>(static_cast<long long>(num_items) * blockIdx.x / gridDim.x);
    sched.last = static_cast<int>(static_cast<long long>(num_items) * (blockIdx.x + 1) / gridDim.x);
    sched.step = 1;
  } else {
    sched.first = blockIdx.x;
    sched.last = num_items;
    sched.step = gridDim.x;
  }
  uint32_t list = 0;  // packed batches: the item list's shared address (set below), or 0
  SeqCache seq_cache;
  auto item_at = [&](int it) {
    return decode_item1<kLayout>(it, sched.grouped, BH, Hq, num_qt, geo, causal, status,
                                 seq_cache, list);
  };
  // The first item at or after `it` (in this CTA's order) with K/V work,
  // described in w (set only when the result is < sched.last).  Items
  // without any (no rows, or rows that see no key; packed layout only) just
  // make the softmax warps write their rows.  Each role decodes an item once.
  auto next_active = [&](int it, Item1& w) {
    for (; it < sched.last; it += sched.step) {
      w = item_at(it);
      if (!kPacked || w.n > 0) break;
    }
    return it;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_done[s], 1);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, C::kSoftmaxWarps);
    mbar_init(p_ready, C::kSoftmaxWarps);
    mbar_init(o_done, 1);
    mbar_init(o_free, C::kSoftmaxWarps);
    mbar_init(st_ready, C::kSoftmaxWarps);
    mbar_init(drain, 2);
    *abort_flag = (status != nullptr &&
                   *reinterpret_cast<volatile int*>(status) == ATTN_ERR_DEVICE_TIMEOUT) ? 2 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (*abort_flag == 2) return;
  // Packed batches: this CTA's item list (the K ring, not yet in use, is the
  // sort's scratch).
  if constexpr (kPacked) {
    static_assert(kSortScratchBytes <= NS * C::TILE_BYTES, "sort scratch fits the K ring");
    const int n = build_item_list<kLayout, 1>(reinterpret_cast<uint32_t*>(smem + C::OFF_LIST),
                                              smem + C::OFF_K, BH, Hq, num_qt, geo, causal,
                                              status);
    if (n >= 0) {
      list = sbase + C::OFF_LIST;
      sched.first = 0;
      sched.last = n;
      sched.step = 1;
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint64_t* bar, int parity) {
    return mbar_wait(bar, static_cast<uint32_t>(parity) & 1u, abort_flag, kWaitLimitNs);
  };
  constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
  constexpr uint64_t kTileStep = C::TILE_BYTES >> 4;

  if (warp < 4) {
    // 128 x 72 + 128 x 184 registers = the 256 x 128 the CTA launched with.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (warp == 0 && (kGather || lane == 0)) {
      // ---------------------------------------------------------- TMA producer
      // K runs one tile ahead of V: a K slot frees when its QK^T is done
      // (k_done), a V slot when its PV is done (pv_done).
      // Issue order K(0), K(1), V(0), K(2), V(1), ...
      // Gathered layouts: the whole warp copies the rows.
      if constexpr (!kGather) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      GatherRetire retire;  // gathered tiles are published one tile late
      auto pwait = [&](uint64_t* bar, int parity) -> bool {
        if constexpr (kGather) {
          if (__all_sync(FULL, mbar_test_wait(bar, static_cast<uint32_t>(parity) & 1u))) return true;
          retire.flush(lane);
          return __all_sync(FULL, wait(bar, parity));
        } else {
          return wait(bar, parity);
        }
      };
      struct Cur {
        int it, j, n, c1, c2;  // tile j of n; TMA coordinates (rows, heads) of tile 0
        PageCursor pages;      // paged cache: this item's pages, one tile ahead
        GatherCursor gath;     // gathered layouts: this item's block ids, one tile ahead
      };
      auto enter = [&](Cur& c, int it) {
        Item1 w;
        c.it = next_active(it, w);
        c.j = 0;
        c.n = 0;
        if (c.it < sched.last) {
          const int h = w.bh % Hq;
          c.n = w.n;
          c.c1 = packed ? h / group : 0;
          c.c2 = packed ? w.sq.k_off : (w.bh / Hq) * Hkv + h / group;
          if constexpr (kPaged) c.pages.begin(geo, w.bh / Hq, w.sq.lk);
          if constexpr (kGather) c.gath.begin(geo, w.bh / Hq, w.sq.lk, lane);
        }
      };
      auto next = [&](Cur& c) {
        if (++c.j < c.n) return;
        enter(c, c.it + sched.step);
      };
      Cur ck, cv;
      enter(ck, sched.first);
      enter(cv, sched.first);
      int tk = 0, tv = 0;  // K / V tiles issued
      bool ok = true;
      auto load_k = [&]() -> bool {
        const int st = tk % NS;
        if (tk >= NS && !pwait(&k_done[st], (tk / NS) + 1)) return false;
        if constexpr (kGather) {
          gather_tile<1>(smem + C::OFF_K + st * C::TILE_BYTES,
                         static_cast<const __nv_bfloat16*>(geo.k_raw), geo, ck.gath, ck.c1, Hkv,
                         lane, status);
          retire.committed(&k_full[st], lane);
          ck.gath.advance(lane);
        } else if constexpr (kPaged) {
          mbar_arrive_expect_tx(&k_full[st], C::TILE_BYTES);
          int pg[PageCursor::NP];
          ck.pages.take(pg, geo, status);
          tma_load_pages<1, C::TILE_BYTES>(smem + C::OFF_K + st * C::TILE_BYTES, &tm_k,
                                           &k_full[st], pg, ck.c1);
        } else {
          mbar_arrive_expect_tx(&k_full[st], C::TILE_BYTES);
          tma_load_3d(smem + C::OFF_K + st * C::TILE_BYTES, &tm_k, &k_full[st], 0,
                      packed ? ck.c1 : ck.j * BN, packed ? ck.c2 + ck.j * BN : ck.c2);
        }
        ++tk;
        next(ck);
        return true;
      };
      auto load_v = [&]() -> bool {
        const int st = tv % NS;
        if (tv >= NS && !pwait(&pv_done[st], (tv / NS) + 1)) return false;
        if constexpr (kGather) {
          gather_tile<1>(smem + C::OFF_V + st * C::TILE_BYTES,
                         static_cast<const __nv_bfloat16*>(geo.v_raw), geo, cv.gath, cv.c1, Hkv,
                         lane, status);
          retire.committed(&v_full[st], lane);
          cv.gath.advance(lane);
        } else if constexpr (kPaged) {
          mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
          int pg[PageCursor::NP];
          cv.pages.take(pg, geo, status);
          tma_load_pages<1, C::TILE_BYTES>(smem + C::OFF_V + st * C::TILE_BYTES, &tm_v,
                                           &v_full[st], pg, cv.c1);
        } else {
          mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
          tma_load_3d(smem + C::OFF_V + st * C::TILE_BYTES, &tm_v, &v_full[st], 0,
                      packed ? cv.c1 : cv.j * BN, packed ? cv.c2 + cv.j * BN : cv.c2);
        }
        ++tv;
        next(cv);
        return true;
      };
      if (ck.it < sched.last) ok = load_k();
      while (ok && cv.it < sched.last) {
        if (ck.it < sched.last) ok = load_k();
        if (ok) ok = load_v();
      }
      if (!ok && lane == 0) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: every issued copy has landed before the CTA may exit (k_full
      // and v_full count TMA bytes or cp.async arrivals; copies always complete).
      if constexpr (kGather) retire.flush(lane);
      int no_abort = 0;
      for (int u = tk > NS ? tk - NS : 0; u < tk; ++u)
        mbar_wait(&k_full[u % NS], (u / NS) & 1, &no_abort, kWaitLimitNs);
      for (int u = tv > NS ? tv - NS : 0; u < tv; ++u)
        mbar_wait(&v_full[u % NS], (u / NS) & 1, &no_abort, kWaitLimitNs);
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------- Q producer
      // Q tiles go out as soon as their buffer frees, about an item ahead of
      // the K/V stream.  Dense layout: the buffer of the item NQ back holds
      // that item's staged O tile, which is stored first.
      prefetch_tmap(&tm_q);
      if constexpr (kTmaStore) prefetch_tmap(&tm_o);
      int nq = 0;
      bool ok = true;
      Item1 w;
      int back_bh[NQ] = {}, back_qt[NQ] = {};  // dense: the item whose O a buffer holds
      auto store_o = [&](int i) -> bool {  // O tile of the nq-th item i (dense)
        const int qs = i % NQ;
        if (!wait(st_ready, i)) return false;
        tma_store_3d(&tm_o, smem + C::OFF_Q + qs * C::TILE_BYTES, 0, back_qt[qs] * BM, back_bh[qs]);
        bulk_commit_group();
        bulk_wait_read_all();
        return true;
      };
      for (int it = next_active(sched.first, w); ok && it < sched.last;
           it = next_active(it + sched.step, w)) {
        const int qs = nq % NQ;
        if (nq >= NQ) {
          if constexpr (kTmaStore) ok = store_o(nq - NQ);
          else ok = wait(&q_empty[qs], (nq / NQ) - 1);
          if (!ok) break;
        }
        if constexpr (kTmaStore) {
          back_bh[qs] = w.bh;
          back_qt[qs] = w.qt;
        }
        mbar_arrive_expect_tx(&q_full[qs], C::TILE_BYTES);
        tma_load_3d(smem + C::OFF_Q + qs * C::TILE_BYTES, &tm_q, &q_full[qs], 0,
                    packed ? w.bh % Hq : w.qt * BM,
                    packed ? w.sq.q_off + w.qt * BM : w.bh / q_div);
        ++nq;
      }
      if constexpr (kTmaStore) {
        for (int i = nq > NQ ? nq - NQ : 0; ok && i < nq; ++i) ok = store_o(i);
        bulk_wait_all();  // every O store has completed before the CTA exits
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      int no_abort = 0;
      for (int i = nq > NQ ? nq - NQ : 0; i < nq; ++i)
        mbar_wait(&q_full[i % NQ], (i / NQ) & 1, &no_abort, kWaitLimitNs);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- QK issuer
      // Descriptors are built once; a K step or a ring slot only moves the
      // start-address field (address >> 4), which never carries (shared
      // addresses stay below 256 KB).
      const uint64_t q_desc0 = smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sbase + C::OFF_K, 16, 1024);
      int nq = 0;  // items started
      int t = 0;   // global step
      bool ok = true;
      Item1 w;
      for (int it = next_active(sched.first, w); ok && it < sched.last;
           it = next_active(it + sched.step, w)) {
        const uint64_t qd = q_desc0 + static_cast<uint64_t>(nq % NQ) * kTileStep;
        if (!wait(&q_full[nq % NQ], nq / NQ)) { ok = false; break; }
        for (int j = 0; j < w.n; ++j, ++t) {
          if (!wait(&k_full[t % NS], t / NS) || (t > 0 && !wait(s_read, t - 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = k_desc0 + static_cast<uint64_t>(t % NS) * kTileStep;
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_bf16_ss(tmem, qd + k * 2, kd + k * 2, idesc_qk, k > 0 ? 1u : 0u);
          mma_commit(s_full);
          mma_commit(&k_done[t % NS]);
          if constexpr (!kTmaStore)
            if (j + 1 == w.n) mma_commit(&q_empty[nq % NQ]);  // that Q buffer may be refilled
        }
        ++nq;
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      mma_commit(drain);
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------------- PV issuer
      const uint64_t v_desc0 = smem_desc_sw128(sbase + C::OFF_V, C::TILE_BYTES, 1024);
      int nitem = 0;
      int t = 0;
      bool ok = true;
      Item1 w;
      for (int it = next_active(sched.first, w); ok && it < sched.last;
           it = next_active(it + sched.step, w)) {
        for (int j = 0; j < w.n; ++j, ++t) {
          if (!wait(&v_full[t % NS], t / NS) || !wait(p_ready, t) ||
              (j == 0 && nitem > 0 && !wait(o_free, nitem - 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t vd = v_desc0 + static_cast<uint64_t>(t % NS) * kTileStep;
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_bf16_ts(tmem + C::O_COL, tmem + C::P_COL + k * 8, vd + static_cast<uint64_t>(k) * 128,
                        idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(&pv_done[t % NS]);
        }
        ++nitem;
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      mma_commit(drain);
    }
    if (warp == 1 || warp == 2) {
      // Drain: all MMAs of both issuers are complete before teardown.
      int no_abort = 0;
      if (lane == 0) mbar_wait(drain, 0, &no_abort, kWaitLimitNs);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory");
    // ------------------------------------------------------------ softmax warps
    // An item's epilogue (O / l and the LSE) is deferred into the next
    // item's first step: that step computes its P while the previous item's
    // last PV completes (pv_done of the step before), hands P to the tensor
    // core, then reads the finished O, releases it (o_free: the new item's
    // first PV waits for it) and normalises and stores the old rows, so the
    // wait for the last PV and the stores overlap the new item's MMAs.
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;  // row within the Q tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off;
    const uint32_t p_addr = tmem + lane_off + C::P_COL;
    const uint32_t o_addr = tmem + lane_off + C::O_COL;
    int t = 0;       // global step of the current item's K/V tile 0
    int nitem = 0;
    bool ok = true;
    // The item whose O is still in TMEM (its epilogue pending).
    bool pend_on = false, pend_live = false;
    float pend_m = 0.f, pend_l = 0.f;
    size_t pend_orow = 0;
    int pend_slot = 0;
    for (int it = sched.first; ok && it < sched.last; it += sched.step) {
      const Item1 w = item_at(it);
      const int n = w.n;
      const int grow = w.qt * BM + row;
      const int h = w.bh % Hq;
      // Output row: dense [heads, rows], packed [rows, heads].
      const size_t orow_index = packed ? static_cast<size_t>(w.sq.q_off + grow) * Hq + h
                                       : static_cast<size_t>(w.bh) * geo.Lq + grow;
      if (n == 0) {
        if constexpr (kPacked) {
          if (w.zero && grow < w.sq.lq) {  // rows that see no key
            uint4* op = reinterpret_cast<uint4*>(o + orow_index * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr) lse[orow_index] = -INFINITY;
          }
        }
        continue;
      }
      float m_s = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int tt = t + j;
        ok = __all_sync(FULL, wait(s_full, tt));
        if (!ok) break;
        tc_fence_after();
        // S and, from the load itself, the maximum of each 32-column chunk.
        float sr[4][32], cmax[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(s_addr + c * 32, sr[c], cmax[c]);
        tmem_ld_wait();
        float* s = &sr[0][0];
        // S is in registers: S(tt + 1) may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_read);

        const bool need_mask = kPacked ? tile_needs_mask(w.sq, w.qt, j, causal)
                                       : (j == n - 1) && (causal || (geo.Lk % BN) != 0);
        if (need_mask) {
          // Element mask by compare-and-select (straight-line, no branches).
          const int kv = row_kmax(w.sq, grow, causal) - j * BN;  // last visible column
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = mask_col(s[c], c, kv);
        }
        // Row max: an unmasked tile takes it from the load; a masked one
        // reduces the masked scores as 8 independent chains.
        float mt = fmaxf(fmaxf(cmax[0], cmax[1]), fmaxf(cmax[2], cmax[3]));
        if (need_mask) {
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int c = 16; c < BN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
          mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        }
        const float mt_s = mt * scale_log2;
        float alpha = 1.f;
        if (mt_s > m_s + kRescaleThreshold) {
          alpha = ex2(m_s - mt_s);  // 0 on the first tile (m_s = -inf)
          m_s = mt_s;
        }
        // A row that sees no key yet (every score -inf, possible when causal
        // is aligned bottom-right with lq > lk) keeps m = -inf: subtract 0
        // instead so that its p are exp(-inf) = 0, not NaN.
        const float m_sub = kPacked && m_s == -INFINITY ? 0.f : m_s;
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_sub, -m_sub);
        float2 rs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.f, 0.f);
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          float2 e = ffma2(make_float2(s[c], s[c + 1]), sc2, nm2);
          e.x = ex2(e.x);
          e.y = ex2(e.y);
          rs[(c >> 1) & 3] = fadd2(rs[(c >> 1) & 3], e);
          pk[c >> 6][(c >> 1) & 31] = attn::pack_bf16x2(e.x, e.y);
        }
        const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
        const float2 r2 = fadd2(r01, r23);
        l = l * alpha + (r2.x + r2.y);
        // PV of the previous step (at j = 0: the previous item's last PV)
        // has read P and updated O.
        if (tt > 0) {
          ok = __all_sync(FULL, wait(&pv_done[(tt - 1) % NS], (tt - 1) / NS));
          if (!ok) break;
          tc_fence_after();
        }
        if (j > 0 && __any_sync(FULL, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o32[32];
            tmem_ld32(o_addr + c * 32, o32);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
            tmem_st32(o_addr + c * 32, o32);
          }
        }
        tmem_st32(p_addr, pk[0]);
        tmem_st32(p_addr + 32, pk[1]);
        if constexpr (kPaged) {
          if (has_v_tail(w.sq.lk, j, geo.block_shift)) {
            ok = __all_sync(FULL, wait(&v_full[tt % NS], tt / NS));
            clear_v_tail<1, C::TILE_BYTES>(smem + C::OFF_V + (tt % NS) * C::TILE_BYTES, row,
                                           w.sq.lk, j, geo.block_shift);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
        if (j == 0 && pend_on) {
          // The previous item's last PV completed before this step's wait on
          // pv_done: read its O, release it (this item's first PV may then
          // overwrite it) and finish its rows.
          uint32_t r[2][32];
          tmem_ld32(o_addr, r[0]);
          tmem_ld32(o_addr + 32, r[1]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);
          finish_row<kTmaStore>(r, pend_l, pend_m, pend_live, pend_orow, o, lse,
                                smem + C::OFF_Q + pend_slot * C::TILE_BYTES, row, lane,
                                st_ready);
          pend_on = false;
        }
      }
      if (!ok) break;
      pend_on = true;
      pend_m = m_s;
      pend_l = l;
      pend_orow = orow_index;
      pend_live = grow < w.sq.lq;
      pend_slot = nitem % NQ;
      ++nitem;
      t += n;
    }
    // The last item: its final PV, then its epilogue.
    if (ok && pend_on) {
      ok = __all_sync(FULL, wait(&pv_done[(t - 1) % NS], (t - 1) / NS));
      if (ok) {
        tc_fence_after();
        uint32_t r[2][32];
        tmem_ld32(o_addr, r[0]);
        tmem_ld32(o_addr + 32, r[1]);
        tmem_ld_wait();
        finish_row<kTmaStore>(r, pend_l, pend_m, pend_live, pend_orow, o, lse,
                              smem + C::OFF_Q + pend_slot * C::TILE_BYTES, row, lane, st_ready);
      }
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Packed rows: [total rows, H heads] x d bf16 viewed as {d, H, total}; box
// {64, 1, 128} (128 rows of one head, the same shared-memory tile as the
// dense box).  Rows past total read as zeros.
bool make_map_packed(CUtensorMap* m, const void* base, int D, int H, int total) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(total)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Paged cache [num_pages, block slots, Hkv, d] bf16 viewed as {d, Hkv,
// block, num_pages}; box {64, 1, block, 1}: one block of one KV head, 64
// columns, in the tile's 128-byte swizzle.  The block coordinate num_pages
// (past the tensor) reads as zeros.
bool make_map_pages(CUtensorMap* m, const void* base, int D, int Hkv, int block, int num_pages) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(Hkv) * D * 2,
                                 static_cast<cuuint64_t>(block) * Hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(block), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH heads, L rows] x d bf16 viewed as a 3-D tensor {d, L, BH}; box
// {64, 128, 1} with 128-byte swizzle.  Rows past L read as zeros.
bool make_map(CUtensorMap* m, const void* base, int D, int L, int BH) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(L) * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kLayout>
attn_status_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                     int Hkv, const Geo& geo, int causal, float scale, int q_div,
                     cudaStream_t stream) {
  // d = 64 runs the two-CTAs-per-SM kernel on single Q tiles, d = 128 the
  // Q-tile-pair ping-pong kernel.
  constexpr bool kD64 = D == 64;
  constexpr int smem_bytes = (kD64 ? Cfg64::SMEM_BYTES : Cfg<D>::SMEM_BYTES) +
                             (!kD64 || kLayout != kDenseLayout ? kListBytes : 0);
  // Opt-in limit of one CTA (227 KB); at d = 64 two CTAs (each with 1 KB the
  // hardware reserves) share the SM's 228 KB.
  static_assert(Cfg<128>::SMEM_BYTES + kListBytes <= 227 * 1024, "d = 128 shared memory");
  static_assert(2 * (Cfg64::SMEM_BYTES + kListBytes + 1024) <= 228 * 1024, "d = 64 shared memory");
  static bool attr_set[64] = {};  // per device: kernel attributes are per device
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return ATTN_ERR_CUDA;
  if (!attr_set[dev]) {
    const void* fn;
    if constexpr (kD64)
      fn = reinterpret_cast<const void*>(prefill_bf16_d64_kernel<kLayout>);
    else
      fn = reinterpret_cast<const void*>(prefill_bf16_kernel<D, kLayout>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
            cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap mq, mk, mv, mo;
  if (q_div < 1 || (B * Hq) % q_div != 0) return ATTN_ERR_INVALID_ARG;
  bool maps_ok;
  if constexpr (kLayout == kPagedLayout)  // 16-token pages
    maps_ok = make_map_packed(&mq, q, D, Hq, geo.total_q) &&
              make_map_pages(&mk, k, D, Hkv, kPage, geo.num_pages) &&
              make_map_pages(&mv, v, D, Hkv, kPage, geo.num_pages);
  else if constexpr (kLayout == kGatherLayout) {  // K/V rows gathered from plain pointers
    maps_ok = make_map_packed(&mq, q, D, Hq, geo.total_q);
    mk = mq;
    mv = mq;
  }
  else if constexpr (kLayout == kPackedLayout)
    maps_ok = make_map_packed(&mq, q, D, Hq, geo.total_q) &&
              make_map_packed(&mk, k, D, Hkv, geo.total_k) &&
              make_map_packed(&mv, v, D, Hkv, geo.total_k);
  else
    maps_ok = make_map(&mq, q, D, geo.Lq, B * Hq / q_div) && make_map(&mk, k, D, geo.Lk, B * Hkv) &&
              make_map(&mv, v, D, geo.Lk, B * Hkv);
  // The d = 64 dense kernel stores O tiles by TMA (the other layouts ignore mo).
  if (maps_ok && kD64 && kLayout == kDenseLayout) maps_ok = make_map(&mo, o, D, geo.Lq, B * Hq);
  else mo = mq;
  if (!maps_ok) return ATTN_ERR_CUDA;
  const int num_qt = (geo.Lq + BM - 1) / BM;
  const long long items = static_cast<long long>(B) * Hq * (kD64 ? num_qt : (num_qt + 1) / 2);
  if (items > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  const int sms = attn_host::num_sms();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const long long slots = static_cast<long long>(sms) * (kD64 ? 2 : 1);
  const int grid = static_cast<int>(items < slots ? items : slots);
  const float scale_log2 = scale * attn::kLog2e;
  if constexpr (kD64) {
    prefill_bf16_d64_kernel<kLayout><<<grid, Cfg64::THREADS, smem_bytes, stream>>>(
        mq, mk, mv, mo, static_cast<__nv_bfloat16*>(o), lse, B * Hq, Hq, Hkv, geo, causal,
        scale_log2, q_div, attn_host::device_status_ptr());
  } else {
    prefill_bf16_kernel<D, kLayout><<<grid, NUM_THREADS, smem_bytes, stream>>>(
        mq, mk, mv, static_cast<__nv_bfloat16*>(o), lse, B * Hq, Hq, Hkv, geo, causal,
        scale_log2, q_div, attn_host::device_status_ptr());
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

attn_status_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                  float scale, int q_div, cudaStream_t stream) {
  const Geo geo{nullptr, nullptr, Lq, Lk, 0, 0, nullptr, nullptr, 0, 0, nullptr, 0, 4, nullptr, nullptr};
  if (d == 64) return launch<64, kDenseLayout>(q, k, v, o, lse, B, Hq, Hkv, geo, causal, scale, q_div, stream);
  if (d == 128)
    return launch<128, kDenseLayout>(q, k, v, o, lse, B, Hq, Hkv, geo, causal, scale, q_div, stream);
  return ATTN_ERR_UNSUPPORTED;
}

attn_status_t launch_prefill_bf16_varlen(const void* q, const void* k, const void* v, void* o,
                                         float* lse, const int* cu_q, const int* cu_k, int B,
                                         int max_q, int max_k, int total_q, int total_k, int Hq,
                                         int Hkv, int d, int causal, float scale,
                                         cudaStream_t stream) {
  const Geo geo{cu_q, cu_k, max_q, max_k, total_q, total_k, nullptr, nullptr, 0, 0,
                nullptr, 0, 4, nullptr, nullptr};
  if (d == 64)
    return launch<64, kPackedLayout>(q, k, v, o, lse, B, Hq, Hkv, geo, causal, scale, 1, stream);
  if (d == 128)
    return launch<128, kPackedLayout>(q, k, v, o, lse, B, Hq, Hkv, geo, causal, scale, 1, stream);
  return ATTN_ERR_UNSUPPORTED;
}

attn_status_t launch_prefill_bf16_paged(const void* q, const void* k_pages, const void* v_pages,
                                        const int* block_table, const int* kv_indptr, int nnz,
                                        int block_size, const int* cu_q, const int* seq_lens_k,
                                        void* o, float* lse, int B, int max_q, int max_k,
                                        int total_q, int Hq, int Hkv, int d, int max_pages,
                                        int num_pages, int causal, float scale,
                                        cudaStream_t stream) {
  int shift = 0;
  while ((1 << shift) < block_size) ++shift;
  if ((1 << shift) != block_size || shift > 7) return ATTN_ERR_UNSUPPORTED;
  // 16-token pages: one TMA copy per page; other block sizes: row gathers.
  const bool tma = block_size == 16;
  const Geo geo{cu_q, nullptr, max_q, max_k, total_q, 0, seq_lens_k, block_table, max_pages,
                num_pages, kv_indptr, nnz, shift, k_pages, v_pages};
  if (d == 64)
    return tma ? launch<64, kPagedLayout>(q, k_pages, v_pages, o, lse, B, Hq, Hkv, geo, causal,
                                          scale, 1, stream)
               : launch<64, kGatherLayout>(q, k_pages, v_pages, o, lse, B, Hq, Hkv, geo, causal,
                                           scale, 1, stream);
  if (d == 128)
    return tma ? launch<128, kPagedLayout>(q, k_pages, v_pages, o, lse, B, Hq, Hkv, geo, causal,
                                           scale, 1, stream)
               : launch<128, kGatherLayout>(q, k_pages, v_pages, o, lse, B, Hq, Hkv, geo, causal,
                                            scale, 1, stream);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn_host
