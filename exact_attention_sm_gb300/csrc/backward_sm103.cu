// Attention backward pass, bf16 in / bf16 gradients, fp32 accumulation.
//
// "10.3 FlashAttention" (LLM Internals), "backward and recomputation", and
// the tiling blog's section 07: the forward keeps only O and the per-row LSE;
// the backward reads Q_i, K_j, V_j tile by tile again, rebuilds
// S_ij = scale Q_i K_j^T and P_ij = exp(S_ij - LSE_i) on chip, and
// accumulates dQ, dK, dV, so no L x L matrix reaches HBM.  With dO given:
//     dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i * O_i),
//     dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels, no atomics (every gradient element is written by exactly
// one CTA, sums run in a fixed order, so results are bitwise reproducible):
//   bwd_rowdot_kernel   D = rowsum(dO * O) per query row (fp32), written as
//                       -D next to -LSE log2e, both padded to whole Q tiles.
//   bwd_dkdv_kernel     work item (request, KV head, key tile j): K_j, V_j
//                       stay in shared memory while the Q tiles of every
//                       query head of the group stream past; per Q tile four
//                       tcgen05 MMAs with the 128 keys as the M dimension:
//                         S^T  = K_j Q_i^T           (TMEM, fp32)
//                         dP^T = V_j dO_i^T          (TMEM, fp32)
//                         dV  += P^T dO_i            (P^T bf16 from TMEM)
//                         dK  += dS^T Q_i            (dS^T bf16 from TMEM)
//                       so neither P nor dS is ever transposed.
//   bwd_dq_kernel       work item (request, query head, Q tile i): Q_i and
//                       dO_i stay while the K/V tiles stream past; per K/V
//                       tile three MMAs with the queries as M:
//                         S = Q_i K_j^T,  dP = dO_i V_j^T,  dQ += dS K_j.
// Recomputing S and dP in both kernels costs two extra GEMMs per tile pair
// against a single kernel that adds dQ with atomics; in exchange the result
// does not depend on the order in which CTAs finish.
//
// Both MMA kernels run one persistent CTA per SM (384 threads) that takes
// work items from a counter, heaviest first, and loads the next item's
// tiles while it works on the current one.  Roles: warps 0 and 2 (lane 0)
// load tiles with TMA, warp 1 lane 0 issues the MMAs, warps 4-11 do the
// elementwise work in two groups of four, one per half of the tile pair
// (the 64-query halves of S^T in bwd_dkdv, the 64-key halves of S in
// bwd_dq); in a group one thread owns one TMEM lane (a key row in bwd_dkdv,
// a query row in bwd_dq).  S and dP are whole 128 x 128 products (N = 128
// per instruction), and every hand-off between the issuer and the groups is
// one barrier, so the single issuing thread stalls the tensor core as
// little as possible; S of the next tile pair goes into a second TMEM
// buffer while the groups work on this one (bwd_dq, and bwd_dkdv at
// d = 64).  Every wait is bounded (ATTN_ERR_DEVICE_TIMEOUT, CTA abort,
// drain, TMEM freed), as in the forward kernels.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace {

using namespace sm103;

constexpr int T = 128;               // rows of a Q or K/V tile (MMA M and N)
constexpr int THREADS = 384;         // 12 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 50000000ull;
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

template <int D>
struct BwdCfg {
  static constexpr int KB = D / 64;             // 64-column, 128-byte swizzle blocks per row
  static constexpr int BLOCK_BYTES = T * 128;   // one 128-row block
  static constexpr int TILE_BYTES = T * D * 2;  // one bf16 tile
  // TMEM columns: S (or S^T) 0..127, dP (or dP^T) 128..255, then the fp32
  // accumulators, and a second S buffer at 384..511 where the accumulators
  // leave room.  P^T / dS^T / dS (bf16 pairs) of a 64-column half overwrite
  // the first 32 columns of that half.
  static constexpr uint32_t S_COL = 0, DP_COL = 128, ACC0_COL = 256, ACC1_COL = 256 + D,
                            S1_COL = 384;
};

// Instruction descriptor: kind::f16, bf16 A/B, fp32 D, M = 128.
__host__ __device__ constexpr uint32_t idesc(int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(T >> 4) << 24);
}

// The elementwise groups split a tile pair into two halves of H = 64 rows
// (queries in bwd_dkdv, keys in bwd_dq).  Half h of a K-major or MN-major
// tile starts 64 rows (8 KB, eight whole swizzle atoms) into each column
// block.
constexpr int H = T / 2;
constexpr uint64_t kHalfStep = (H * 128) >> 4;  // descriptor start-address step of a half

// D(tmem, 128 x 128 fp32) = A B^T for the 128-row K-major tiles A and B:
// one MMA per 16 columns of D (N = 128: a wider product per instruction
// keeps the tensor core busier than two N = 64 halves).
template <int D>
__device__ __forceinline__ void mma_kmajor_full(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint64_t kBlk = BwdCfg<D>::BLOCK_BYTES >> 4;
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint64_t off = (k >> 2) * kBlk + (k & 3) * 2;
    mma_bf16_ss(d_tmem, a_desc + off, b_desc + off, idesc(T, false), k > 0 ? 1u : 0u);
  }
}

// D(tmem) (+)= A(tmem, 128 rows x H bf16 in H / 2 columns) B, B half of an
// MN-major smem tile ([H rows = the K dimension][D] bf16): one MMA per 16
// rows of B.
template <int D>
__device__ __forceinline__ void mma_tmem_a_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                bool accumulate) {
#pragma unroll
  for (int k = 0; k < H / 16; ++k)
    mma_bf16_ts(d_tmem, a_tmem + k * 8, b_desc + static_cast<uint64_t>(k) * 128, idesc(D, true),
                (accumulate || k > 0) ? 1u : 0u);
}

// D = rowsum(dO * O) for every query row: one warp per row, fp32 sums of the
// bf16 products in a fixed lane order.
// D = rowsum(dO * O) for the rows of the padded [B Hq][nq 128] layout,
// written as nd = -D next to nl = -LSE log2e (-inf where the row does not
// exist or sees no key, so that P = 0; nd = 0 there).  A row is read by D / 8
// lanes with one 16-byte load of O and one of dO each, so a warp covers
// 32 / (D / 8) rows per pass and the loads are whole 128-byte lines; the
// grid strides over the rows.  The sum runs in a fixed lane order.  Block 0
// also zeroes the two work counters of the MMA kernels that follow on the
// same stream.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
                      const float* __restrict__ lse, float* __restrict__ nl,
                      float* __restrict__ nd, long long heads, int Lq, int Lq_pad, int* work) {
  constexpr int G = D / 8;     // lanes per row
  constexpr int RPW = 32 / G;  // rows per warp and pass
  if (blockIdx.x == 0 && threadIdx.x < 2) work[threadIdx.x] = 0;
  const int lane = threadIdx.x & 31;
  const int sub = lane / G, gl = lane % G;
  const long long total = heads * Lq_pad;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp_id * RPW; base < total; base += nwarps * RPW) {
    const long long rp = base + sub;
    float acc = 0.f;
    bool live = false;
    long long r = 0;
    if (rp < total) {
      const long long h = rp / Lq_pad;
      const int row = static_cast<int>(rp - h * Lq_pad);
      live = row < Lq;
      r = h * Lq + row;
      if (live) {
        const uint4 a = attn::ld_stream_v4(o + r * D + gl * 8);
        const uint4 g = attn::ld_stream_v4(d_o + r * D + gl * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc = fmaf(attn::bf16_lo(av[c]), attn::bf16_lo(gv[c]), acc);
          acc = fmaf(attn::bf16_hi(av[c]), attn::bf16_hi(gv[c]), acc);
        }
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(FULL, acc, off);
    if (gl == 0 && rp < total) {
      if (!live) {
        nl[rp] = -INFINITY;
        nd[rp] = 0.f;
      } else {
        const float x = lse[r];
        nl[rp] = x == -INFINITY ? -INFINITY : -x * attn::kLog2e;
        nd[rp] = -acc;
      }
    }
  }
}

}  // namespace
namespace {

// Stage counts and shared-memory layout of both MMA kernels.  Each kernel
// holds two operand tiles for a whole work item (K, V in bwd_dkdv; Q, dO in
// bwd_dq) in NF slots, so the next item's pair loads during this one at
// d = 64, and streams the other two (Q, dO; K, V) through an NS-stage ring
// deep enough to cover the load latency.  Then the ring's per-query values
// (-LSE log2e and -D of the Q tile, bwd_dkdv), the item ring, the barriers.
// Two producer threads load the tiles, one the first and one the second
// tile of every pair: the copies one thread issues complete one after
// another (about 24 bytes per clock from L2), so one thread alone would not
// keep up with the tensor core at d = 64.  Producer 0 arms each pair's
// barrier for both tiles; producer 1's copy only completes bytes on it.
// At d = 64 the item's gradient tiles (STG of them: dV and dK, or dQ) are
// staged in shared memory in the 128-byte swizzle and written by one TMA
// store each, instead of one 128-byte row per thread; bwd_dkdv gives up a
// ring stage for its two staging tiles.
template <int D, int STG>
struct BwdSmem {
  using C = BwdCfg<D>;
  static constexpr int NF = D == 64 ? 2 : 1;
  static constexpr int NS = D == 64 ? (STG == 2 ? 3 : 4) : 2;
  static constexpr int TILES = 2 * NF + 2 * NS;
  static constexpr int OFF_STG = TILES * C::TILE_BYTES;  // STG staging tiles
  static constexpr int OFF_VEC = OFF_STG + STG * C::TILE_BYTES;  // [NS][-LSE log2e | -D][128] fp32
  static constexpr int OFF_BAR = OFF_VEC + NS * 2 * T * 4;
  static constexpr int BYTES = OFF_BAR + 512 + 1024;  // barriers, item ring, alignment slack
};
// Staging tiles of each kernel: only at d = 64 (one tile holds a 64-column row block).
template <int D> constexpr int kDkdvStg = D == 64 ? 2 : 0;
template <int D> constexpr int kDqStg = D == 64 ? 1 : 0;
static_assert(BwdSmem<64, 2>::BYTES <= 227 * 1024 && BwdSmem<64, 1>::BYTES <= 227 * 1024 &&
                  BwdSmem<128, 0>::BYTES <= 227 * 1024,
              "shared memory of one CTA");

constexpr int kItemRing = 8;  // published work items in flight

struct BwdBars {
  uint64_t* hold_full;    // [NF] the item's held pair has landed
  uint64_t* hold_empty;   // [NF] the item's products are done with it
  uint64_t* ring_full;    // [NS] a streamed pair has landed
  uint64_t* ring_empty;   // [NS] the products are done with it
  uint64_t* s_full;       // [2 S buffers]: S (S^T) is in TMEM
  uint64_t* dp_full;      // [2 dP buffers]: dP (dP^T) is in TMEM
  uint64_t* p_ready;      // [2 iteration parities]: P^T written (bwd_dkdv); [0]: S read (bwd_dq)
  uint64_t* ds_ready;     // [2 iteration parities]: dS (dS^T) written
  uint64_t* acc_done;     // the item's accumulators are final
  uint64_t* drain;
  uint64_t* st_ready;     // [2 groups] the group's rows are in its staging tile
  uint64_t* st_free;      // [2 groups] the group's last tile store has read its staging tile
  uint64_t* item_full;    // [kItemRing] item id published
  int* items;             // [kItemRing]
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ BwdBars carve_bars(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base);
  BwdBars r;
  r.hold_full = b;
  r.hold_empty = b + 2;
  r.ring_full = b + 4;
  r.ring_empty = b + 8;
  r.s_full = b + 12;
  r.dp_full = b + 14;
  r.p_ready = b + 16;
  r.ds_ready = b + 18;
  r.acc_done = b + 20;
  r.drain = b + 21;
  r.st_ready = b + 22;
  r.st_free = b + 24;
  r.item_full = b + 26;
  r.items = reinterpret_cast<int*>(b + 26 + kItemRing);
  r.tmem_slot = reinterpret_cast<uint32_t*>(r.items + kItemRing);
  r.abort_flag = reinterpret_cast<volatile int*>(r.tmem_slot + 1);
  return r;
}
static_assert((26 + kItemRing) * 8 + kItemRing * 4 + 8 <= 512, "barrier area");
static_assert(BwdSmem<64, 1>::NF <= 2 && BwdSmem<64, 1>::NS <= 4 && BwdSmem<128, 0>::NF <= 2 &&
                  BwdSmem<128, 0>::NS <= 4,
              "barrier counts");

// Barrier set-up, the pending-timeout check and the TMEM allocation shared
// by both kernels.  Returns false when the CTA must skip its work.
template <int NF, int NS>
__device__ __forceinline__ bool bwd_prologue(const BwdBars& bb, int* status) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < NF; ++s) {
      mbar_init(&bb.hold_full[s], 1);
      mbar_init(&bb.hold_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bb.ring_full[s], 1);
      mbar_init(&bb.ring_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb.s_full[s], 1);
      mbar_init(&bb.dp_full[s], 1);
      mbar_init(&bb.p_ready[s], 8);   // one arrival per elementwise warp
      mbar_init(&bb.ds_ready[s], 8);
      mbar_init(&bb.st_ready[s], 4);  // one arrival per warp of the group
      mbar_init(&bb.st_free[s], 1);
    }
    for (int s = 0; s < kItemRing; ++s) mbar_init(&bb.item_full[s], 1);
    mbar_init(bb.acc_done, 1);
    mbar_init(bb.drain, 1);
    *bb.abort_flag = (status != nullptr &&
                      *reinterpret_cast<volatile int*>(status) == ATTN_ERR_DEVICE_TIMEOUT) ? 2 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (*bb.abort_flag == 2) return false;
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(bb.tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return true;
}

__device__ __forceinline__ void bwd_epilogue(const BwdBars& bb) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*bb.tmem_slot, TMEM_COLS);
  }
}

// Writes NC x 32 fp32 columns of this thread's TMEM lane (from `taddr`)
// times `mul` as bf16 to global memory (16-byte stores).
template <int NC>
__device__ __forceinline__ void store_cols_bf16(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                                bool live) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_ld_wait();
    if (live) {
#pragma unroll
      for (int v8 = 0; v8 < 4; ++v8) {
        uint4 w;
        w.x = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 0]) * mul, __uint_as_float(r[v8 * 8 + 1]) * mul);
        w.y = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 2]) * mul, __uint_as_float(r[v8 * 8 + 3]) * mul);
        w.z = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 4]) * mul, __uint_as_float(r[v8 * 8 + 5]) * mul);
        w.w = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 6]) * mul, __uint_as_float(r[v8 * 8 + 7]) * mul);
        *reinterpret_cast<uint4*>(dst + c * 32 + v8 * 8) = w;
      }
    }
  }
}

// One 64-column fp32 TMEM row (from `taddr`) times `mul` as bf16 into row r
// of a staging tile in the 128-byte swizzle the TMA store expects (16-byte
// chunk q of row r at position q ^ (r % 8)).
__device__ __forceinline__ void stage_row64_bf16(uint32_t taddr, float mul, uint8_t* tile, int r) {
  uint32_t v[2][32];
  tmem_ld32(taddr, v[0]);
  tmem_ld32(taddr + 32, v[1]);
  tmem_ld_wait();
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t* x = &v[q >> 2][(q & 3) * 8];
    uint4 w;
    w.x = attn::pack_bf16x2(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul);
    w.y = attn::pack_bf16x2(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul);
    w.z = attn::pack_bf16x2(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul);
    w.w = attn::pack_bf16x2(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul);
    *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) << 4)) = w;
  }
}

// -inf where column c lies past kv (c > kv) / before lo (c < lo), else x:
// a compare and a select, no branch.
__device__ __forceinline__ float neg_inf_if_gt(float x, int c, int kv) {
  float r;
  asm("{\n\t.reg .pred q;\n\tsetp.gt.s32 q, %2, %3;\n\tselp.f32 %0, 0fFF800000, %1, q;\n\t}"
      : "=f"(r)
      : "f"(x), "r"(c), "r"(kv));
  return r;
}
__device__ __forceinline__ float neg_inf_if_lt(float x, int c, int lo) {
  float r;
  asm("{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %2, %3;\n\tselp.f32 %0, 0fFF800000, %1, q;\n\t}"
      : "=f"(r)
      : "f"(x), "r"(c), "r"(lo));
  return r;
}

// Work items of both kernels, in the order the CTAs claim them: the heads in
// groups of kHeadGroup; within a group tile index t = 0 (the heaviest under
// the causal rule) of every head first, then t = 1, ...  The items running
// at the same time then re-read the same few heads' streamed tiles (Q and dO
// in bwd_dkdv, K and V in bwd_dq) from L2, and the lightest come last.
constexpr int kHeadGroup = 32;
__device__ __forceinline__ void item_order(int x, int nt, int heads, int& t, int& head) {
  const int per_group = kHeadGroup * nt;
  const int g0 = (x / per_group) * kHeadGroup;
  const int rem = x % per_group;
  const int gsz = min(kHeadGroup, heads - g0);
  t = rem / gsz;
  head = g0 + rem % gsz;
}

// Persistent CTAs take items from a counter in the workspace (zeroed by
// bwd_rowdot_kernel, which runs first on the same stream): the producer
// claims one item ahead and publishes each id in the item ring (-1: none
// left); the issuer and the elementwise warps read the ids in order.  A
// slot is rewritten only kItemRing items later, after the held-pair and ring
// barriers have forced every reader past it.
__device__ __forceinline__ void publish_item(const BwdBars& bb, int k, int x) {
  bb.items[k % kItemRing] = x;
  mbar_arrive(&bb.item_full[k % kItemRing]);  // release: the id is visible to the waiters
}

// dK, dV item: key tile j of KV head bhk; iteration n runs over (query head
// of the group, Q tile i) with the Q tiles that can see tile j: all of them,
// or i >= j under the causal (square) rule.
struct KvItem {
  int j, bhk, b, hk, i0, per_head, n_iter;
};
__device__ __forceinline__ KvItem kv_item(int x, int nk, int nq, int B, int Hq, int Hkv,
                                          int causal) {
  KvItem w;
  item_order(x, nk, B * Hkv, w.j, w.bhk);
  w.b = w.bhk / Hkv;
  w.hk = w.bhk % Hkv;
  w.i0 = causal ? w.j : 0;
  w.per_head = nq - w.i0;
  w.n_iter = (Hq / Hkv) * w.per_head;
  return w;
}

// dQ item: Q tile i of query head bhq (the last Q tiles, heaviest under the
// causal rule, first) against the n_iter K/V tiles it sees.
struct QItem {
  int i, bhq, bhk, n_iter;
};
__device__ __forceinline__ QItem q_item(int x, int nk, int nq, int B, int Hq, int Hkv,
                                        int causal) {
  QItem w;
  int t;
  item_order(x, nq, B * Hq, t, w.bhq);
  w.i = nq - 1 - t;
  w.bhk = (w.bhq / Hq) * Hkv + (w.bhq % Hq) / (Hq / Hkv);
  w.n_iter = causal ? min(nk, w.i + 1) : nk;
  return w;
}

}  // namespace

namespace {

// dK, dV of key tiles (persistent CTAs, one item after another).
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const float* __restrict__ nlse,
                    const float* __restrict__ nd, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int B, int Hq, int Hkv, int Lq, int Lk,
                    int causal, float scale, int* work, int* status) {
  using C = BwdCfg<D>;
  using L = BwdSmem<D, kDkdvStg<D>>;
  constexpr bool kTmaEpi = kDkdvStg<D> > 0;
  constexpr int NF = L::NF, NS = L::NS;
  // Two S^T buffers where TMEM has room (d = 64): S^T of the next Q tile is
  // computed while the elementwise warps still work on this one.  At d = 128
  // the accumulators take columns 256..511 and S^T(n + 1) waits for the dV
  // products that read P^T(n) from S^T(n)'s columns.
  constexpr bool kTwoS = C::ACC1_COL + D <= C::S1_COL;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const BwdBars bb = carve_bars(smem + L::OFF_BAR);
  float* vec = reinterpret_cast<float*>(smem + L::OFF_VEC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (Lk + T - 1) / T, nq = (Lq + T - 1) / T;
  const int num_items = nk * B * Hkv;
  const int g = Hq / Hkv;
  const int Lq_pad = nq * T;
  if (!bwd_prologue<NF, NS>(bb, status)) return;
  const uint32_t tmem = *bb.tmem_slot;
  // Tiles: K, V of held slot f at 2f, 2f + 1; Q, dO of ring stage s at
  // 2 NF + 2s, 2 NF + 2s + 1.
  auto tile = [&](int t) { return smem + t * C::TILE_BYTES; };
  auto taddr = [&](int t) { return sbase + static_cast<uint32_t>(t * C::TILE_BYTES); };
  auto wait = [&](uint64_t* bar, int phase_count) {
    return mbar_wait(bar, static_cast<uint32_t>(phase_count) & 1u, bb.abort_flag, kWaitLimitNs);
  };
  auto ring_wait = [&](int n) { return wait(&bb.ring_full[n % NS], n / NS); };
  auto read_item = [&](int k, KvItem& w) -> int {  // 1: item, 0: none left, -1: wait failed
    if (!wait(&bb.item_full[k % kItemRing], k / kItemRing)) return -1;
    const int x = *reinterpret_cast<volatile int*>(&bb.items[k % kItemRing]);
    if (x < 0) return 0;
    w = kv_item(x, nk, nq, B, Hq, Hkv, causal);
    return 1;
  };
  // S^T(n) (n counts the CTA's iterations over all its items): its TMEM
  // columns, its barrier for half hh and that barrier's phase.
  auto s_col = [&](int n) -> uint32_t { return (kTwoS && (n & 1)) ? C::S1_COL : C::S_COL; };
  auto s_bar = [&](int n) { return &bb.s_full[kTwoS ? (n & 1) : 0]; };
  auto s_phase = [&](int n) { return kTwoS ? (n >> 1) : n; };

  if (warp == 0 || warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producers
      // Producer 0 (warp 0) claims and publishes the items and loads K and
      // Q; producer 1 (warp 2) reads the published ids and loads V and dO.
      const int role = warp >> 1;
      prefetch_tmap(role ? &tm_v : &tm_k);
      prefetch_tmap(role ? &tm_do : &tm_q);
      bool ok = true;
      int k = 0, it = 0;
      int x = role ? 0 : atomicAdd(&work[0], 1);
      for (;; ++k) {
        KvItem w;
        if (role == 0) {
          const int cur = x < num_items ? x : -1;
          if (cur >= 0) x = atomicAdd(&work[0], 1);  // the next claim's latency overlaps this item
          publish_item(bb, k, cur);
          if (cur < 0) break;
          w = kv_item(cur, nk, nq, B, Hq, Hkv, causal);
        } else {
          const int got = read_item(k, w);
          if (got < 0) { ok = false; break; }
          if (got == 0) break;
        }
        const int f = k % NF;
        if (k >= NF && !wait(&bb.hold_empty[f], k / NF - 1)) { ok = false; break; }
        uint64_t* hb = &bb.hold_full[f];
        if (role == 0) mbar_arrive_expect_tx(hb, 2 * C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(tile(2 * f + role) + kb * C::BLOCK_BYTES, role ? &tm_v : &tm_k, hb, kb * 64,
                      w.j * T, w.bhk);
        for (int n = 0; n < w.n_iter; ++n, ++it) {
          const int st = it % NS;
          if (it >= NS && !wait(&bb.ring_empty[st], it / NS - 1)) { ok = false; break; }
          const int bhq = w.b * Hq + w.hk * g + n / w.per_head;
          const int i = w.i0 + n % w.per_head;
          uint64_t* rb = &bb.ring_full[st];
          if (role == 0) mbar_arrive_expect_tx(rb, 2 * C::TILE_BYTES + 2 * T * 4);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(tile(2 * NF + 2 * st + role) + kb * C::BLOCK_BYTES, role ? &tm_do : &tm_q, rb,
                        kb * 64, i * T, bhq);
          // The Q tile's -LSE log2e (producer 0) or -D (producer 1).
          bulk_load(vec + (2 * st + role) * T, (role ? nd : nlse) + static_cast<size_t>(bhq) * Lq_pad + i * T,
                    T * 4, rb);
        }
        if (!ok) { ++k; break; }
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      // Drain: every copy this thread issued (k items' held tiles, `it`
      // ring tiles) has landed before the CTA may exit.  After an abort the
      // other producer may not have armed a barrier: the short limit then
      // ends the wait (a copy lands within microseconds).
      int no_abort = 0;
      for (int kk = k > NF ? k - NF : 0; kk < k; ++kk)
        mbar_wait(&bb.hold_full[kk % NF], (kk / NF) & 1, &no_abort, kDrainLimitNs);
      for (int n = it > NS ? it - NS : 0; n < it; ++n)
        mbar_wait(&bb.ring_full[n % NS], (n / NS) & 1, &no_abort, kDrainLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      bool ok = true;
      int it = 0;
      for (int k = 0; ok; ++k) {
        KvItem w;
        const int got = read_item(k, w);
        if (got <= 0) { ok = got == 0; break; }
        const int f = k % NF;
        const uint64_t k_desc = smem_desc_sw128(taddr(2 * f), 16, 1024);
        const uint64_t v_desc = smem_desc_sw128(taddr(2 * f + 1), 16, 1024);
        // S^T(n) = K Q_n^T (keys as rows, queries as columns).
        auto issue_s = [&](int n) {
          const uint64_t q_k = smem_desc_sw128(taddr(2 * NF + 2 * (n % NS)), 16, 1024);
          mma_kmajor_full<D>(tmem + s_col(n), k_desc, q_k);
          mma_commit(s_bar(n));
        };
        // dP^T(n) = V dO_n^T.
        auto issue_dp = [&](int n) {
          const uint64_t do_k = smem_desc_sw128(taddr(2 * NF + 2 * (n % NS) + 1), 16, 1024);
          mma_kmajor_full<D>(tmem + C::DP_COL, v_desc, do_k);
          mma_commit(&bb.dp_full[0]);
        };
        if (!wait(&bb.hold_full[f], k / NF) || !ring_wait(it)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(it);
        issue_dp(it);
        for (int n = 0; ok && n < w.n_iter; ++n, ++it) {
          const int st = it % NS;
          const bool more = n + 1 < w.n_iter;
          if (kTwoS && more) {
            if (!ring_wait(it + 1)) { ok = false; break; }
            tc_fence_after();
            issue_s(it + 1);
          }
          // dV += P^T dO_n once both groups have written P^T (bf16 pairs in
          // the first 32 columns of each query half's S^T columns; dO rows
          // h * 64..).  The first product of an item overwrites the
          // accumulator: both groups have stored the previous item's
          // gradients before their P^T(n) arrival.
          const uint64_t q_mn = smem_desc_sw128(taddr(2 * NF + 2 * st), C::BLOCK_BYTES, 1024);
          const uint64_t do_mn = smem_desc_sw128(taddr(2 * NF + 2 * st + 1), C::BLOCK_BYTES, 1024);
          if (!wait(&bb.p_ready[it & 1], it >> 1)) { ok = false; break; }
          tc_fence_after();
          for (int hh = 0; hh < 2; ++hh)
            mma_tmem_a_half<D>(tmem + C::ACC1_COL, tmem + s_col(it) + hh * H,
                               do_mn + hh * kHalfStep, n > 0 || hh > 0);
          if (!kTwoS && more) {
            if (!ring_wait(it + 1)) { ok = false; break; }
            tc_fence_after();
            issue_s(it + 1);  // over P^T(n), after the dV products that read it
          }
          // dK += dS^T Q_n once both groups have written dS^T, then dP^T(n + 1)
          // over the dP^T columns those products read.
          if (!wait(bb.ds_ready, it)) { ok = false; break; }
          tc_fence_after();
          for (int hh = 0; hh < 2; ++hh)
            mma_tmem_a_half<D>(tmem + C::ACC0_COL, tmem + C::DP_COL + hh * H,
                               q_mn + hh * kHalfStep, n > 0 || hh > 0);
          if (more) issue_dp(it + 1);
          mma_commit(&bb.ring_empty[st]);  // Q and dO of this stage may be refilled
        }
        if (!ok) break;
        mma_commit(bb.acc_done);
        mma_commit(&bb.hold_empty[f]);     // K and V of this slot may be refilled
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      int no_abort = 0;
      mma_commit(bb.drain);
      mbar_wait(bb.drain, 0, &no_abort, kWaitLimitNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise
    // Two groups of four warps: group hh works on query half hh of every
    // tile pair, each thread on key row c (its TMEM lane).
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int c = quad * 32 + lane;               // key row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float scale_log2 = scale * attn::kLog2e;
    KvItem w, nxt;
    int got = __shfl_sync(FULL, read_item(0, w), 0);
    bool ok = got >= 0;
    int it = 0;
    for (int k = 0; ok && got > 0; ++k) {
      int got_next = 0;
      int i = w.i0;                                // iteration n's Q tile
      for (int n = 0; n < w.n_iter; ++n, ++it) {
        const int st = it & 1;
        // The Q tile's -LSE log2e and -D came with it into ring stage it % NS.
        ok = __all_sync(FULL, wait(&bb.ring_full[it % NS], it / NS));
        if (!ok) break;
        const float* l2s = vec + (it % NS) * 2 * T;
        const float* ds_ = l2s + T;
        // P^T row c over this group's query half: P[r] = 2^(S^T[c][r] scale
        // log2e - LSE_r log2e), 0 for queries before key c on the diagonal
        // tile; bf16 pairs over the half's first 32 S^T columns.
        ok = __all_sync(FULL, wait(s_bar(it), s_phase(it)));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_off + s_col(it) + half * H;
        uint32_t pw[H / 2];
        {
          uint32_t sr[2][32];
          tmem_ld32(s_addr, sr[0]);
          tmem_ld32(s_addr + 32, sr[1]);
          tmem_ld_wait();
          float x[H];
          const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
          for (int e = 0; e < H; e += 4) {
            const float4 nl = *reinterpret_cast<const float4*>(&l2s[half * H + e]);
            const float2 xa = ffma2(make_float2(__uint_as_float(sr[e >> 5][e & 31]),
                                                __uint_as_float(sr[e >> 5][(e & 31) + 1])),
                                    sc2, make_float2(nl.x, nl.y));
            const float2 xb = ffma2(make_float2(__uint_as_float(sr[e >> 5][(e & 31) + 2]),
                                                __uint_as_float(sr[e >> 5][(e & 31) + 3])),
                                    sc2, make_float2(nl.z, nl.w));
            x[e] = xa.x;
            x[e + 1] = xa.y;
            x[e + 2] = xb.x;
            x[e + 3] = xb.y;
          }
          if (causal && i == w.j) {                // query i T + half H + e < key j T + c
            const int lo = c - half * H;
#pragma unroll
            for (int e = 0; e < H; ++e) x[e] = neg_inf_if_lt(x[e], e, lo);
          }
#pragma unroll
          for (int e = 0; e < H; e += 2) pw[e >> 1] = attn::pack_bf16x2(ex2(x[e]), ex2(x[e + 1]));
        }
        tmem_st32(s_addr, pw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.p_ready[st]);
        if (++i == nq) i = w.i0;
        if (n + 1 == w.n_iter) {                   // the next item, while dP^T is computed
          got_next = read_item(k + 1, nxt);
          ok = __all_sync(FULL, got_next >= 0);
          if (!ok) break;
        }
        // dS^T row c: dS[r] = P[r] (dP^T[c][r] - D_r), with P as handed to
        // the MMA, over the half's first 32 dP^T columns (already read).
        ok = __all_sync(FULL, wait(bb.dp_full, it));
        if (!ok) break;
        tc_fence_after();
        const uint32_t dp_addr = tmem + lane_off + C::DP_COL + half * H;
        uint32_t dr[2][32];
        tmem_ld32(dp_addr, dr[0]);
        tmem_ld32(dp_addr + 32, dr[1]);
        tmem_ld_wait();
        uint32_t sw[H / 2];
        const float2 zero2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < H; e += 4) {
          const float4 nd = *reinterpret_cast<const float4*>(&ds_[half * H + e]);
          const float2 xa = fadd2(make_float2(__uint_as_float(dr[e >> 5][e & 31]),
                                              __uint_as_float(dr[e >> 5][(e & 31) + 1])),
                                  make_float2(nd.x, nd.y));
          const float2 xb = fadd2(make_float2(__uint_as_float(dr[e >> 5][(e & 31) + 2]),
                                              __uint_as_float(dr[e >> 5][(e & 31) + 3])),
                                  make_float2(nd.z, nd.w));
          const uint32_t p0 = pw[e >> 1], p1 = pw[(e >> 1) + 1];
          const float2 sa = ffma2(make_float2(attn::bf16_lo(p0), attn::bf16_hi(p0)), xa, zero2);
          const float2 sb = ffma2(make_float2(attn::bf16_lo(p1), attn::bf16_hi(p1)), xb, zero2);
          sw[e >> 1] = attn::pack_bf16x2(sa.x, sa.y);
          sw[(e >> 1) + 1] = attn::pack_bf16x2(sb.x, sb.y);
        }
        tmem_st32(dp_addr, sw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bb.ds_ready);
      }
      if (!ok) break;
      // The item's gradients: group 0 writes dV row j T + c, group 1 dK.
      ok = __all_sync(FULL, wait(bb.acc_done, k));
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc_col = half == 0 ? C::ACC1_COL : C::ACC0_COL;
      const float mul = half == 0 ? 1.f : scale;
      if constexpr (kTmaEpi) {
        // Into the group's staging tile (once the previous item's store has
        // read it: its issuing thread checks and signals here, an item
        // later, so the store overlaps that item), then the group's first
        // warp stores the tile with TMA; rows past Lk are clipped by the map.
        if (k > 0) {
          if (quad == 0 && lane == 0) {
            bulk_wait_read_all();
            mbar_arrive(&bb.st_free[half]);
          }
          ok = __all_sync(FULL, wait(&bb.st_free[half], k - 1));
          if (!ok) break;
        }
        uint8_t* stg = smem + L::OFF_STG + half * C::TILE_BYTES;
        stage_row64_bf16(tmem + lane_off + acc_col, mul, stg, c);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.st_ready[half]);
        if (quad == 0 && lane == 0) {
          if (wait(&bb.st_ready[half], k)) {
            tma_store_3d(half == 0 ? &tm_dv : &tm_dk, stg, 0, w.j * T, w.bhk);
            bulk_commit_group();
          } else {
            ok = false;
          }
        }
        ok = __shfl_sync(FULL, ok, 0);
        if (!ok) break;
      } else {
        const int kk = w.j * T + c;
        const bool live = kk < Lk;
        const size_t out_row = (static_cast<size_t>(w.bhk) * Lk + (live ? kk : 0)) * D;
        store_cols_bf16<D / 32>(tmem + lane_off + acc_col, mul, (half == 0 ? dv : dk) + out_row,
                                live);
      }
      tc_fence_before();
      w = nxt;
      got = got_next;
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *bb.abort_flag = 1;
    }
    if constexpr (kTmaEpi)
      if (quad == 0 && lane == 0) bulk_wait_all();  // the tile stores have completed
  }
  bwd_epilogue(bb);
}

}  // namespace

namespace {

// dQ of Q tiles (persistent CTAs, one item after another): the K/V tiles an
// item sees stream through the ring.
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ nlse,
                  const float* __restrict__ nd, __nv_bfloat16* __restrict__ dq, int B, int Hq,
                  int Hkv, int Lq, int Lk, int causal, float scale, int* work, int* status) {
  using C = BwdCfg<D>;
  using L = BwdSmem<D, kDqStg<D>>;
  constexpr bool kTmaEpi = kDqStg<D> > 0;
  constexpr int NF = L::NF, NS = L::NS;
  // d = 64: one S buffer and two dP buffers (TMEM columns 128 and 384; the
  // accumulator takes D columns from 256).  The elementwise warps turn S
  // into P first and signal (p_ready[0]), so S and dP of the next K/V tile
  // are computed while they work on dS of this one.  d = 128 (long
  // products): two S buffers (0 and 384) and one dP buffer; S of the next
  // tile is issued early, its dP after the dQ products that read dS.
  constexpr bool kEarlyS = D == 64;
  static_assert(C::ACC0_COL + D <= C::S1_COL, "TMEM columns");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const BwdBars bb = carve_bars(smem + L::OFF_BAR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (Lk + T - 1) / T, nq = (Lq + T - 1) / T;
  const int num_items = nq * B * Hq;
  const int Lq_pad = nq * T;
  if (!bwd_prologue<NF, NS>(bb, status)) return;
  const uint32_t tmem = *bb.tmem_slot;
  // Tiles: Q, dO of held slot f at 2f, 2f + 1; K, V of ring stage s at
  // 2 NF + 2s, 2 NF + 2s + 1.
  auto tile = [&](int tt) { return smem + tt * C::TILE_BYTES; };
  auto taddr = [&](int tt) { return sbase + static_cast<uint32_t>(tt * C::TILE_BYTES); };
  auto wait = [&](uint64_t* bar, int phase_count) {
    return mbar_wait(bar, static_cast<uint32_t>(phase_count) & 1u, bb.abort_flag, kWaitLimitNs);
  };
  auto ring_wait = [&](int n) { return wait(&bb.ring_full[n % NS], n / NS); };
  auto read_item = [&](int k, QItem& w) -> int {  // 1: item, 0: none left, -1: wait failed
    if (!wait(&bb.item_full[k % kItemRing], k / kItemRing)) return -1;
    const int x = *reinterpret_cast<volatile int*>(&bb.items[k % kItemRing]);
    if (x < 0) return 0;
    w = q_item(x, nk, nq, B, Hq, Hkv, causal);
    return 1;
  };
  auto dp_col = [&](int it) -> uint32_t {
    return (kEarlyS && (it & 1)) ? C::S1_COL : C::DP_COL;
  };
  auto s_col = [&](int it) -> uint32_t {
    return (!kEarlyS && (it & 1)) ? C::S1_COL : C::S_COL;
  };
  // S(it) / dP(it): barrier and phase.
  auto s_bar = [&](int it) { return &bb.s_full[kEarlyS ? 0 : (it & 1)]; };
  auto s_ph = [&](int it) { return kEarlyS ? it : (it >> 1); };
  auto dp_bar = [&](int it) { return &bb.dp_full[kEarlyS ? (it & 1) : 0]; };
  auto dp_ph = [&](int it) { return kEarlyS ? (it >> 1) : it; };
  uint64_t* s_read = &bb.p_ready[0];  // every elementwise warp has read S (d = 64)

  if (warp == 0 || warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producers
      // Producer 0 (warp 0) claims and publishes the items and loads Q and
      // K; producer 1 (warp 2) reads the published ids and loads dO and V.
      const int role = warp >> 1;
      prefetch_tmap(role ? &tm_do : &tm_q);
      prefetch_tmap(role ? &tm_v : &tm_k);
      bool ok = true;
      int k = 0, it = 0;
      int x = role ? 0 : atomicAdd(&work[1], 1);
      for (;; ++k) {
        QItem w;
        if (role == 0) {
          const int cur = x < num_items ? x : -1;
          if (cur >= 0) x = atomicAdd(&work[1], 1);
          publish_item(bb, k, cur);
          if (cur < 0) break;
          w = q_item(cur, nk, nq, B, Hq, Hkv, causal);
        } else {
          const int got = read_item(k, w);
          if (got < 0) { ok = false; break; }
          if (got == 0) break;
        }
        const int f = k % NF;
        if (k >= NF && !wait(&bb.hold_empty[f], k / NF - 1)) { ok = false; break; }
        uint64_t* hb = &bb.hold_full[f];
        if (role == 0) mbar_arrive_expect_tx(hb, 2 * C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(tile(2 * f + role) + kb * C::BLOCK_BYTES, role ? &tm_do : &tm_q, hb, kb * 64,
                      w.i * T, w.bhq);
        for (int jt = 0; jt < w.n_iter; ++jt, ++it) {
          const int st = it % NS;
          if (it >= NS && !wait(&bb.ring_empty[st], it / NS - 1)) { ok = false; break; }
          uint64_t* rb = &bb.ring_full[st];
          if (role == 0) mbar_arrive_expect_tx(rb, 2 * C::TILE_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(tile(2 * NF + 2 * st + role) + kb * C::BLOCK_BYTES, role ? &tm_v : &tm_k, rb,
                        kb * 64, jt * T, w.bhk);
        }
        if (!ok) { ++k; break; }
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      int no_abort = 0;
      for (int kk = k > NF ? k - NF : 0; kk < k; ++kk)
        mbar_wait(&bb.hold_full[kk % NF], (kk / NF) & 1, &no_abort, kDrainLimitNs);
      for (int n = it > NS ? it - NS : 0; n < it; ++n)
        mbar_wait(&bb.ring_full[n % NS], (n / NS) & 1, &no_abort, kDrainLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      bool ok = true;
      int it = 0;
      for (int k = 0; ok; ++k) {
        QItem w;
        const int got = read_item(k, w);
        if (got <= 0) { ok = got == 0; break; }
        const int f = k % NF;
        const uint64_t q_desc = smem_desc_sw128(taddr(2 * f), 16, 1024);
        const uint64_t do_desc = smem_desc_sw128(taddr(2 * f + 1), 16, 1024);
        // S(n) = Q K^T (queries as rows, keys as columns); at d = 64 once
        // the warps have read S(n - 1).
        auto issue_s = [&](int n) {
          const uint64_t k_k = smem_desc_sw128(taddr(2 * NF + 2 * (n % NS)), 16, 1024);
          mma_kmajor_full<D>(tmem + s_col(n), q_desc, k_k);
          mma_commit(s_bar(n));
        };
        // dP(n) = dO V^T into its buffer, whose dS the dQ products issued
        // earlier read.
        auto issue_dp = [&](int n) {
          const uint64_t v_k = smem_desc_sw128(taddr(2 * NF + 2 * (n % NS) + 1), 16, 1024);
          mma_kmajor_full<D>(tmem + dp_col(n), do_desc, v_k);
          mma_commit(dp_bar(n));
        };
        if (!wait(&bb.hold_full[f], k / NF) || !ring_wait(it) ||
            (kEarlyS && it > 0 && !wait(s_read, it - 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(it);
        issue_dp(it);
        for (int jt = 0; ok && jt < w.n_iter; ++jt, ++it) {
          const int st = it % NS;
          const bool more = jt + 1 < w.n_iter;
          if (more) {
            if (!ring_wait(it + 1) || (kEarlyS && !wait(s_read, it))) { ok = false; break; }
            tc_fence_after();
            issue_s(it + 1);
            if (kEarlyS) issue_dp(it + 1);
          }
          // dQ += dS K once both groups have written dS (bf16 pairs in the
          // first 32 columns of each key half of dP buffer it & 1; K rows
          // h * 64..).  The item's first product overwrites the accumulator:
          // group 0, which alone stores dQ, has done so before its dS arrival.
          const uint64_t k_mn = smem_desc_sw128(taddr(2 * NF + 2 * st), C::BLOCK_BYTES, 1024);
          if (!wait(&bb.ds_ready[it & 1], it >> 1)) { ok = false; break; }
          tc_fence_after();
          for (int hh = 0; hh < 2; ++hh)
            mma_tmem_a_half<D>(tmem + C::ACC0_COL, tmem + dp_col(it) + hh * H,
                               k_mn + hh * kHalfStep, jt > 0 || hh > 0);
          if (!kEarlyS && more) issue_dp(it + 1);  // over dS(it), after the products above
          mma_commit(&bb.ring_empty[st]);  // K and V of this stage may be refilled
        }
        if (!ok) break;
        mma_commit(bb.acc_done);
        mma_commit(&bb.hold_empty[f]);     // Q and dO of this slot may be refilled
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      int no_abort = 0;
      mma_commit(bb.drain);
      mbar_wait(bb.drain, 0, &no_abort, kWaitLimitNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise
    // Two groups of four warps: group hh works on key half hh of every K/V
    // tile, each thread on query row r (its TMEM lane).
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float scale_log2 = scale * attn::kLog2e;
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    const float2 zero2 = make_float2(0.f, 0.f);
    // -LSE log2e (-inf where the row does not exist or sees no key: P = 0)
    // and -D of this thread's query row in item w.
    // -LSE log2e and -D of this thread's query row in item w (padded
    // layout: rows past Lq hold -inf and 0).  The next item's values are
    // loaded in this item's last iteration, which hides their latency.
    float pre_l = 0.f, pre_d = 0.f;
    auto fetch = [&](const QItem& w) {
      const size_t at = static_cast<size_t>(w.bhq) * Lq_pad + w.i * T + r;
      pre_l = nlse[at];
      pre_d = nd[at];
    };
    QItem w, nxt;
    int got = __shfl_sync(FULL, read_item(0, w), 0);
    bool ok = got >= 0;
    if (got > 0) fetch(w);
    int it = 0;
    for (int k = 0; ok && got > 0; ++k) {
      const float2 nl2 = make_float2(pre_l, pre_l), nd2 = make_float2(pre_d, pre_d);
      const int qrow = w.i * T + r;
      // Keys past Lk, and past the query under the causal rule, get P = 0;
      // only the diagonal tile and a ragged last tile hold any.
      const int kmax = causal ? min(Lk - 1, qrow) : Lk - 1;
      int got_next = 0;
      for (int jt = 0; jt < w.n_iter; ++jt, ++it) {
        if (jt + 1 == w.n_iter) {                  // the next item's row values
          got_next = read_item(k + 1, nxt);
          ok = __all_sync(FULL, got_next >= 0);
          if (!ok) break;
          if (got_next > 0) fetch(nxt);
        }
        const bool need_mask = (causal && jt == w.i) || (jt + 1) * T > Lk;
        // P over this group's 64 keys (rounded to bf16 as in the forward's
        // P V product and in bwd_dkdv), then the S columns are released.
        ok = __all_sync(FULL, wait(s_bar(it), s_ph(it)));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_off + s_col(it) + half * H;
        uint32_t pw[H / 2];
        {
          uint32_t sr[2][32];
          tmem_ld32(s_addr, sr[0]);
          tmem_ld32(s_addr + 32, sr[1]);
          tmem_ld_wait();
          float x[H];
#pragma unroll
          for (int e = 0; e < H; e += 2) {
            const float2 p = ffma2(make_float2(__uint_as_float(sr[e >> 5][e & 31]),
                                               __uint_as_float(sr[e >> 5][(e & 31) + 1])),
                                   sc2, nl2);
            x[e] = p.x;
            x[e + 1] = p.y;
          }
          if (need_mask) {
            const int kv = kmax - (jt * T + half * H);
#pragma unroll
            for (int e = 0; e < H; ++e) x[e] = neg_inf_if_gt(x[e], e, kv);
          }
#pragma unroll
          for (int e = 0; e < H; e += 2) pw[e >> 1] = attn::pack_bf16x2(ex2(x[e]), ex2(x[e + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_read);
        // dS = P (dP - D) over the half's first 32 columns of dP buffer it & 1
        // (already read).
        ok = __all_sync(FULL, wait(dp_bar(it), dp_ph(it)));
        if (!ok) break;
        tc_fence_after();
        const uint32_t dp_addr = tmem + lane_off + dp_col(it) + half * H;
        uint32_t dr[2][32];
        tmem_ld32(dp_addr, dr[0]);
        tmem_ld32(dp_addr + 32, dr[1]);
        tmem_ld_wait();
        uint32_t sw[H / 2];
#pragma unroll
        for (int e = 0; e < H; e += 2) {
          const float2 xd = fadd2(make_float2(__uint_as_float(dr[e >> 5][e & 31]),
                                              __uint_as_float(dr[e >> 5][(e & 31) + 1])),
                                  nd2);
          const uint32_t p = pw[e >> 1];
          const float2 ds2 = ffma2(make_float2(attn::bf16_lo(p), attn::bf16_hi(p)), xd, zero2);
          sw[e >> 1] = attn::pack_bf16x2(ds2.x, ds2.y);
        }
        tmem_st32(dp_addr, sw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.ds_ready[it & 1]);
      }
      if (!ok) break;
      if (half == 0) {
        // Group 0 writes dQ row qrow (all D columns): at d = 64 through its
        // staging tile and one TMA store by warp 4 (rows past Lq clipped).
        ok = __all_sync(FULL, wait(bb.acc_done, k));
        if (!ok) break;
        tc_fence_after();
        if constexpr (kTmaEpi) {
          if (k > 0) {  // the previous item's store has read the staging tile
            if (quad == 0 && lane == 0) {
              bulk_wait_read_all();
              mbar_arrive(&bb.st_free[0]);
            }
            ok = __all_sync(FULL, wait(&bb.st_free[0], k - 1));
            if (!ok) break;
          }
          uint8_t* stg = smem + L::OFF_STG;
          stage_row64_bf16(tmem + lane_off + C::ACC0_COL, scale, stg, r);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb.st_ready[0]);
          if (quad == 0 && lane == 0) {
            if (wait(&bb.st_ready[0], k)) {
              tma_store_3d(&tm_dq, stg, 0, w.i * T, w.bhq);
              bulk_commit_group();
            } else {
              ok = false;
            }
          }
          ok = __shfl_sync(FULL, ok, 0);
          if (!ok) break;
        } else {
          const bool live = qrow < Lq;
          const size_t out_row = (static_cast<size_t>(w.bhq) * Lq + (live ? qrow : 0)) * D;
          store_cols_bf16<D / 32>(tmem + lane_off + C::ACC0_COL, scale, dq + out_row, live);
        }
        tc_fence_before();
      }
      w = nxt;
      got = got_next;
    }
    if (!ok) {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *bb.abort_flag = 1;
    }
    if constexpr (kTmaEpi)
      if (half == 0 && quad == 0 && lane == 0) bulk_wait_all();  // the tile stores have completed
  }
  bwd_epilogue(bb);
}

}  // namespace

namespace {

// [BH heads, L rows] x d bf16 as a 3-D tensor {d, L, BH}; box {64, 128, 1}
// with 128-byte swizzle (the layout the MMA descriptors above assume).  Rows
// past L read as zeros.
bool make_map_rows(CUtensorMap* m, const void* base, int D, int L, int BH) {
  attn_host::EncodeTiledFn enc = attn_host::encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(L) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(T), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                         float* dd, int B, int Hq, int Hkv, int Lq, int Lk, int causal,
                         float scale, cudaStream_t stream) {
  using LK = BwdSmem<D, kDkdvStg<D>>;
  using LQ = BwdSmem<D, kDqStg<D>>;
  static bool attr_set[64] = {};  // per device: kernel attributes are per device
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return ATTN_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LK::BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LQ::BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!make_map_rows(&mq, q, D, Lq, B * Hq) || !make_map_rows(&mk, k, D, Lk, B * Hkv) ||
      !make_map_rows(&mv, v, D, Lk, B * Hkv) || !make_map_rows(&mdo, d_o, D, Lq, B * Hq) ||
      !make_map_rows(&mdq, dq, D, Lq, B * Hq) || !make_map_rows(&mdk, dk, D, Lk, B * Hkv) ||
      !make_map_rows(&mdv, dv, D, Lk, B * Hkv))
    return ATTN_ERR_CUDA;
  const long long nq = (Lq + T - 1) / T, nk = (Lk + T - 1) / T;
  const long long dq_ctas = nq * B * Hq, dkdv_ctas = nk * B * Hkv;
  if (static_cast<long long>(B) * Hq * nq * T / 8 > 0x7fffffffLL || nq * T > 0x7fffffffLL ||
      dq_ctas > 0x7fffffffLL || dkdv_ctas > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  int* status = attn_host::device_status_ptr();
  // Workspace: -LSE log2e and -D in the padded [B Hq][nq 128] layout, then
  // the two work counters (each part at a 256-byte boundary).
  const size_t part = (static_cast<size_t>(B) * Hq * nq * T * sizeof(float) + 255) & ~size_t{255};
  float* nlse = dd;
  float* nd = reinterpret_cast<float*>(reinterpret_cast<char*>(dd) + part);
  int* work = reinterpret_cast<int*>(reinterpret_cast<char*>(dd) + 2 * part);
  const long long sms = attn_host::num_sms();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const long long heads = static_cast<long long>(B) * Hq;
  const long long rows_pad = heads * nq * T;
  const long long rd_blocks = std::min((rows_pad + 8 * (256 / D) - 1) / (8 * (256 / D)), sms * 16);
  bwd_rowdot_kernel<D><<<static_cast<unsigned>(rd_blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), lse, nlse, nd,
      heads, Lq, static_cast<int>(nq * T), work);
  bwd_dkdv_kernel<D><<<static_cast<unsigned>(std::min(dkdv_ctas, sms)), THREADS, LK::BYTES, stream>>>(
      mq, mk, mv, mdo, mdk, mdv, nlse, nd, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
      B, Hq, Hkv, Lq, Lk, causal, scale, work, status);
  bwd_dq_kernel<D><<<static_cast<unsigned>(std::min(dq_ctas, sms)), THREADS, LQ::BYTES, stream>>>(
      mq, mk, mv, mdo, mdq, nlse, nd, static_cast<__nv_bfloat16*>(dq), B, Hq, Hkv, Lq, Lk, causal,
      scale, work, status);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

attn_status_t launch_bwd_bf16(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                              float* dd, int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                              float scale, cudaStream_t stream) {
  if (d == 64)
    return launch_bwd<64>(q, k, v, o, lse, d_o, dq, dk, dv, dd, B, Hq, Hkv, Lq, Lk, causal, scale,
                          stream);
  if (d == 128)
    return launch_bwd<128>(q, k, v, o, lse, d_o, dq, dk, dv, dd, B, Hq, Hkv, Lq, Lk, causal,
                           scale, stream);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn_host
