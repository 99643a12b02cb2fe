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
//   bwd_rowdot_kernel   D = rowsum(dO * O) per query row (fp32).
//   bwd_dkdv_kernel     one CTA per (request, KV head, key tile j): K_j, V_j
//                       stay in shared memory while the Q tiles of every
//                       query head of the group stream past; per Q tile four
//                       tcgen05 MMAs with the 128 keys as the M dimension:
//                         S^T  = K_j Q_i^T           (TMEM, fp32)
//                         dP^T = V_j dO_i^T          (TMEM, fp32)
//                         dV  += P^T dO_i            (P^T bf16 from TMEM)
//                         dK  += dS^T Q_i            (dS^T bf16 from TMEM)
//                       so neither P nor dS is ever transposed.
//   bwd_dq_kernel       one CTA per (request, query head, Q tile i): Q_i and
//                       dO_i stay while the K/V tiles stream past; per K/V
//                       tile three MMAs with the queries as M:
//                         S = Q_i K_j^T,  dP = dO_i V_j^T,  dQ += dS K_j.
// Recomputing S and dP in both kernels costs two extra GEMMs per tile pair
// against a single kernel that adds dQ with atomics; in exchange the result
// does not depend on the order in which CTAs finish.
//
// Roles (both MMA kernels, 256 threads, one CTA per SM): warp 0 lane 0 loads
// tiles with TMA, warp 1 lane 0 issues the MMAs, warps 4-7 (one thread per
// TMEM lane, i.e. per key row in bwd_dkdv and per query row in bwd_dq) do
// the elementwise work.  Every wait is bounded (ATTN_ERR_DEVICE_TIMEOUT, CTA
// abort, drain, TMEM freed), as in the forward kernels.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace {

using namespace sm103;

constexpr int T = 128;               // rows of a Q or K/V tile (MMA M and N)
constexpr int THREADS = 256;         // 8 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
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
  // accumulators.  P^T / dS^T (bf16 pairs) overwrite the first 64 columns
  // of S^T / dP^T.
  static constexpr uint32_t S_COL = 0, DP_COL = 128, ACC0_COL = 256, ACC1_COL = 256 + D;
};

// Instruction descriptor: kind::f16, bf16 A/B, fp32 D, M = 128.
__host__ __device__ constexpr uint32_t idesc(int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(T >> 4) << 24);
}

// A tile is processed in two halves of H = 64 rows (queries in bwd_dkdv,
// keys in bwd_dq): the elementwise warps start on the first half while the
// tensor core computes the second.  Half h of a K-major or MN-major tile
// starts 64 rows (8 KB, eight whole swizzle atoms) into each column block.
constexpr int H = T / 2;
constexpr uint64_t kHalfStep = (H * 128) >> 4;  // descriptor start-address step of a half

// D(tmem, 128 x H fp32) = A B^T for the 128-row K-major tile A and half of
// the K-major tile B ([rows][D] bf16, 128-byte swizzle, KB column blocks of
// BLOCK_BYTES): one MMA per 16 columns of D.
template <int D>
__device__ __forceinline__ void mma_kmajor_half(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint64_t kBlk = BwdCfg<D>::BLOCK_BYTES >> 4;
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint64_t off = (k >> 2) * kBlk + (k & 3) * 2;
    mma_bf16_ss(d_tmem, a_desc + off, b_desc + off, idesc(H, false), k > 0 ? 1u : 0u);
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
__global__ void bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ o,
                                  const __nv_bfloat16* __restrict__ d_o, float* __restrict__ dd,
                                  long long rows, int d) {
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint32_t* op = reinterpret_cast<const uint32_t*>(o + r * d);
  const uint32_t* gp = reinterpret_cast<const uint32_t*>(d_o + r * d);
  float acc = 0.f;
  for (int c = lane; c < d / 2; c += 32) {
    const uint32_t a = op[c], b = gp[c];
    acc = fmaf(attn::bf16_lo(a), attn::bf16_lo(b), acc);
    acc = fmaf(attn::bf16_hi(a), attn::bf16_hi(b), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(FULL, acc, off);
  if (lane == 0) dd[r] = acc;
}

}  // namespace

namespace {

// Shared-memory layout of both MMA kernels: six bf16 tiles, then two stages
// of 128 fp32 per-query values (LSE and D) used by bwd_dkdv, then barriers.
template <int D>
struct BwdSmem {
  using C = BwdCfg<D>;
  // 6 tiles at t * TILE_BYTES
  static constexpr int OFF_VEC = 6 * C::TILE_BYTES;
  static constexpr int OFF_BAR = OFF_VEC + 4 * T * 4;
  static constexpr int USED = OFF_BAR + 256 + 1024;  // barriers + alignment slack
  // d = 64 would fit two CTAs per SM; each CTA takes all 512 TMEM columns,
  // so the request is padded to keep one CTA per SM.
  static constexpr int BYTES = USED > 120 * 1024 ? USED : 120 * 1024;
};

struct BwdBars {
  uint64_t* kv_full;   // [2]
  uint64_t* kv_empty;  // [2]
  uint64_t* q_full;    // [2]
  uint64_t* q_empty;   // [2]
  uint64_t* s_full;    // [2] per half: S (S^T) of the half is in TMEM
  uint64_t* dp_full;   // [2] per half: dP (dP^T)
  uint64_t* p_ready;   // [2] per half: P^T written (bwd_dkdv)
  uint64_t* ds_ready;  // [2] per half: dS (dS^T) written
  uint64_t* acc_done;
  uint64_t* drain;
  uint64_t* vec_full;  // [2] per-query values staged by the elementwise warps
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ BwdBars carve_bars(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base);
  BwdBars r;
  r.kv_full = b;
  r.kv_empty = b + 2;
  r.q_full = b + 4;
  r.q_empty = b + 6;
  r.s_full = b + 8;
  r.dp_full = b + 10;
  r.p_ready = b + 12;
  r.ds_ready = b + 14;
  r.acc_done = b + 16;
  r.drain = b + 17;
  r.vec_full = b + 18;
  r.tmem_slot = reinterpret_cast<uint32_t*>(b + 20);
  r.abort_flag = reinterpret_cast<volatile int*>(r.tmem_slot + 1);
  return r;
}

// Barrier set-up, the pending-timeout check and the TMEM allocation shared
// by both kernels.  Returns false when the CTA must skip its work.
__device__ __forceinline__ bool bwd_prologue(const BwdBars& bb, int* status) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb.kv_full[s], 1);
      mbar_init(&bb.kv_empty[s], 1);
      mbar_init(&bb.q_full[s], 1);
      mbar_init(&bb.q_empty[s], 1);
      mbar_init(&bb.s_full[s], 1);
      mbar_init(&bb.dp_full[s], 1);
      mbar_init(&bb.p_ready[s], 4);   // one arrival per elementwise warp
      mbar_init(&bb.ds_ready[s], 4);
    }
    mbar_init(bb.acc_done, 1);
    mbar_init(bb.drain, 1);
    mbar_init(&bb.vec_full[0], 4);
    mbar_init(&bb.vec_full[1], 4);
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

// Writes one 128-column-or-less fp32 TMEM row (D columns from `col`) times
// `mul` as bf16 to global memory (16-byte stores).
template <int D>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                               bool live) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
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

}  // namespace

namespace {

// dK, dV of one key tile j of one (request, KV head).  Iteration n runs over
// (query head of the group, Q tile i) with the Q tiles that can see tile j:
// all of them, or i >= j under the causal (square) rule.
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                    const float* __restrict__ dd, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int B, int Hq, int Hkv, int Lq, int Lk,
                    int causal, float scale, int* status) {
  using C = BwdCfg<D>;
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const BwdBars bb = carve_bars(smem + L::OFF_BAR);
  float* vec = reinterpret_cast<float*>(smem + L::OFF_VEC);  // [2 stages][LSE*log2e | D][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (Lk + T - 1) / T, nq = (Lq + T - 1) / T;
  const int BHkv = B * Hkv;
  // Heaviest first under the causal rule: all key tiles 0, then tiles 1, ...
  const int j = static_cast<int>(blockIdx.x) / BHkv;
  const int bhk = static_cast<int>(blockIdx.x) % BHkv;
  const int b = bhk / Hkv, hk = bhk % Hkv;
  const int g = Hq / Hkv;
  const int i0 = causal ? j : 0;                 // first Q tile that sees key tile j
  const int per_head = nq - i0;
  const int n_iter = g * per_head;               // >= 1
  if (j >= nk) return;
  if (!bwd_prologue(bb, status)) return;
  const uint32_t tmem = *bb.tmem_slot;
  // Tile slots: K, V, Q[2], dO[2].
  constexpr int TK = 0, TV = 1, TQ = 2, TDO = 4;
  auto tile = [&](int t) { return smem + t * C::TILE_BYTES; };
  auto wait = [&](uint64_t* bar, int phase_count) {
    return mbar_wait(bar, static_cast<uint32_t>(phase_count) & 1u, bb.abort_flag, kWaitLimitNs);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(&bb.kv_full[0], 2 * C::TILE_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_3d(tile(TK) + kb * C::BLOCK_BYTES, &tm_k, &bb.kv_full[0], kb * 64, j * T, bhk);
        tma_load_3d(tile(TV) + kb * C::BLOCK_BYTES, &tm_v, &bb.kv_full[0], kb * 64, j * T, bhk);
      }
      bool ok = true;
      int issued = 0;
      for (int n = 0; n < n_iter; ++n) {
        const int st = n & 1;
        if (n >= 2 && !wait(&bb.q_empty[st], (n >> 1) - 1)) { ok = false; break; }
        const int bhq = b * Hq + hk * g + n / per_head;
        const int i = i0 + n % per_head;
        mbar_arrive_expect_tx(&bb.q_full[st], 2 * C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(tile(TQ + st) + kb * C::BLOCK_BYTES, &tm_q, &bb.q_full[st], kb * 64, i * T, bhq);
          tma_load_3d(tile(TDO + st) + kb * C::BLOCK_BYTES, &tm_do, &bb.q_full[st], kb * 64, i * T,
                      bhq);
        }
        issued = n + 1;
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      int no_abort = 0;
      mbar_wait(&bb.kv_full[0], 0, &no_abort, kWaitLimitNs);
      for (int n = issued > 2 ? issued - 2 : 0; n < issued; ++n)
        mbar_wait(&bb.q_full[n & 1], (n >> 1) & 1, &no_abort, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint64_t k_desc = smem_desc_sw128(sbase + TK * C::TILE_BYTES, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sbase + TV * C::TILE_BYTES, 16, 1024);
      bool ok = wait(&bb.kv_full[0], 0);
      for (int n = 0; ok && n < n_iter; ++n) {
        const int st = n & 1;
        const uint32_t q_addr = sbase + (TQ + st) * C::TILE_BYTES;
        const uint32_t do_addr = sbase + (TDO + st) * C::TILE_BYTES;
        if (!wait(&bb.q_full[st], n >> 1)) { ok = false; break; }
        tc_fence_after();
        // S^T = K Q^T, then dP^T = V dO^T (keys as rows), query half by half:
        // columns h * 64.. of S^T and dP^T.
        const uint64_t q_k = smem_desc_sw128(q_addr, 16, 1024);
        const uint64_t do_k = smem_desc_sw128(do_addr, 16, 1024);
        for (int hh = 0; hh < 2; ++hh) {
          mma_kmajor_half<D>(tmem + C::S_COL + hh * H, k_desc, q_k + hh * kHalfStep);
          mma_commit(&bb.s_full[hh]);
        }
        for (int hh = 0; hh < 2; ++hh) {
          mma_kmajor_half<D>(tmem + C::DP_COL + hh * H, v_desc, do_k + hh * kHalfStep);
          mma_commit(&bb.dp_full[hh]);
        }
        // dV += P^T dO, half by half as P^T arrives (P^T of half h in
        // columns h * 32.. as bf16 pairs; dO rows h * 64..).
        const uint64_t do_mn = smem_desc_sw128(do_addr, C::BLOCK_BYTES, 1024);
        const uint64_t q_mn = smem_desc_sw128(q_addr, C::BLOCK_BYTES, 1024);
        for (int hh = 0; ok && hh < 2; ++hh) {
          if (!wait(&bb.p_ready[hh], n)) { ok = false; break; }
          tc_fence_after();
          mma_tmem_a_half<D>(tmem + C::ACC1_COL, tmem + C::S_COL + hh * (H / 2),
                             do_mn + hh * kHalfStep, n > 0 || hh > 0);
        }
        // dK += dS^T Q, half by half as dS^T arrives.
        for (int hh = 0; ok && hh < 2; ++hh) {
          if (!wait(&bb.ds_ready[hh], n)) { ok = false; break; }
          tc_fence_after();
          mma_tmem_a_half<D>(tmem + C::ACC0_COL, tmem + C::DP_COL + hh * (H / 2),
                             q_mn + hh * kHalfStep, n > 0 || hh > 0);
        }
        if (!ok) break;
        mma_commit(&bb.q_empty[st]);  // Q and dO of this stage may be refilled
      }
      if (ok) mma_commit(bb.acc_done);
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
    const int quad = warp & 3;
    const int c = quad * 32 + lane;               // key row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float scale_log2 = scale * attn::kLog2e;
    const int kk = j * T + c;                      // this thread's key
    // Per-query values of iteration n for query column c (this thread
    // stages one of the 128), negated for the packed FMAs: -LSE in the log2
    // domain (-inf where the query row does not exist or sees no key, so
    // that P = 0) and -D.
    auto fetch = [&](int n, float& l2, float& dv_) {
      l2 = -INFINITY;
      dv_ = 0.f;
      if (n < n_iter) {
        const int bhq = b * Hq + hk * g + n / per_head;
        const int row = (i0 + n % per_head) * T + c;
        if (row < Lq) {
          const float x = lse[static_cast<size_t>(bhq) * Lq + row];
          if (x != -INFINITY) l2 = -x * attn::kLog2e;
          dv_ = -dd[static_cast<size_t>(bhq) * Lq + row];
        }
      }
    };
    float pre_l2, pre_d;
    fetch(0, pre_l2, pre_d);
    bool ok = true;
    for (int n = 0; n < n_iter; ++n) {
      const int st = n & 1;
      float* l2s = vec + st * 2 * T;
      float* ds_ = l2s + T;
      // Every warp writes its 32 values, then waits for the other three
      // (an mbarrier, so the wait stays bounded).  A warp's arrival for n
      // follows its last read of stage n - 1, so once all four have arrived
      // for n, stage (n + 1) & 1 may be overwritten.
      l2s[c] = pre_l2;
      ds_[c] = pre_d;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb.vec_full[st]);
      ok = __all_sync(FULL, wait(&bb.vec_full[st], n >> 1));
      if (!ok) break;
      fetch(n + 1, pre_l2, pre_d);
      const int i = i0 + n % per_head;
      const bool diag = causal && i == j;          // keys past the query are masked here
      // P^T row c, query half by half: P[r] = 2^(S^T[c][r] scale log2e -
      // LSE_r log2e) as bf16 pairs, written to columns h * 32.. (over S^T
      // columns this thread has already read).
      uint32_t pw[64];
      for (int hh = 0; ok && hh < 2; ++hh) {
        ok = __all_sync(FULL, wait(&bb.s_full[hh], n));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32(tmem + lane_off + C::S_COL + hh * H, sr[0]);
        tmem_ld32(tmem + lane_off + C::S_COL + hh * H + 32, sr[1]);
        tmem_ld_wait();
        const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
        for (int e = 0; e < H; e += 4) {
          const int r = hh * H + e;
          const float4 nl = *reinterpret_cast<const float4*>(&l2s[r]);
          float2 pa = ffma2(make_float2(__uint_as_float(sr[e >> 5][e & 31]),
                                        __uint_as_float(sr[e >> 5][(e & 31) + 1])),
                            sc2, make_float2(nl.x, nl.y));
          float2 pb = ffma2(make_float2(__uint_as_float(sr[e >> 5][(e & 31) + 2]),
                                        __uint_as_float(sr[e >> 5][(e & 31) + 3])),
                            sc2, make_float2(nl.z, nl.w));
          pa.x = ex2(pa.x);
          pa.y = ex2(pa.y);
          pb.x = ex2(pb.x);
          pb.y = ex2(pb.y);
          if (diag) {
            if (kk > i * T + r) pa.x = 0.f;
            if (kk > i * T + r + 1) pa.y = 0.f;
            if (kk > i * T + r + 2) pb.x = 0.f;
            if (kk > i * T + r + 3) pb.y = 0.f;
          }
          pw[r >> 1] = attn::pack_bf16x2(pa.x, pa.y);
          pw[(r >> 1) + 1] = attn::pack_bf16x2(pb.x, pb.y);
        }
        tmem_st32(tmem + lane_off + C::S_COL + hh * (H / 2),
                  *reinterpret_cast<uint32_t(*)[32]>(&pw[hh * 32]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.p_ready[hh]);
      }
      if (!ok) break;
      // dS^T row c: dS[r] = P[r] (dP^T[c][r] - D_r), with P as handed to the
      // MMA, written over dP^T columns this thread has already read.
      for (int hh = 0; ok && hh < 2; ++hh) {
        ok = __all_sync(FULL, wait(&bb.dp_full[hh], n));
        if (!ok) break;
        tc_fence_after();
        uint32_t dr[2][32];
        tmem_ld32(tmem + lane_off + C::DP_COL + hh * H, dr[0]);
        tmem_ld32(tmem + lane_off + C::DP_COL + hh * H + 32, dr[1]);
        tmem_ld_wait();
        uint32_t sw[32];
        const float2 zero2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < H; e += 4) {
          const int r = hh * H + e;
          const float4 nd = *reinterpret_cast<const float4*>(&ds_[r]);
          const float2 xa = fadd2(make_float2(__uint_as_float(dr[e >> 5][e & 31]),
                                              __uint_as_float(dr[e >> 5][(e & 31) + 1])),
                                  make_float2(nd.x, nd.y));
          const float2 xb = fadd2(make_float2(__uint_as_float(dr[e >> 5][(e & 31) + 2]),
                                              __uint_as_float(dr[e >> 5][(e & 31) + 3])),
                                  make_float2(nd.z, nd.w));
          const uint32_t p0 = pw[r >> 1], p1 = pw[(r >> 1) + 1];
          const float2 sa = ffma2(make_float2(attn::bf16_lo(p0), attn::bf16_hi(p0)), xa, zero2);
          const float2 sb = ffma2(make_float2(attn::bf16_lo(p1), attn::bf16_hi(p1)), xb, zero2);
          sw[e >> 1] = attn::pack_bf16x2(sa.x, sa.y);
          sw[(e >> 1) + 1] = attn::pack_bf16x2(sb.x, sb.y);
        }
        tmem_st32(tmem + lane_off + C::DP_COL + hh * (H / 2), sw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.ds_ready[hh]);
      }
      if (!ok) break;
    }
    if (ok) ok = __all_sync(FULL, wait(bb.acc_done, 0));
    if (ok) {
      tc_fence_after();
      const bool live = kk < Lk;
      const size_t out_row = (static_cast<size_t>(bhk) * Lk + (live ? kk : 0)) * D;
      store_row_bf16<D>(tmem + lane_off + C::ACC0_COL, scale, dk + out_row, live);
      store_row_bf16<D>(tmem + lane_off + C::ACC1_COL, 1.f, dv + out_row, live);
    } else {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *bb.abort_flag = 1;
    }
  }
  bwd_epilogue(bb);
}

}  // namespace

namespace {

// dQ of one Q tile i of one (request, query head): the K/V tiles it sees
// stream through a two-stage ring.
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                  const float* __restrict__ dd, __nv_bfloat16* __restrict__ dq, int B, int Hq,
                  int Hkv, int Lq, int Lk, int causal, float scale, int* status) {
  using C = BwdCfg<D>;
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const BwdBars bb = carve_bars(smem + L::OFF_BAR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (Lk + T - 1) / T, nq = (Lq + T - 1) / T;
  const int BHq = B * Hq;
  // Heaviest first under the causal rule: the last Q tiles of every head first.
  const int i = nq - 1 - static_cast<int>(blockIdx.x) / BHq;
  const int bhq = static_cast<int>(blockIdx.x) % BHq;
  const int b = bhq / Hq, h = bhq % Hq;
  const int bhk = b * Hkv + h / (Hq / Hkv);
  const int n_iter = causal ? min(nk, i + 1) : nk;  // K/V tiles this Q tile sees
  if (i < 0) return;
  if (!bwd_prologue(bb, status)) return;
  const uint32_t tmem = *bb.tmem_slot;
  // Tile slots: Q, dO, K[2], V[2].
  constexpr int TQ = 0, TDO = 1, TK = 2, TV = 4;
  auto tile = [&](int t) { return smem + t * C::TILE_BYTES; };
  auto wait = [&](uint64_t* bar, int phase_count) {
    return mbar_wait(bar, static_cast<uint32_t>(phase_count) & 1u, bb.abort_flag, kWaitLimitNs);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(&bb.q_full[0], 2 * C::TILE_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_3d(tile(TQ) + kb * C::BLOCK_BYTES, &tm_q, &bb.q_full[0], kb * 64, i * T, bhq);
        tma_load_3d(tile(TDO) + kb * C::BLOCK_BYTES, &tm_do, &bb.q_full[0], kb * 64, i * T, bhq);
      }
      bool ok = true;
      int issued = 0;
      for (int jt = 0; jt < n_iter; ++jt) {
        const int st = jt & 1;
        if (jt >= 2 && !wait(&bb.kv_empty[st], (jt >> 1) - 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bb.kv_full[st], 2 * C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(tile(TK + st) + kb * C::BLOCK_BYTES, &tm_k, &bb.kv_full[st], kb * 64, jt * T, bhk);
          tma_load_3d(tile(TV + st) + kb * C::BLOCK_BYTES, &tm_v, &bb.kv_full[st], kb * 64, jt * T, bhk);
        }
        issued = jt + 1;
      }
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *bb.abort_flag = 1;
      }
      int no_abort = 0;
      mbar_wait(&bb.q_full[0], 0, &no_abort, kWaitLimitNs);
      for (int jt = issued > 2 ? issued - 2 : 0; jt < issued; ++jt)
        mbar_wait(&bb.kv_full[jt & 1], (jt >> 1) & 1, &no_abort, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint64_t q_desc = smem_desc_sw128(sbase + TQ * C::TILE_BYTES, 16, 1024);
      const uint64_t do_desc = smem_desc_sw128(sbase + TDO * C::TILE_BYTES, 16, 1024);
      bool ok = wait(&bb.q_full[0], 0);
      for (int jt = 0; ok && jt < n_iter; ++jt) {
        const int st = jt & 1;
        const uint32_t k_addr = sbase + (TK + st) * C::TILE_BYTES;
        const uint32_t v_addr = sbase + (TV + st) * C::TILE_BYTES;
        if (!wait(&bb.kv_full[st], jt >> 1)) { ok = false; break; }
        tc_fence_after();
        // S = Q K^T and dP = dO V^T (queries as rows), key half by half:
        // columns h * 64.. of S and dP.
        const uint64_t k_k = smem_desc_sw128(k_addr, 16, 1024);
        const uint64_t v_k = smem_desc_sw128(v_addr, 16, 1024);
        for (int hh = 0; hh < 2; ++hh) {
          mma_kmajor_half<D>(tmem + C::S_COL + hh * H, q_desc, k_k + hh * kHalfStep);
          mma_commit(&bb.s_full[hh]);
          mma_kmajor_half<D>(tmem + C::DP_COL + hh * H, do_desc, v_k + hh * kHalfStep);
          mma_commit(&bb.dp_full[hh]);
        }
        // dQ += dS K, half by half as dS arrives (dS of half h in columns
        // DP_COL + h * 32.. as bf16 pairs; K rows h * 64..).
        const uint64_t k_mn = smem_desc_sw128(k_addr, C::BLOCK_BYTES, 1024);
        for (int hh = 0; ok && hh < 2; ++hh) {
          if (!wait(&bb.ds_ready[hh], jt)) { ok = false; break; }
          tc_fence_after();
          mma_tmem_a_half<D>(tmem + C::ACC0_COL, tmem + C::DP_COL + hh * (H / 2),
                             k_mn + hh * kHalfStep, jt > 0 || hh > 0);
        }
        if (!ok) break;
        mma_commit(&bb.kv_empty[st]);  // K and V of this stage may be refilled
      }
      if (ok) mma_commit(bb.acc_done);
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
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float scale_log2 = scale * attn::kLog2e;
    const int qrow = i * T + r;
    const bool live = qrow < Lq;
    float l2 = INFINITY, drow = 0.f;             // +inf: a row that does not exist has P = 0
    if (live) {
      const float x = lse[static_cast<size_t>(bhq) * Lq + qrow];
      if (x != -INFINITY) l2 = x * attn::kLog2e;
      drow = dd[static_cast<size_t>(bhq) * Lq + qrow];
    }
    bool ok = true;
    for (int jt = 0; ok && jt < n_iter; ++jt) {
      // Keys past Lk, and past the query under the causal rule, get P = 0.
      const int kmax = causal ? min(Lk - 1, qrow) : Lk - 1;
      for (int hh = 0; ok && hh < 2; ++hh) {
        ok = __all_sync(FULL, wait(&bb.s_full[hh], jt)) &&
             __all_sync(FULL, wait(&bb.dp_full[hh], jt));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[2][32], dr[2][32];
        tmem_ld32(tmem + lane_off + C::S_COL + hh * H, sr[0]);
        tmem_ld32(tmem + lane_off + C::S_COL + hh * H + 32, sr[1]);
        tmem_ld32(tmem + lane_off + C::DP_COL + hh * H, dr[0]);
        tmem_ld32(tmem + lane_off + C::DP_COL + hh * H + 32, dr[1]);
        tmem_ld_wait();
        uint32_t sw[32];
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nl2 = make_float2(-l2, -l2), nd2 = make_float2(-drow, -drow);
        const float2 zero2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < H; e += 2) {
          const int key = jt * T + hh * H + e;
          float2 p = ffma2(make_float2(__uint_as_float(sr[e >> 5][e & 31]),
                                       __uint_as_float(sr[e >> 5][(e & 31) + 1])),
                           sc2, nl2);
          p.x = key > kmax ? 0.f : ex2(p.x);
          p.y = key + 1 > kmax ? 0.f : ex2(p.y);
          // P is rounded to bf16 as in the forward's P V product and in bwd_dkdv.
          const uint32_t pw = attn::pack_bf16x2(p.x, p.y);
          const float2 x = fadd2(make_float2(__uint_as_float(dr[e >> 5][e & 31]),
                                             __uint_as_float(dr[e >> 5][(e & 31) + 1])),
                                 nd2);
          const float2 ds2 = ffma2(make_float2(attn::bf16_lo(pw), attn::bf16_hi(pw)), x, zero2);
          sw[e >> 1] = attn::pack_bf16x2(ds2.x, ds2.y);
        }
        // Over dP columns this thread has already read (half 1 lands on
        // half 0's dP columns).
        tmem_st32(tmem + lane_off + C::DP_COL + hh * (H / 2), sw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb.ds_ready[hh]);
      }
    }
    if (ok) ok = __all_sync(FULL, wait(bb.acc_done, 0));
    if (ok) {
      tc_fence_after();
      const size_t out_row = (static_cast<size_t>(bhq) * Lq + (live ? qrow : 0)) * D;
      store_row_bf16<D>(tmem + lane_off + C::ACC0_COL, scale, dq + out_row, live);
    } else {
      if (lane == 0) attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
      *bb.abort_flag = 1;
    }
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
  using L = BwdSmem<D>;
  static bool attr_set[64] = {};  // per device: kernel attributes are per device
  const int dev = attn_host::current_device_slot();
  if (dev < 0) return ATTN_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_rows(&mq, q, D, Lq, B * Hq) || !make_map_rows(&mk, k, D, Lk, B * Hkv) ||
      !make_map_rows(&mv, v, D, Lk, B * Hkv) || !make_map_rows(&mdo, d_o, D, Lq, B * Hq))
    return ATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * Hq * Lq;
  const long long nq = (Lq + T - 1) / T, nk = (Lk + T - 1) / T;
  const long long dq_ctas = nq * B * Hq, dkdv_ctas = nk * B * Hkv;
  if ((rows + 7) / 8 > 0x7fffffffLL || dq_ctas > 0x7fffffffLL || dkdv_ctas > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  int* status = attn_host::device_status_ptr();
  bwd_rowdot_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), dd, rows, D);
  bwd_dkdv_kernel<D><<<static_cast<unsigned>(dkdv_ctas), THREADS, L::BYTES, stream>>>(
      mq, mk, mv, mdo, lse, dd, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
      B, Hq, Hkv, Lq, Lk, causal, scale, status);
  bwd_dq_kernel<D><<<static_cast<unsigned>(dq_ctas), THREADS, L::BYTES, stream>>>(
      mq, mk, mv, mdo, lse, dd, static_cast<__nv_bfloat16*>(dq), B, Hq, Hkv, Lq, Lk, causal,
      scale, status);
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
