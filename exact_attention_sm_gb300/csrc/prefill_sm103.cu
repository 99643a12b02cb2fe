// Fused exact-attention prefill for sm_103a: TMA + tcgen05 MMAs into tensor
// memory (TMEM), warp-specialised.
//
// The method ("10.3 FlashAttention: IO-aware algorithm design", 10.3.2 tiled
// forward in FlashAttention-2 order; "FlashAttention tiling, online softmax
// and IO" blog, sections 03 and 06): a CTA owns one 128-row Q tile of one
// (batch, head) and streams 128-key K/V tiles; per tile
//   S = Q K^T (scaled), m_new = max(m, rowmax S), P = exp(S - m_new),
//   l = l e^(m - m_new) + rowsum P,  O~ = O~ e^(m - m_new) + P V,
// and finally O = O~ / l, LSE = m + ln l.  S and P never leave the SM.
//
// GB300 mapping (the pages' FlashAttention-4 section, 10.3.6, names the
// primitives; this layout is ours):
//   warp 0      TMA producer: Q once, then K_j / V_j into an NS-stage ring of
//               128-byte-swizzled shared-memory tiles (mbarrier full/empty).
//   warp 1      allocates 512 TMEM columns; one thread issues
//               S_j = Q K_j^T (M=128, N=128, K=d) into TMEM buffer j%2, then
//               O += P_{j-1} V_{j-1} (M=128, N=d, K=128) into the TMEM O tile.
//   warps 2..5  softmax: thread r owns query row r (TMEM lane r); reads S_j
//               with tcgen05.ld, masks, keeps (m, l) in registers, writes P_j
//               as bf16 into a swizzled shared tile, rescales O in TMEM when
//               needed, and finally writes O / l and the LSE.
// QK^T of tile j+1 and PV of tile j-1 run on the tensor core while the
// softmax of tile j runs.  Scores are kept in the base-2 domain with
// log2(e) folded into the scale (exp2 on the MUFU unit).
//
// Conditional rescale (the lecture's FlashAttention-4 notes; its threshold is
// not given there): the running max m used for the exponentials is only
// raised when a tile's max exceeds it by more than 8 (base 2).  Otherwise the
// stale m is kept, P <= 2^8, and since l and O~ are scaled by the same m the
// result O~ / l and LSE = m + log2 l are unchanged.
//
// Causal: Q tile i reads K/V tiles 0..i only (tiles above the diagonal are
// skipped); the diagonal tile is masked element-wise; keys past Lk are
// masked in the last tile.  CTAs are ordered heaviest-first.
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

constexpr int BM = 128;               // query rows per CTA (MMA M)
constexpr int BN = 128;               // keys per K/V tile
constexpr int NUM_THREADS = 192;      // 6 warps
constexpr uint32_t TMEM_COLS = 512;   // S double buffer (2 x 128) + O (d)
constexpr uint32_t O_COL = 2 * BN;    // first TMEM column of the O accumulator
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                 // 128-byte swizzle column blocks per row
  static constexpr int BLOCK_BYTES = BM * 128;      // one 128-row x 128-byte column block
  static constexpr int TILE_BYTES = BM * D * 2;     // a Q, K or V tile
  static constexpr int NS = D == 64 ? 4 : 2;        // K/V pipeline stages
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_P = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // barriers + alignment slack
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
                        float* __restrict__ lse, int Hq, int Hkv, int Lq, int Lk, int causal,
                        float scale_log2, int* status) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NS;
  uint64_t* kv_empty = v_full + NS;
  uint64_t* s_full = kv_empty + NS;  // [2]
  uint64_t* s_free = s_full + 2;     // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int h = bh % Hq, b = bh / Hq;
  const int bh_kv = b * Hkv + h / (Hq / Hkv);
  const int qt = gridDim.y - 1 - blockIdx.y;  // heaviest Q tiles first
  const int n_kv = (Lk + BN - 1) / BN;
  const int n_tiles = causal ? min(n_kv, qt + 1) : n_kv;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    // After a timeout anywhere on the device the remaining CTAs do no work
    // until the host has read (and cleared) the status word.
    *abort_flag = (status != nullptr &&
                   *reinterpret_cast<volatile int*>(status) == ATTN_ERR_DEVICE_TIMEOUT) ? 2 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (*abort_flag == 2) return;
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(smem + C::OFF_Q + kb * C::BLOCK_BYTES, &tm_q, q_full, kb * 64, qt * BM, bh);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NS;
        if (j >= NS && !mbar_wait(&kv_empty[st], ((j / NS) + 1) & 1, abort_flag, kWaitLimitNs)) {
          attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* kdst = smem + C::OFF_K + st * C::TILE_BYTES;
        uint8_t* vdst = smem + C::OFF_V + st * C::TILE_BYTES;
        mbar_arrive_expect_tx(&k_full[st], C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(kdst + kb * C::BLOCK_BYTES, &tm_k, &k_full[st], kb * 64, j * BN, bh_kv);
        mbar_arrive_expect_tx(&v_full[st], C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(vdst + kb * C::BLOCK_BYTES, &tm_v, &v_full[st], kb * 64, j * BN, bh_kv);
        issued = j + 1;
      }
      // Drain: every issued copy has landed before the CTA may exit (these
      // waits ignore the abort flag; TMA copies always complete).
      int no_abort = 0;
      mbar_wait(q_full, 0, &no_abort, kWaitLimitNs);
      for (int j = issued > NS ? issued - NS : 0; j < issued; ++j) {
        mbar_wait(&k_full[j % NS], (j / NS) & 1, &no_abort, kWaitLimitNs);
        mbar_wait(&v_full[j % NS], (j / NS) & 1, &no_abort, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      const uint32_t q_addr = sbase + C::OFF_Q;
      const uint32_t p_addr = sbase + C::OFF_P;
      bool ok = mbar_wait(q_full, 0, abort_flag, kWaitLimitNs);

      auto issue_pv = [&](int i) -> bool {
        const int st = i % NS;
        if (!mbar_wait(p_full, i & 1, abort_flag, kWaitLimitNs)) return false;
        if (!mbar_wait(&v_full[st], (i / NS) & 1, abort_flag, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t v_addr = sbase + C::OFF_V + st * C::TILE_BYTES;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          // A = P: K-major, 16 keys per step inside a 64-key swizzle block.
          const uint64_t a = smem_desc_sw128(p_addr + (k >> 2) * C::BLOCK_BYTES + (k & 3) * 32, 16, 1024);
          // B = V: MN-major (d contiguous); 16 keys = 2 eight-row groups of
          // 128 bytes; LBO steps to the next 64-column block of d.
          const uint64_t bd = smem_desc_sw128(v_addr + k * 16 * 128, C::BLOCK_BYTES, 1024);
          mma_bf16_ss(tmem + O_COL, a, bd, idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&kv_empty[st]);
        return true;
      };

      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % NS, sb = j & 1;
        if (!mbar_wait(&k_full[st], (j / NS) & 1, abort_flag, kWaitLimitNs)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&s_free[sb], ((j - 2) >> 1) & 1, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = sbase + C::OFF_K + st * C::TILE_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * C::BLOCK_BYTES + (k & 3) * 32;
          const uint64_t a = smem_desc_sw128(q_addr + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(k_addr + off, 16, 1024);
          mma_bf16_ss(tmem + sb * BN, a, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[sb]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && n_tiles > 0) ok = issue_pv(n_tiles - 1);
      if (!ok) {
        attn::record_status(status, ATTN_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: all MMAs issued by this thread are complete before teardown.
      int no_abort = 0;
      mma_commit(drain);
      mbar_wait(drain, 0, &no_abort, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const int grow = qt * BM + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float m_s = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + sb * BN + c * 32, sr[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s_free[sb]);

      float* s = reinterpret_cast<float*>(&sr[0][0]);
      const bool need_mask = (j == n_tiles - 1) && (causal || (Lk % BN) != 0);
      float mt = -INFINITY;
      if (need_mask) {
        const int kmax = causal ? min(Lk - 1, grow) : Lk - 1;  // last visible key
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          if (j * BN + c > kmax) s[c] = -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) mt = fmaxf(mt, s[c]);
      }
      const float mt_s = mt * scale_log2;
      float alpha = 1.f;
      if (mt_s > m_s + kRescaleThreshold) {
        alpha = ex2(m_s - mt_s);  // 0 on the first tile (m_s = -inf)
        m_s = mt_s;
      }
      const float neg_m = -m_s;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        s[c] = ex2(fmaf(s[c], scale_log2, neg_m));
        s[c + 1] = ex2(fmaf(s[c + 1], scale_log2, neg_m));
        rs0 += s[c];
        rs1 += s[c + 1];
      }
      l = l * alpha + (rs0 + rs1);

      if (j > 0) {
        // PV of the previous tile must be done: P's buffer is free, O is stable.
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + O_COL + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(lane_base + O_COL + c * 32, r);
          }
          tmem_st_wait();
        }
      }
      // P (bf16) into the 128-byte-swizzled K-major tile: row r, 16-byte
      // chunk c of a 64-key block lands at chunk c ^ (r % 8).
      uint8_t* prow = smem + C::OFF_P + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const int k0 = kb * 64 + c16 * 8;
          uint4 w;
          w.x = attn::pack_bf16x2(s[k0], s[k0 + 1]);
          w.y = attn::pack_bf16x2(s[k0 + 2], s[k0 + 3]);
          w.z = attn::pack_bf16x2(s[k0 + 4], s[k0 + 5]);
          w.w = attn::pack_bf16x2(s[k0 + 6], s[k0 + 7]);
          *reinterpret_cast<uint4*>(prow + kb * C::BLOCK_BYTES + ((c16 ^ (row & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }

    if (ok) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(o_done, (n_tiles - 1) & 1, abort_flag, kWaitLimitNs));
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool live = grow < Lq;
      __nv_bfloat16* orow = o + (static_cast<size_t>(bh) * Lq + (live ? grow : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + O_COL + c * 32, r);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            uint4 w;
            w.x = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 0]) * inv, __uint_as_float(r[v8 * 8 + 1]) * inv);
            w.y = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 2]) * inv, __uint_as_float(r[v8 * 8 + 3]) * inv);
            w.z = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 4]) * inv, __uint_as_float(r[v8 * 8 + 5]) * inv);
            w.w = attn::pack_bf16x2(__uint_as_float(r[v8 * 8 + 6]) * inv, __uint_as_float(r[v8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + v8 * 8) = w;
          }
        }
      }
      if (live && lse != nullptr)
        lse[static_cast<size_t>(bh) * Lq + grow] =
            l > 0.f ? (m_s + log2f(l)) * attn::kLn2 : -INFINITY;
    } else {
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

// [rows = L, BH heads] x d bf16 viewed as a 3-D tensor {d, L, BH}; box
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

template <int D>
attn_status_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                     int Hkv, int Lq, int Lk, int causal, float scale, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(prefill_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set = true;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, D, Lq, B * Hq) || !make_map(&mk, k, D, Lk, B * Hkv) ||
      !make_map(&mv, v, D, Lk, B * Hkv))
    return ATTN_ERR_CUDA;
  const int num_qt = (Lq + BM - 1) / BM;
  if (num_qt > 65535) return ATTN_ERR_UNSUPPORTED;
  dim3 grid(B * Hq, num_qt);
  prefill_bf16_kernel<D><<<grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(o), lse, Hq, Hkv, Lq, Lk, causal,
      scale * attn::kLog2e, attn_host::device_status_ptr());
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

attn_status_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                  float scale, cudaStream_t stream) {
  if (d == 64) return launch<64>(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, causal, scale, stream);
  if (d == 128) return launch<128>(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, causal, scale, stream);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn_host
