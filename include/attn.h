/*
 * attn.h - C ABI of the GB300 (sm_103a) exact-attention library (libattn.so).
 *
 * Exact scaled-dot-product attention O = softmax(Q K^T * scale) V, computed
 * as fused kernels that never write the L x L score matrix to device memory,
 * plus its memory-bound decode form over a paged, grouped-query KV cache and
 * the LSE merge operator that combines split-KV partial states.
 *
 * Pages the operations follow (cited by title below):
 *   [Lecture 4]   "Lecture 4 - Efficient attention kernels: FlashAttention and
 *                 FlashInfer" (Stanford CS349D course notes)
 *   [Tiling blog] "The attention formula did not change, so why is it several
 *                 times faster? FlashAttention's tiling, online softmax and IO"
 *   [LLM book]    "10.3 FlashAttention: IO-aware algorithm design"
 *   [CUDA book]   "FlashAttention and inference operators" (CUDA advanced
 *                 handbook)
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer to a dense, row-major
 *     (contiguous) array in the layout stated per call; the caller allocates,
 *     owns and frees all of them, including any workspace.  The library never
 *     allocates or frees device memory and keeps no per-call state.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on it and returns; results are valid once the
 *     stream has synchronised.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a status and touches no memory.  A launch failure
 *     returns ATTN_ERR_CUDA.  Problems found on the device (a block-table
 *     entry outside [0, num_pages), a bounded wait that ran out) do not fault:
 *     the kernel skips the access, records the error in a device status word
 *     and the next attn_get_device_status() call reports it.
 *   - dtype ATTN_BF16: bf16 inputs and outputs, fp32 accumulation, fp32 LSE.
 *     dtype ATTN_F32: fp32 everywhere (computed on CUDA cores in fp32).
 *   - LSE is the natural-log log-sum-exp of the scaled scores of a row,
 *     LSE = m + ln(l) ([LLM book] 10.3.2 "LSE").  A row that sees no key gets
 *     O = 0 and LSE = -inf (never NaN).
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* == cudaStream_t */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null pointer, size <= 0, Hq % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2,    /* valid but not implemented (d, page size, causal Lq != Lk) */
  ATTN_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  ATTN_ERR_CUDA = 4,           /* a CUDA runtime call or a launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out (device status) */
  ATTN_ERR_BAD_INDEX = 6       /* a block-table entry was out of range (device status) */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/*
 * attn_fwd - fused prefill attention forward with per-row LSE.
 *
 * Computes, for every batch b and query head h (KV head h / (Hq / Hkv),
 * [CUDA book] GQA exercise):
 *   S = Q_bh K_b,kvh^T * scale, P = softmax(S), O_bh = P V_b,kvh
 * ([Tiling blog] section 01), row by row with the online softmax over K/V
 * tiles ([LLM book] 10.3.2 tiled forward, FlashAttention-2 order).  With
 * causal != 0 query i sees key j only when j <= i; K/V tiles entirely above
 * the diagonal are skipped and diagonal tiles are masked element-wise
 * ([Tiling blog] section 06).
 *
 *   q   [B, Hq,  Lq, d]   input, dtype
 *   k   [B, Hkv, Lk, d]   input, dtype
 *   v   [B, Hkv, Lk, d]   input, dtype
 *   o   [B, Hq,  Lq, d]   output, dtype (written in full)
 *   lse [B, Hq,  Lq]      output, fp32, natural log; may be NULL
 *   d in {64, 128}; Hq % Hkv == 0; B, Hq, Hkv, Lq, Lk >= 1.
 *   causal requires Lq == Lk (ATTN_ERR_UNSUPPORTED otherwise).
 *   scale: usually 1/sqrt(d); must be finite and > 0.
 *   bf16 pointers must be 16-byte aligned (tensor-memory-access copies).
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                       attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_decode_plan - host-side split-KV planner (no device work).
 *
 * Chooses one chunk length C (a multiple of page_size) shared by every
 * request; request b is cut into max(1, ceil(len_b / C)) segments.
 * Reading of [Lecture 4] section 4.2 and exercise 6 (whose answer is the
 * finest split that still fits in one round of the SMs): a work unit is
 * (request, KV head, segment) and `slots` workers run one unit each at a
 * time.  C is the shortest multiple of page_size for which the non-empty
 * units Hkv * sum_b ceil(len_b / C) fit in `slots`; if even unsplit
 * requests do not fit, nothing is split.
 * num_splits > 0 forces C = ceil(ceil(max_len / num_splits) / page_size) *
 * page_size instead.  slots <= 0 means "ask the current device": SM count x
 * resident decode CTAs per SM.
 *
 *   seq_lens_host [B]  host array of context lengths (>= 0)
 *   chunk_out          host scalar: C
 *   max_splits_out     host scalar: max_b segments (the workspace's S)
 */
attn_status_t attn_decode_plan(const int32_t* seq_lens_host, int B, int Hkv, int page_size,
                               int num_splits, int slots, int32_t* chunk_out,
                               int32_t* max_splits_out);

/*
 * attn_decode_workspace_bytes - bytes of workspace attn_decode_paged needs
 * when the plan has `max_splits` segments per request (0 when max_splits
 * <= 1: the decode kernel then writes O and LSE directly).  Layout: fp32
 * partial outputs [B*Hq, max_splits, d] followed by fp32 partial LSE
 * [B*Hq, max_splits], 256-byte aligned.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_splits);

/*
 * attn_decode_paged - one query token per request against a paged KV cache.
 *
 * For request b and query head h (KV head h / (Hq / Hkv)) the keys are
 * tokens t < seq_lens[b]; token t lives in page block_table[b][t / page_size],
 * slot t % page_size ([CUDA book] "PagedAttention"; cache layout of
 * [LLM book] 10.3.7).  With more than one segment per request (split-KV,
 * Flash-Decoding: [LLM book] 10.3.7, [CUDA book] "Flash-Decoding and
 * split-K") each segment's normalised O_s and LSE_s go to the workspace and
 * are combined by the LSE merge (attn_merge_states) in a fixed order, so
 * results are bitwise reproducible.
 *
 *   q            [B, Hq, d]                          input, dtype
 *   k_pages      [num_pages, page_size, Hkv, d]      input, dtype
 *   v_pages      [num_pages, page_size, Hkv, d]      input, dtype
 *   block_table  [B, max_pages_per_seq] int32        input; entries at or past
 *                ceil(seq_lens[b] / page_size) are never read (may be -1)
 *   seq_lens     [B] int32 (device)                  input, 0 <= len <=
 *                max_pages_per_seq * page_size
 *   seq_lens_host [B] int32 (host) or NULL           lengths for the planner;
 *                when NULL and num_splits != 1 the library copies seq_lens
 *                to the host and synchronises `stream` first.
 *   page_size    16 (ATTN_ERR_UNSUPPORTED otherwise)
 *   num_splits   0 = planner's choice, >= 1 forces at most that many segments
 *   o            [B, Hq, d] output, dtype;  lse [B, Hq] fp32 output or NULL
 *   workspace    device buffer of >= attn_decode_workspace_bytes(B, Hq, d, S)
 *                bytes for the plan's S (may be NULL when S == 1)
 *   d in {64, 128} (bf16 only).
 */
attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const int32_t* seq_lens_host, int page_size, int num_splits,
                                void* o, float* lse, int B, int Hq, int Hkv, int d,
                                int max_pages_per_seq, int num_pages, float scale,
                                void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                                attn_stream_t stream);

/*
 * attn_decode_paged_noalloc - attn_decode_paged for callers that cannot
 * allocate device memory.  No counterpart in the source pages: this is a
 * convenience of this library.
 *
 * Who needs it: code that is handed only its inputs and outputs and is not
 * allowed to call cudaMalloc or any other allocator - for example a plugin
 * inside a host framework that owns all device memory through its own pool,
 * or a latency-critical path where an allocation (and the device-wide
 * synchronisation cudaMalloc can imply) is not acceptable.  Such a caller
 * cannot provide the split-KV workspace that attn_decode_paged wants.
 *
 * Instead of a caller-provided workspace this call uses one fixed scratch
 * array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes that lives inside the
 * library as a static device variable: every GPU that loads libattn.so holds
 * it until the process exits.  The call itself allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 *
 *   Arguments are those of attn_decode_paged minus the workspace, with one
 *   difference: seq_lens_host must not be NULL unless num_splits == 1 (the
 *   split planner runs on the host and this call will not allocate a host
 *   copy either).
 *   Returns ATTN_ERR_WORKSPACE, touching no memory, when the plan needs more
 *   than ATTN_DECODE_NOALLOC_SCRATCH_BYTES (attn_decode_workspace_bytes(B,
 *   Hq, d, S) for the plan's S); use attn_decode_paged with your own
 *   workspace for such sizes.
 *   The first call on a device looks up the scratch array's device address
 *   (one cudaGetSymbolAddress per device, with that device current); make
 *   that first call before any stream capture.
 *   All calls on a device share the one scratch array, and it keeps whatever
 *   the last call wrote (every used entry is overwritten before it is read,
 *   so nothing needs clearing).  Calls whose kernels overlap on the GPU (on
 *   different streams, or from different host threads) race on that array:
 *   serialise them.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        const int32_t* seq_lens_host, int page_size,
                                        int num_splits, void* o, float* lse, int B, int Hq,
                                        int Hkv, int d, int max_pages_per_seq, int num_pages,
                                        float scale, attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_varlen - prefill over sequences packed end to end ("10.3
 * FlashAttention", 10.3.8 variable-length batching).
 *
 *   q  [total_q, Hq, d]  k, v [total_k, Hkv, d]  bf16, row-major, 16-byte
 *   aligned; o [total_q, Hq, d] bf16; lse [total_q, Hq] fp32 or NULL.
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1], cumulative lengths
 *   (lengths 3, 5, 2 -> [0, 3, 8, 10]); sequence b owns q rows
 *   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and k/v rows cu_seqlens_k[b] ..,
 *   and sees nothing of the other sequences.  max_seqlen_q / max_seqlen_k
 *   bound every length (they size the work list); total_q / total_k are the
 *   row counts of q and k.  GQA: query head h reads KV head h / (Hq / Hkv).
 *
 * Causal is aligned bottom-right (the pages define only the square case):
 * query i of a sequence with Lq queries and Lk keys sees key j <= i + Lk - Lq,
 * i.e. the queries are the last Lq tokens of the sequence (chunked prefill).
 * Rows that see no key (Lq > Lk) get O = 0, LSE = -inf.  Lengths may be 0;
 * total_q = 0 returns ATTN_OK without any launch (every pointer may be
 * NULL), and total_k = 0 (k, v may be NULL) gives every row O = 0,
 * LSE = -inf.
 *
 * d in {64, 128}, bf16 only.  Errors: ATTN_ERR_INVALID_ARG for NULLs, bad
 * sizes or misalignment; ATTN_ERR_UNSUPPORTED for other d or dtypes.  A
 * cu_seqlens entry that breaks its bounds (decreasing, past total, longer
 * than max_seqlen) is reported as ATTN_ERR_BAD_INDEX in the device status
 * word and that sequence is left unwritten; nothing outside the tensors is
 * touched.
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                              int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                              int Hkv, int d, int causal, float scale, attn_dtype_t dtype,
                              attn_stream_t stream);

/*
 * Load-balanced decode with a fixed grid ("Lecture 4" section 5.6: the
 * FlashInfer-style scheduler and its CUDA-graph workspace).
 *
 * attn_decode_schedule (host work plus one host-to-device copy into the
 * workspace; not inside a stream capture): with G = Hkv * ceil((Hq/Hkv) / 4)
 * head groups (a CTA serves up to 4 query heads of one KV head),
 *   L_kv = ceil(ceil(sum_b len_b * G / num_ctas) / page_size) * page_size,
 *   every (request, group) is cut into consecutive segments of at most L_kv
 *   tokens (a request of length 0 keeps one empty segment), and the segments
 *   are dealt longest first (ties in (request, group, segment) order) to the
 *   CTA with the least work so far (lowest index on ties).
 * attn_decode_paged_balanced: num_ctas persistent CTAs (the same grid for
 *   every plan of a given (B, Hq, Hkv, num_ctas)) walk their segments and
 *   write each as a normalised partial state; a merge kernel combines the
 *   segments of every output row in token order (bitwise reproducible).
 *   The plan is read from the workspace at run time, so one captured CUDA
 *   graph of this call replays correctly after attn_decode_schedule has
 *   written a new plan for new lengths.  Plan entries are checked on the
 *   device (ATTN_ERR_BAD_INDEX, entry skipped), and each segment is clamped
 *   to the device seq_lens and the block table's capacity.
 * attn_decode_schedule_host: the same plan into host memory (plan_ints
 *   >= the plan's int32 count), for inspection and tests.
 * attn_decode_sched_workspace_bytes: plan + partial states for (B, Hq, Hkv,
 *   d, num_ctas), 256-byte aligned.
 *
 *   num_ctas <= 0: SM count x resident CTAs per SM of the balanced kernel.
 *   Other arguments as attn_decode_paged (d = 128, page_size 16, bf16).
 *   Errors: ATTN_ERR_INVALID_ARG for NULLs, bad sizes, negative lengths or
 *   misalignment; ATTN_ERR_UNSUPPORTED for other d, page sizes or dtypes;
 *   ATTN_ERR_WORKSPACE if the workspace is missing, short or misaligned.
 */
size_t attn_decode_sched_workspace_bytes(int B, int Hq, int Hkv, int d, int num_ctas);
attn_status_t attn_decode_schedule(const int32_t* seq_lens_host, int B, int Hq, int Hkv,
                                   int page_size, int num_ctas, void* workspace,
                                   size_t workspace_bytes, attn_stream_t stream);
attn_status_t attn_decode_schedule_host(const int32_t* seq_lens_host, int B, int Hq, int Hkv,
                                        int page_size, int num_ctas, int32_t* plan_out,
                                        size_t plan_ints);
attn_status_t attn_decode_paged_balanced(const void* q, const void* k_pages, const void* v_pages,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int page_size, void* o, float* lse, int B, int Hq,
                                         int Hkv, int d, int max_pages_per_seq, int num_pages,
                                         float scale, int num_ctas, void* workspace,
                                         size_t workspace_bytes, attn_dtype_t dtype,
                                         attn_stream_t stream);

/*
 * attn_bwd - backward pass of attn_fwd (bf16), for training.
 *
 * "10.3 FlashAttention", backward and recomputation: from Q, K, V, the
 * forward's O and LSE, and the output gradient dO, the kernels rebuild
 * S = scale Q K^T and P = exp(S - LSE) tile by tile on chip and return
 *   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q
 * (dK, dV of a KV head sum over its Hq / Hkv query heads).  No L x L matrix
 * is stored.  Every gradient element is written by one CTA in a fixed
 * order (no atomics): results are bitwise reproducible.
 *
 *   q, o, d_o, dq  [B, Hq, Lq, d] bf16     k, v, dk, dv  [B, Hkv, Lk, d] bf16
 *   lse            [B, Hq, Lq] fp32 (natural log, as attn_fwd writes it)
 *   workspace      attn_bwd_workspace_bytes(B, Hq, Lq) bytes, 256-byte
 *                  aligned (holds -LSE log2e and -D per query row, padded to
 *                  128-row tiles, and the kernels' work counters, which the
 *                  call resets); device memory owned by the caller.
 *                  Calls that may run at the same time need separate
 *                  workspaces.
 *   causal requires Lq == Lk (square rule, as attn_fwd).
 * d in {64, 128}, bf16 only.  Errors: ATTN_ERR_INVALID_ARG for NULLs, bad
 * sizes or misalignment; ATTN_ERR_UNSUPPORTED for other d or dtypes or
 * causal with Lq != Lk; ATTN_ERR_WORKSPACE if the workspace is missing,
 * short or misaligned; device timeouts through the status word.
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Lq);
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* d_o, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                       void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                       attn_stream_t stream);

/*
 * attn_prefill_paged - chunked prefill of packed queries against a paged KV
 * cache ("Lecture 4" section 5.2: attention over KV in shuffled physical
 * blocks equals attention over the blocks gathered contiguously; "10.3
 * FlashAttention" 10.3.7 block-table addressing, 10.3.8 packing).
 *
 *   q [total_q, Hq, d] bf16 packed as in attn_fwd_varlen with
 *   cu_seqlens_q [B + 1] (DEVICE int32); o [total_q, Hq, d] bf16; lse
 *   [total_q, Hq] fp32 or NULL.
 *   k_pages, v_pages [num_pages, page_size, Hkv, d] bf16 (the decode cache
 *   layout at page_size 16); block_table [B, max_pages_per_seq] int32 and
 *   seq_lens_k [B] int32, both on the device: sequence b's keys are tokens
 *   0 .. seq_lens_k[b]-1, token t in page block_table[b][t / page_size],
 *   slot t % page_size.  Entries at or past ceil(seq_lens_k[b] / page_size)
 *   are never read.
 *   max_seqlen_q / max_seqlen_k bound the lengths (max_seqlen_k <=
 *   max_pages_per_seq * page_size).
 *   page_size: a power of two from 1 to 128.  16-token pages go to shared
 *   memory as one TMA copy each; other sizes are gathered row by row
 *   (slower: many 16-byte copies).
 *
 * Causal is aligned bottom-right as in attn_fwd_varlen: the chunk's queries
 * are the last Lq of the sequence's Lk tokens (their K/V already appended).
 * Slots of a sequence's last page past its length may hold anything: they
 * never reach the result.  d in {64, 128}, bf16.  total_q = 0 returns
 * ATTN_OK without a launch.  Errors: ATTN_ERR_INVALID_ARG for NULLs, bad
 * sizes or misalignment; ATTN_ERR_UNSUPPORTED for other d, page sizes or
 * dtypes.  On the device, a cu_seqlens_q entry or length out of bounds, or a
 * needed block-table entry outside [0, num_pages), is reported as
 * ATTN_ERR_BAD_INDEX (the sequence is skipped, or the page reads as zeros and
 * that sequence's rows are not meaningful); nothing outside the tensors is
 * read or written.
 */
attn_status_t attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens_k, void* o, float* lse, int B,
                                 int max_seqlen_q, int max_seqlen_k, int total_q, int Hq, int Hkv,
                                 int d, int page_size, int max_pages_per_seq, int num_pages,
                                 int causal, float scale, attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_prefill_bsr - prefill against a KV cache addressed in block-sparse
 * row (BSR) form ("Lecture 4" section 5.2, "block-sparse format: unifying
 * KV layouts"): the batch's "query rows x physical KV blocks" matrix is
 * block-sparse; kv_indices lists the non-zero blocks (physical block ids) of
 * every request end to end and request b's blocks, in logical order, are
 * kv_indices[kv_indptr[b] .. kv_indptr[b + 1]).  A vLLM page table is this
 * form with block_size 16, SGLang's radix tree with block_size 1 (the
 * lecture's exercise 9 (a)).
 *
 *   q [total_q, Hq, d] bf16 packed with cu_seqlens_q [B + 1]; o, lse as in
 *   attn_prefill_paged.
 *   k_blocks, v_blocks [num_blocks, block_size, Hkv, d] bf16.
 *   kv_indptr [B + 1], kv_indices [nnz], seq_lens_k [B]: int32 on the
 *   device.  Request b's keys are tokens 0 .. seq_lens_k[b]-1, token t in
 *   block kv_indices[kv_indptr[b] + t / block_size], slot t % block_size;
 *   kv_indptr[b + 1] - kv_indptr[b] >= ceil(seq_lens_k[b] / block_size).
 *   block_size: a power of two from 1 to 128 (16: one TMA copy per block;
 *   other sizes: row gathers into the same shared-memory tiles).
 *   Decode is the case of one query per request.
 *
 * Causal is aligned bottom-right (the request's queries are its last Lq
 * tokens).  d in {64, 128}, bf16.  Errors as attn_prefill_paged; on the
 * device, kv_indptr entries outside [0, nnz] or decreasing, too few blocks
 * for a length, and needed block ids outside [0, num_blocks) are reported as
 * ATTN_ERR_BAD_INDEX and never dereferenced.
 */
attn_status_t attn_prefill_bsr(const void* q, const void* k_blocks, const void* v_blocks,
                               const int32_t* kv_indptr, const int32_t* kv_indices, int nnz,
                               const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o,
                               float* lse, int B, int max_seqlen_q, int max_seqlen_k, int total_q,
                               int Hq, int Hkv, int d, int block_size, int num_blocks, int causal,
                               float scale, attn_dtype_t dtype, attn_stream_t stream);

/*
 * Cascade (shared-prefix) decode ([Lecture 4] 4.4 "cascade attention" and
 * 5.3 "composable formats").  B requests share one prefix of prefix_len
 * tokens, stored once as prefix_k / prefix_v [Hkv, prefix_len, d] bf16
 * (the dense (n, B_c) block of 5.3), and each has its own suffix in the
 * paged cache (k_pages, v_pages, block_table, seq_lens as in
 * attn_decode_paged; seq_lens holds the SUFFIX lengths, 0 allowed).  The
 * result equals decode over prefix + suffix as one sequence:
 *   1. the query rows of each KV head, from all B requests, are stacked into
 *      one (B * g) x d matrix (g = Hq / Hkv) and attend to the prefix ONCE,
 *      on the tensor cores (the prefill kernel; the prefix is cut into
 *      prefix_chunks chunks, each a divisor of prefix_len, for parallelism);
 *   2. each request attends to its own suffix (the paged decode kernel);
 *   3. the prefix-chunk and suffix states of every row are merged with the
 *      LSE operator in a fixed order (prefix chunks, then suffix segments).
 * The prefix is read once instead of B times ([Lecture 4] exercise 7).
 *
 * attn_cascade_plan: prefix_chunks = the chunk count c (a divisor of
 *   prefix_len with chunks of >= 128 tokens, or 1) minimising
 *   ceil(Hkv x ceil(B*g/256) x c / prefix_slots) x (2 + ceil(prefix_len/c/128)),
 *   the waves of prefill items times their K/V tiles plus a 2-tile per-item
 *   overhead; ties go to fewer chunks.  The suffix split plan is
 *   attn_decode_plan with suffix_slots.  prefix_slots <= 0 / suffix_slots <= 0 query the
 *   current device, as attn_decode_cascade does: half its SMs for the prefix
 *   pass (the suffix decode runs beside it on the other half) / its resident
 *   decode CTAs.
 * attn_cascade_workspace_bytes: bytes attn_decode_cascade needs for the plan
 *   (stacked queries, prefix-chunk states, suffix states), 256-byte aligned.
 * attn_decode_cascade: q [B, Hq, d], o [B, Hq, d] bf16, lse [B, Hq] fp32 or
 *   NULL.  d = 64 or 128, page_size = 16, bf16 only.  seq_lens_host (host copy of
 *   the suffix lengths) is required: it fixes the plan.  prefix_len >= 1.
 *   Pointers: device, 16-byte aligned (workspace 256-byte aligned), owned
 *   by the caller.  Errors: ATTN_ERR_INVALID_ARG for bad sizes, NULLs,
 *   misalignment or a suffix length outside [0, max_pages_per_seq * 16];
 *   ATTN_ERR_WORKSPACE if the workspace is missing, short or misaligned;
 *   ATTN_ERR_UNSUPPORTED for other d, page_size != 16 or non-bf16; device
 *   errors as attn_fwd / attn_decode_paged (status word).
 */
attn_status_t attn_cascade_plan(int B, int Hq, int Hkv, int prefix_len,
                                const int32_t* suffix_lens_host, int page_size, int num_splits,
                                int prefix_slots, int suffix_slots, int32_t* prefix_chunks_out,
                                int32_t* suffix_chunk_out, int32_t* suffix_splits_out);
size_t attn_cascade_workspace_bytes(int B, int Hq, int d, int prefix_chunks, int suffix_splits);
attn_status_t attn_decode_cascade(const void* q, const void* prefix_k, const void* prefix_v,
                                  int prefix_len, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const int32_t* seq_lens_host, int page_size, int num_splits,
                                  void* o, float* lse, int B, int Hq, int Hkv, int d,
                                  int max_pages_per_seq, int num_pages, float scale,
                                  void* workspace, size_t workspace_bytes, attn_dtype_t dtype,
                                  attn_stream_t stream);

/*
 * attn_merge_states - the LSE merge operator over S partial states per row.
 *
 * For each row r: M = max_s LSE[r,s] over non-empty states, w_s =
 * exp(LSE[r,s] - M), O[r] = sum_s w_s O_parts[r,s] / sum_s w_s,
 * LSE[r] = M + ln(sum_s w_s) ([LLM book] 10.3.2 "LSE"; [CUDA book]
 * "Flash-Decoding and split-K" and its merge exercise).  States with
 * LSE = -inf are skipped (their O is not read); a row whose states are all
 * empty gets O = 0, LSE = -inf.  The summation order is fixed by (S, d)
 * alone (states dealt round-robin to 4 warps, the warps then added in
 * order) and uses no atomics, so results are bitwise reproducible
 * ([Lecture 4] 4.3 and 5.6 on determinism).
 *
 *   o_parts   [rows, S, d] fp32 input     lse_parts [rows, S] fp32 input
 *   o_out     [rows, d] output in out_dtype   lse_out [rows] fp32 or NULL
 *   d % 4 == 0, 1 <= d <= 512, S >= 1.
 */
attn_status_t attn_merge_states(const float* o_parts, const float* lse_parts, int rows, int S,
                                int d, void* o_out, float* lse_out, attn_dtype_t out_dtype,
                                attn_stream_t stream);

/*
 * attn_get_device_status - waits for `stream`, then reads and clears the
 * device status word shared by all kernels of this library on the current
 * device.  Returns ATTN_OK, ATTN_ERR_BAD_INDEX or ATTN_ERR_DEVICE_TIMEOUT
 * (the first recorded), or ATTN_ERR_CUDA if the stream itself failed.
 */
attn_status_t attn_get_device_status(attn_stream_t stream);

/*
 * attn_selftest_wait_timeout - failure-detection self-test (no counterpart in
 * the pages).  Launches one thread that waits on an mbarrier nothing will
 * ever arrive at, using the same bounded wait as the pipelined attention
 * kernels, with a limit of `limit_ms` milliseconds (1..10000).  The wait
 * runs out, the kernel records ATTN_ERR_DEVICE_TIMEOUT in the device status
 * word and returns normally: nothing faults or hangs and the context stays
 * usable.  Read (and clear) the result with attn_get_device_status(); until
 * it is cleared, prefill CTAs skip their work.
 */
attn_status_t attn_selftest_wait_timeout(int limit_ms, attn_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(attn_status_t status);

/* Library version as major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
