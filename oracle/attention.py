"""Float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library in
``exact_attention_sm_gb300/csrc`` and its Python binding) imports, calls or
links this module.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may use it.  It shares no code,
constants or helpers with the CUDA path; the only thing both sides share are
the seeded input generators in ``exact_attention_sm_gb300/inputs.py``, which
hold none of the method's arithmetic.

Every function is the plain definition (or the pages' algorithm, step by step)
in float64 with numpy; ``@`` (a BLAS matmul) is the only library primitive used
as a step.  Nothing is blocked, fused or reordered beyond what the cited
passage states.

Pages cited (by title; the short tag is used below):

* [Lecture 4]   "Lecture 4 - Efficient attention kernels: FlashAttention and
                FlashInfer" (Stanford CS349D course notes, semidirectx.com)
* [Tiling blog] "The attention formula did not change, so why is it several
                times faster? FlashAttention's tiling, online softmax and IO"
                (zwjcode.cn blog)
* [LLM book]    "10.3 FlashAttention: IO-aware algorithm design" (LLM
                Internals book, yeasy.gitbook.io)
* [CUDA book]   "FlashAttention and inference operators" (CUDA advanced
                handbook, anrans.github.io ai-infra-handbooks)

Parity pins (see tests/test_oracle_pins.py): every function below is pinned
by at least one of worked examples printed on the pages, closed forms,
brute force on tiny inputs, or torch's own float64 math attention.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Softmax building blocks
# --------------------------------------------------------------------------

def safe_softmax(x):
    """Numerically safe softmax of one row.

    [Lecture 4] section 3.2 (online softmax): m(x) = max_i x_i,
    f(x) = exp(x - m(x)), l(x) = sum_i f(x)_i, softmax(x) = f(x) / l(x).
    Returns (softmax, m, l).
    """
    x = _f64(x)
    m = float(x.max())
    f = np.exp(x - m)
    l = float(f.sum())
    return f / l, m, l


def online_softmax_stats(x, block):
    """Stream a row in blocks of ``block`` values keeping only (m, l).

    [Lecture 4] section 3.2: when a new block arrives, compute its local max
    and local sum; if the overall max grows, the old l is multiplied by
    exp(m_old - m_new) before the new block's contribution is added.
    [LLM book] 10.3.2 "Online Softmax" states the same update element-wise.
    Returns the final (m, l) and the list of (m, l) after each block.
    """
    x = _f64(x)
    m, l = NEG_INF, 0.0
    trace = []
    for start in range(0, x.size, block):
        xb = x[start:start + block]
        mb = float(xb.max())
        lb = float(np.exp(xb - mb).sum())
        m_new = max(m, mb)
        old_scale = 0.0 if m == NEG_INF else math.exp(m - m_new)
        l = old_scale * l + math.exp(mb - m_new) * lb
        m = m_new
        trace.append((m, l))
    return m, l, trace


def merge_row_states(state1, state2):
    """Merge two partial row states (m, l, a).

    [Tiling blog] section 03 ("online softmax keeps only three states"):
    m' = max(m, m_b); l' = exp(m - m') l + exp(m_b - m') l_b;
    a' = exp(m - m') a + exp(m_b - m') a_b, where a is the not-yet-divided
    weighted value sum.  An empty state has m = -inf, l = 0, a = 0.
    """
    m1, l1, a1 = state1
    m2, l2, a2 = state2
    m = max(m1, m2)
    if m == NEG_INF:
        return NEG_INF, 0.0, _f64(a1) * 0.0
    c1 = 0.0 if m1 == NEG_INF else math.exp(m1 - m)
    c2 = 0.0 if m2 == NEG_INF else math.exp(m2 - m)
    return m, c1 * l1 + c2 * l2, c1 * _f64(a1) + c2 * _f64(a2)


def block_state(scores, values):
    """The (m, l, a) state of one block of scores with their value rows.

    [Tiling blog] section 03: m_b = block max, l_b = sum exp(s - m_b),
    a_b = sum exp(s - m_b) v.
    """
    s = _f64(scores)
    v = _f64(values)
    mb = float(s.max())
    e = np.exp(s - mb)
    return mb, float(e.sum()), e @ v


# --------------------------------------------------------------------------
# Dense attention: the definition the fused kernel must reproduce
# --------------------------------------------------------------------------

def attention_dense(q, k, v, scale, causal=False, causal_offset=0):
    """Standard (materialising) attention for one head, in float64.

    [Tiling blog] section 01: S = Q K^T * scale, P = softmax(S), O = P V,
    with the scale applied to the scores before the max.  Causal masking
    follows [Tiling blog] section 06: query i sees key j only if j <= i, and
    masked scores are -inf before the max and the sum.  The per-row
    log-sum-exp is LSE = m + ln l ([LLM book] 10.3.2, "LSE").

    causal_offset shifts the rule to key j <= i + causal_offset (0: the
    square rule above; Lk - Lq: the bottom-right alignment of prefill_varlen).

    A row with no visible key (all -inf) has l = 0; its output is O = 0 and
    LSE = -inf rather than NaN ([CUDA book] split-K merge exercise: skip
    empty segments; [Tiling blog] section 11: all-masked rows give NaN if
    unguarded).

    q: [Lq, d], k: [Lk, d], v: [Lk, dv].  Returns (O [Lq, dv], LSE [Lq],
    S [Lq, Lk], P [Lq, Lk]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lq, lk = q.shape[0], k.shape[0]
    s = (q @ k.T) * scale
    if causal:
        i = np.arange(lq)[:, None]
        j = np.arange(lk)[None, :]
        s = np.where(j > i + int(causal_offset), NEG_INF, s)
    if lk == 0:
        m = np.full(lq, NEG_INF)
    else:
        m = s.max(axis=1)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    e = np.where(live[:, None], np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    l_safe = np.where(l > 0, l, 1.0)
    p = e / l_safe[:, None]
    o = p @ v
    lse = np.where(l > 0, m_safe + np.log(l_safe), NEG_INF)
    return o, lse, s, p


def attention_blockwise(q, k, v, scale, causal, block_rows, block_cols):
    """FlashAttention-2 loop order, one head, float64.

    [LLM book] 10.3.2 "tiled forward": for each Q row block i: m = -inf,
    l = 0, O~ = 0; for each K/V column block j (skipped if the causal mask
    hides all of it): S = Q_i K_j^T * scale, m_new = max(m, rowmax S),
    l = l e^(m - m_new) + rowsum e^(S - m_new),
    O~ = O~ e^(m - m_new) + e^(S - m_new) V_j, m = m_new; finally
    O_i = O~ / l and LSE_i = m + ln l.  Masked entries inside a diagonal
    block are -inf ([Tiling blog] section 06).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lq, lk = q.shape[0], k.shape[0]
    o = np.zeros((lq, v.shape[1]))
    lse = np.full(lq, NEG_INF)
    for i0 in range(0, lq, block_rows):
        i1 = min(i0 + block_rows, lq)
        qi = q[i0:i1]
        m = np.full(i1 - i0, NEG_INF)
        l = np.zeros(i1 - i0)
        acc = np.zeros((i1 - i0, v.shape[1]))
        for j0 in range(0, lk, block_cols):
            j1 = min(j0 + block_cols, lk)
            if causal and j0 > i1 - 1:
                continue  # whole block above the diagonal
            s = (qi @ k[j0:j1].T) * scale
            if causal:
                ii = np.arange(i0, i1)[:, None]
                jj = np.arange(j0, j1)[None, :]
                s = np.where(jj > ii, NEG_INF, s)
            m_new = np.maximum(m, s.max(axis=1))
            live = np.isfinite(m_new)
            m_new_safe = np.where(live, m_new, 0.0)
            corr = np.where(np.isfinite(m), np.exp(m - m_new_safe), 0.0)
            corr = np.where(live, corr, 1.0)
            p = np.where(live[:, None], np.exp(s - m_new_safe[:, None]), 0.0)
            l = l * corr + p.sum(axis=1)
            acc = acc * corr[:, None] + p @ v[j0:j1]
            m = m_new
        nz = l > 0
        o[i0:i1][nz] = acc[nz] / l[nz][:, None]
        lse[i0:i1][nz] = m[nz] + np.log(l[nz])
    return o, lse


# --------------------------------------------------------------------------
# Merge of attention states (the LSE merge operator)
# --------------------------------------------------------------------------

def merge_states(o_parts, lse_parts):
    """Merge S partial attention states of one row.

    [LLM book] 10.3.2 "LSE": two key segments with LSE_1, LSE_2 combine as
    LSE = ln(e^LSE_1 + e^LSE_2) and the outputs are weighted by
    e^(LSE_k - LSE).  [CUDA book] "Flash-Decoding and split-K": with
    m = max_s m_s, weights w_s = e^(m_s - m) l_s, O = sum_s w_s O_s / l.
    Written here in the LSE form with M = max_s LSE_s as the shift; a
    segment with no keys (LSE = -inf) is skipped ([CUDA book] split-K merge
    exercise).  If every segment is empty, O = 0 and LSE = -inf.

    o_parts: [S, d] (each O_s already normalised), lse_parts: [S].
    """
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    live = np.isfinite(lse_parts)
    if not live.any():
        return np.zeros(o_parts.shape[1]), NEG_INF
    big = float(lse_parts[live].max())
    w = np.where(live, np.exp(np.where(live, lse_parts, 0.0) - big), 0.0)
    total = float(w.sum())
    o = (w[:, None] * np.where(live[:, None], o_parts, 0.0)).sum(axis=0) / total
    return o, big + math.log(total)


def merge_states_batched(o_parts, lse_parts):
    """merge_states applied to every row: o_parts [rows, S, d], lse [rows, S]."""
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    rows = o_parts.shape[0]
    o = np.zeros((rows, o_parts.shape[2]))
    lse = np.zeros(rows)
    for r in range(rows):
        o[r], lse[r] = merge_states(o_parts[r], lse_parts[r])
    return o, lse


# --------------------------------------------------------------------------
# Batched prefill with grouped-query heads
# --------------------------------------------------------------------------

def kv_head_of(h, hq, hkv):
    """GQA head mapping: query head h reads KV head h / (Hq / Hkv).

    [CUDA book] "a paged decode attention kernel (with GQA)" and its GQA
    exercise: with 32 query heads and 8 KV heads, each KV head serves
    32 / 8 = 4 consecutive query heads.
    """
    return h // (hq // hkv)


def prefill(q, k, v, scale, causal):
    """Dense attention for every (batch, query head).

    q: [B, Hq, Lq, d], k and v: [B, Hkv, Lk, d].  Returns O [B, Hq, Lq, d]
    and LSE [B, Hq, Lq] (natural log), each head by attention_dense.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b_, hq, lq, _ = q.shape
    hkv = k.shape[1]
    o = np.zeros(q.shape[:3] + (v.shape[3],))
    lse = np.zeros(q.shape[:3])
    for b in range(b_):
        for h in range(hq):
            kh = kv_head_of(h, hq, hkv)
            o[b, h], lse[b, h], _, _ = attention_dense(q[b, h], k[b, kh], v[b, kh], scale, causal)
    return o, lse


def prefill_rows(q, k, v, scale, causal, rows):
    """Dense attention for selected query rows only.

    rows: iterable of (b, h, i).  Row i of head h sees keys [0, Lk), or
    [0, i] when causal ([Tiling blog] section 06).  Rows are grouped by
    (b, h) so each group is one small dense problem with the masked scores
    materialised.
    """
    rows = [tuple(int(x) for x in r) for r in rows]
    hq, hkv = q.shape[1], k.shape[1]
    out_o = np.zeros((len(rows), v.shape[3]))
    out_lse = np.zeros(len(rows))
    groups = {}
    for n, (b, h, i) in enumerate(rows):
        groups.setdefault((b, h), []).append((n, i))
    for (b, h), items in groups.items():
        kh = kv_head_of(h, hq, hkv)
        idx = np.array([i for _, i in items])
        qi = _f64(q[b, h][idx])
        kk = _f64(k[b, kh])
        vv = _f64(v[b, kh])
        s = (qi @ kk.T) * scale
        if causal:
            s = np.where(np.arange(kk.shape[0])[None, :] > idx[:, None], NEG_INF, s)
        m = s.max(axis=1)
        live = np.isfinite(m)
        m_safe = np.where(live, m, 0.0)
        e = np.where(live[:, None], np.exp(s - m_safe[:, None]), 0.0)
        l = e.sum(axis=1)
        l_safe = np.where(l > 0, l, 1.0)
        o = (e / l_safe[:, None]) @ vv
        lse = np.where(l > 0, m_safe + np.log(l_safe), NEG_INF)
        for (n, _), orow, lrow in zip(items, o, lse):
            out_o[n] = orow
            out_lse[n] = lrow
    return out_o, out_lse


# --------------------------------------------------------------------------
# Variable-length (packed) prefill
# --------------------------------------------------------------------------

def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, causal):
    """Prefill over sequences packed end to end.

    [LLM book] 10.3.8 (variable-length batching): the sequences of a batch
    are concatenated into [total_tokens, heads, d], and cu_seqlens_q /
    cu_seqlens_k of shape [B + 1] hold the cumulative lengths (lengths 3, 5,
    2 give [0, 3, 8, 10]); sequence b owns rows cu[b] .. cu[b+1]-1 and no
    sequence sees another.  GQA as in prefill.

    Causal with Lq != Lk is not defined on the pages; the reading here aligns
    it bottom-right: query i of a sequence with Lq queries and Lk keys sees
    key j <= i + (Lk - Lq), the queries being the last Lq tokens of that
    sequence (chunked prefill).  With Lq = Lk this is the square rule.

    q [total_q, Hq, d]; k, v [total_k, Hkv, d].  Returns O [total_q, Hq, d]
    and LSE [total_q, Hq].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    hq, hkv = q.shape[1], k.shape[1]
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for b in range(len(cu_seqlens_q) - 1):
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        k0, k1 = int(cu_seqlens_k[b]), int(cu_seqlens_k[b + 1])
        for h in range(hq):
            kh = kv_head_of(h, hq, hkv)
            oo, ll, _, _ = attention_dense(q[q0:q1, h], k[k0:k1, kh], v[k0:k1, kh], scale, causal,
                                           (k1 - k0) - (q1 - q0))
            o[q0:q1, h], lse[q0:q1, h] = oo, ll
    return o, lse


# --------------------------------------------------------------------------
# Paged KV cache and decode
# --------------------------------------------------------------------------

def paged_gather(pages, table_row, seq_len, kv_head):
    """Logical-order K (or V) rows of one request and one KV head, in float64.

    [CUDA book] "PagedAttention": token t lives in physical page
    block_table[t / page_size], slot t % page_size.  pages has the layout
    [num_pages, page_size, Hkv, d] ([CUDA book] paged decode listing; [LLM
    book] 10.3.7 k_cache layout).  Table entries past ceil(seq_len /
    page_size) are never read.
    """
    page_size = pages.shape[1]
    t = np.arange(int(seq_len))
    page_of_token = np.asarray(table_row)[t // page_size].astype(np.int64)
    slot_of_token = t % page_size
    return _f64(pages[page_of_token, slot_of_token, kv_head])


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale):
    """One query token per request against its paged KV cache.

    q: [B, Hq, d]; k_pages, v_pages: [num_pages, page_size, Hkv, d];
    block_table: [B, max_pages]; seq_lens: [B].  Gathers keys in logical
    order (paged_gather) and applies attention_dense with Lq = 1 and no
    mask.  Returns O [B, Hq, d] and LSE [B, Hq].
    """
    q = _f64(q)
    b_, hq, _ = q.shape
    hkv = k_pages.shape[2]
    o = np.zeros(q.shape)
    lse = np.zeros((b_, hq))
    for b in range(b_):
        n = int(seq_lens[b])
        for kh in range(hkv):
            kk = paged_gather(k_pages, block_table[b], n, kh)
            vv = paged_gather(v_pages, block_table[b], n, kh)
            heads = [h for h in range(hq) if kv_head_of(h, hq, hkv) == kh]
            oo, ll, _, _ = attention_dense(q[b, heads], kk, vv, scale, False)
            o[b, heads] = oo
            lse[b, heads] = ll
    return o, lse


def prefill_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seq_lens_k, scale, causal):
    """Chunked prefill of packed queries against a paged KV cache.

    [Lecture 4] section 5.2: prefill over KV kept in shuffled physical
    blocks gives exactly the attention over the blocks gathered into
    contiguous arrays; [LLM book] 10.3.7 "addressing by block table":
    block_table [B, max_pages], k_cache [num_pages, page_size, Hkv, d].
    Sequence b's queries are rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of
    q [total_q, Hq, d] ([LLM book] 10.3.8 packing); its keys are tokens
    0 .. seq_lens_k[b]-1 of its pages (paged_gather).  Causal is aligned
    bottom-right as in prefill_varlen: the queries are the last Lq tokens of
    the Lk-token sequence (their K/V already in the cache).

    Returns O [total_q, Hq, d] and LSE [total_q, Hq].
    """
    q = _f64(q)
    hq = q.shape[1]
    hkv = k_pages.shape[2]
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for b in range(len(cu_seqlens_q) - 1):
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        lk = int(seq_lens_k[b])
        for h in range(hq):
            kh = kv_head_of(h, hq, hkv)
            kk = paged_gather(k_pages, block_table[b], lk, kh)
            vv = paged_gather(v_pages, block_table[b], lk, kh)
            oo, ll, _, _ = attention_dense(q[q0:q1, h], kk, vv, scale, causal, lk - (q1 - q0))
            o[q0:q1, h], lse[q0:q1, h] = oo, ll
    return o, lse


def prefill_bsr(q, k_blocks, v_blocks, kv_indptr, kv_indices, cu_seqlens_q, seq_lens_k, scale,
                causal):
    """Prefill against a KV cache addressed in block-sparse-row (BSR) form.

    [Lecture 4] section 5.2: the "query rows x physical KV blocks" matrix of
    a batch is block-sparse; in BSR form indices lists the non-zero blocks
    (physical block ids) of every row end to end and row r's blocks are
    indices[indptr[r] : indptr[r + 1]].  A page table is this matrix with
    block size 16 (vLLM), a radix tree with block size 1 (SGLang); the
    attention over the blocks gathered in order equals the attention over
    the contiguous KV ("max difference 0").  Here row r is request r: its
    keys are tokens 0 .. seq_lens_k[r] - 1, token t in block
    indices[indptr[r] + t // block_size], slot t % block_size, with
    k_blocks, v_blocks [num_blocks, block_size, Hkv, d].  Queries are packed
    (cu_seqlens_q) and causal is aligned bottom-right, as in prefill_paged.

    Returns O [total_q, Hq, d] and LSE [total_q, Hq].
    """
    q = _f64(q)
    hq = q.shape[1]
    hkv = k_blocks.shape[2]
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for b in range(len(cu_seqlens_q) - 1):
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        lk = int(seq_lens_k[b])
        row = np.asarray(kv_indices[int(kv_indptr[b]):int(kv_indptr[b + 1])])
        for h in range(hq):
            kh = kv_head_of(h, hq, hkv)
            kk = paged_gather(k_blocks, row, lk, kh)
            vv = paged_gather(v_blocks, row, lk, kh)
            oo, ll, _, _ = attention_dense(q[q0:q1, h], kk, vv, scale, causal, lk - (q1 - q0))
            o[q0:q1, h], lse[q0:q1, h] = oo, ll
    return o, lse


def decode_split_states(q_row, keys, values, scale, chunk):
    """Split-KV partial states of one query row (Flash-Decoding).

    [LLM book] 10.3.7 and [CUDA book] "Flash-Decoding and split-K": the keys
    are cut along their length into segments of ``chunk`` tokens; each
    segment yields its own normalised output O_s and LSE_s.  Returns
    (o_parts [S, d], lse_parts [S]).
    """
    n = keys.shape[0]
    nsplit = max(1, -(-n // chunk))
    o_parts = np.zeros((nsplit, values.shape[1]))
    lse_parts = np.full(nsplit, NEG_INF)
    for s in range(nsplit):
        lo, hi = s * chunk, min((s + 1) * chunk, n)
        if hi > lo:
            oo, ll, _, _ = attention_dense(_f64(q_row)[None, :], keys[lo:hi], values[lo:hi], scale)
            o_parts[s], lse_parts[s] = oo[0], ll[0]
    return o_parts, lse_parts


# --------------------------------------------------------------------------
# Cascade (shared-prefix) decode
# --------------------------------------------------------------------------

def cascade_kv_tokens(prefix_len, unique_lens):
    """KV tokens read by plain decode and by cascade decode.

    [Lecture 4] section 4.4 and exercise 7: with n requests sharing a prefix,
    plain decode reads the prefix once per request, n * prefix + sum(unique);
    cascade reads it once, prefix + sum(unique).  The same count in blocks
    gives section 5.3's block totals.  Returns (plain, cascade, saving) with
    saving = 1 - cascade / plain.
    """
    unique = [int(u) for u in unique_lens]
    plain = len(unique) * int(prefix_len) + sum(unique)
    cascade = int(prefix_len) + sum(unique)
    return plain, cascade, 1.0 - cascade / plain


def decode_cascade(q, prefix_k, prefix_v, k_pages, v_pages, block_table, suffix_lens, scale):
    """Decode over a shared prefix plus per-request suffixes, the cascade way.

    [Lecture 4] section 4.4 (cascade attention) and 5.3 (composable formats):
      1. prefix part: for each KV head, the query rows of that head from all n
         requests are stacked into one (n * g) x d matrix and attend once to
         the shared prefix K/V: one dense problem, the prefix read once;
      2. unique part: each request's rows attend to its own suffix, read from
         the paged cache (paged_gather);
      3. the two attention states of each row are merged with the LSE
         operator (merge_states).

    q: [B, Hq, d]; prefix_k, prefix_v: [Hkv, P, d] (the shared prefix, stored
    once); k_pages, v_pages, block_table, suffix_lens: the suffixes, as in
    decode_paged.  A request with no suffix tokens keeps the prefix state.
    Returns O [B, Hq, d] and LSE [B, Hq].
    """
    q = _f64(q)
    b_, hq, d = q.shape
    hkv = prefix_k.shape[0]
    o = np.zeros(q.shape)
    lse = np.zeros((b_, hq))
    for kh in range(hkv):
        heads = [h for h in range(hq) if kv_head_of(h, hq, hkv) == kh]
        rows = [(b, h) for b in range(b_) for h in heads]
        stacked = np.stack([q[b, h] for b, h in rows])
        o_pre, lse_pre, _, _ = attention_dense(stacked, prefix_k[kh], prefix_v[kh], scale, False)
        for i, (b, h) in enumerate(rows):
            n = int(suffix_lens[b])
            kk = paged_gather(k_pages, block_table[b], n, kh)
            vv = paged_gather(v_pages, block_table[b], n, kh)
            o_suf, lse_suf, _, _ = attention_dense(q[b, h][None, :], kk, vv, scale, False)
            o[b, h], lse[b, h] = merge_states(np.stack([o_pre[i], o_suf[0]]),
                                              np.array([lse_pre[i], lse_suf[0]]))
    return o, lse


# --------------------------------------------------------------------------
# Backward pass (training)
# --------------------------------------------------------------------------

def attention_backward(q, k, v, do, scale, causal=False):
    """Gradients of O = softmax(scale Q K^T) V for one head, in float64.

    [LLM book] "backward and recomputation" and [Tiling blog] section 07:
    the forward keeps only O and the per-row LSE; the backward rebuilds
    S = scale Q K^T and P = exp(S - LSE) and accumulates dQ, dK, dV.  The
    pages print no gradient formulas; these are the chain rule through
    O = P V and the row softmax, materialised whole:
        dV = P^T dO
        dP = dO V^T
        D_i = sum_j P_ij dP_ij
        dS = P * (dP - D)          (elementwise, D_i along row i)
        dQ = scale dS K,   dK = scale dS^T Q
    Masked entries (causal, square rule as attention_dense) have P = 0 and
    contribute nothing; a row with no visible key gets dQ = 0.
    Returns dQ [Lq, d], dK [Lk, d], dV [Lk, d] and D [Lq].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    _, lse, s, _ = attention_dense(q, k, v, scale, causal)
    with np.errstate(invalid="ignore"):
        p = np.exp(s - lse[:, None])
    p[~np.isfinite(lse)] = 0.0
    p[~np.isfinite(p)] = 0.0
    dv = p.T @ do
    dp = do @ v.T
    dd = (p * dp).sum(axis=1)
    ds = p * (dp - dd[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv, dd


def backward(q, k, v, do, scale, causal):
    """attention_backward over [B, H, L, d] tensors with grouped-query
    heads (kv_head_of): a KV head's dK, dV sum the contributions of all the
    query heads that read it.  Returns dQ [B,Hq,Lq,d], dK and dV
    [B,Hkv,Lk,d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    b_, hq = q.shape[:2]
    hkv = k.shape[1]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(b_):
        for h in range(hq):
            kh = kv_head_of(h, hq, hkv)
            gq, gk, gv, _ = attention_backward(q[b, h], k[b, kh], v[b, kh], do[b, h], scale, causal)
            dq[b, h] = gq
            dk[b, kh] += gk
            dv[b, kh] += gv
    return dq, dk, dv


# --------------------------------------------------------------------------
# Split planning (host integer logic)
# --------------------------------------------------------------------------

def _cdiv(a, b):
    return -(-a // b)


def plan_units(seq_lens, num_kv_heads, chunk):
    """Non-empty work units (request, KV head, segment) when every request is
    cut into segments of `chunk` tokens: Hkv * sum_b ceil(len_b / chunk)."""
    return num_kv_heads * sum(_cdiv(int(n), chunk) for n in seq_lens)


def plan_splits(seq_lens, num_kv_heads, slots, page_size, num_splits=0):
    """Choose the KV chunk length of each request for split-KV decode.

    Returns (chunk [B], splits [B]) with splits_b = ceil(len_b / chunk_b)
    (at least 1) and every chunk a multiple of page_size (one chunk shared by
    all requests).

    Reading of the pages ([Lecture 4] section 4.2, exercise 6 and its answer):
    a work unit is (request, KV head, segment) and `slots` workers run one
    unit each at a time.  The answer to exercise 6 picks the finest split
    whose units still fit in one round of the workers (2 x 8 x 8 = 128 <= 132
    SMs; more segments need a second round with smaller units and only add
    merging), and its rule of thumb asks for requests x KV heads x segments
    just within the worker count.  With requests of different lengths the
    same rule is taken on the chunk length itself:
    * C = the shortest multiple of page_size for which the non-empty units
      Hkv * sum_b ceil(len_b / C) fit in `slots`;
    * if even C = the longest length (no split) gives more units than slots,
      nothing is split ("when the batch is large there are enough work units;
      splitting only adds merge overhead").
    This gives 8 segments for 2 requests x 16384 tokens x 8 KV heads on 132
    SMs (the exercise's answer) and 16 segments (16x faster) for 1 x 32K
    (section 4.2).
    * num_splits > 0 forces at most that many segments per request:
      C = ceil(ceil(max_len / num_splits) / page_size) * page_size.
    """
    lens = [int(x) for x in seq_lens]
    bsz = len(lens)
    longest = max([1] + lens)
    if num_splits > 0:
        c = max(page_size, _cdiv(_cdiv(longest, num_splits), page_size) * page_size)
        return [c] * bsz, [max(1, _cdiv(n, c)) for n in lens]
    full = max(page_size, _cdiv(longest, page_size) * page_size)
    best_c = full
    if plan_units(lens, num_kv_heads, full) <= slots:
        # smallest page multiple that still fits: units(C) never grows with C
        lo, hi = 1, full // page_size          # in pages; hi fits
        while lo < hi:
            mid = (lo + hi) // 2
            if plan_units(lens, num_kv_heads, mid * page_size) <= slots:
                hi = mid
            else:
                lo = mid + 1
        best_c = hi * page_size
    return [best_c] * bsz, [max(1, _cdiv(n, best_c)) for n in lens]


def plan_balanced(seq_lens, num_groups, num_ctas, page_size, unit_cost=lambda n: n):
    """Load-balanced split schedule for decode ([Lecture 4] section 5.6).

    Follows the section's steps for decode (one query row per request, so
    ceil(l_qo / T_q) = 1):
      2. L_kv = ceil(sum_b l_kv(b) * num_groups / num_ctas), here rounded up
         to a multiple of page_size (a segment starts on a page);
      3. the KV of every (request, group) is cut into consecutive segments of
         at most L_kv tokens, each a work unit (a request of length 0 keeps
         one empty unit, so that its output is written);
      4. units are sorted by cost (unit_cost(tokens), 1. in the section:
         alpha l_q + beta l_kv with l_q = 1 fixed) from large to small, ties
         in list order, and each goes to the CTA with the smallest total cost
         so far (lowest index on ties): longest processing time first;
      5. the units of one (request, group), in token order, are what the
         merge combines.
    Returns (units, cta_units): units[u] = (b, group, t_begin, t_end) in
    list order (request, group, segment), cta_units[c] = the unit ids of CTA
    c in the order they were assigned.
    """
    import heapq
    lens = [max(0, int(x)) for x in seq_lens]
    total = sum(lens) * num_groups
    lkv = max(1, -(-total // num_ctas))
    lkv = -(-lkv // page_size) * page_size
    units = []
    for b, n in enumerate(lens):
        for grp in range(num_groups):
            if n == 0:
                units.append((b, grp, 0, 0))
            for t0 in range(0, n, lkv):
                units.append((b, grp, t0, min(n, t0 + lkv)))
    order = sorted(range(len(units)), key=lambda u: (-unit_cost(units[u][3] - units[u][2]), u))
    heap = [(0, c) for c in range(num_ctas)]
    cta_units = [[] for _ in range(num_ctas)]
    for u in order:
        load, c = heapq.heappop(heap)
        cta_units[c].append(u)
        heapq.heappush(heap, (load + unit_cost(units[u][3] - units[u][2]), c))
    return units, cta_units

