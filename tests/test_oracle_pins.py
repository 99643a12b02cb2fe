"""Pins for the float64 oracle against things other than itself.

Each test checks one oracle function against values printed on the pages
(tests/golden/worked_examples.json), closed forms, brute force on tiny
inputs, or an independent library routine (torch's float64 math attention,
scipy's logsumexp / softmax).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import attention as orc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def close(got, want, decimals):
    tol = 10.0 ** (-decimals)
    return abs(float(got) - float(want)) <= tol


# ---------------------------------------------------------------- worked examples

def test_safe_and_online_softmax_lecture_exercise_1():
    g = GOLD["lecture_exercise_1"]
    p, m, l = orc.safe_softmax(g["x"])
    for got, want in zip(p, g["softmax"]):
        assert close(got, want, g["decimals"]["softmax"])
    m_final, l_final, trace = orc.online_softmax_stats(g["x"], 1)
    for (tm, tl), want in zip(trace, g["trace"]):
        assert tm == want["m"]
        assert close(tl, want["l"], g["decimals"]["l"])
    assert m_final == m and abs(l_final - l) < 1e-15


def test_block_merge_tiling_blog_section_04():
    g = GOLD["tiling_blog_two_merges"]
    s, v = np.array(g["scores"], float), np.array(g["values"], float)[:, None]
    b0, b1 = g["blocks"]
    st0 = orc.block_state(s[b0], v[b0])
    assert st0[0] == g["after_first_block"]["m"]
    assert close(st0[1], g["after_first_block"]["l"], g["decimals"]["l"])
    assert close(st0[2][0], g["after_first_block"]["a"], g["decimals"]["a"])
    st = orc.merge_row_states(st0, orc.block_state(s[b1], v[b1]))
    assert st[0] == g["after_merge"]["m"]
    assert close(st[1], g["after_merge"]["l"], g["decimals"]["l"])
    assert close(st[2][0], g["after_merge"]["a"], g["decimals"]["a"])
    assert close(st[2][0] / st[1], g["o"], g["decimals"]["o"])
    # the same row through the dense definition: d = 1, q = 1, k = scores
    o, lse, _, _ = orc.attention_dense([[1.0]], s[:, None], v, 1.0)
    assert close(o[0, 0], g["o"], g["decimals"]["o"])


@pytest.mark.parametrize("name", ["llm_book_max_not_refreshed", "llm_book_max_refreshed"])
def test_online_update_llm_book(name):
    g = GOLD[name]
    s, v = np.array(g["scores"], float), np.array(g["values"], float)[:, None]
    b0, b1 = g["blocks"]
    st0 = orc.block_state(s[b0], v[b0])
    assert st0[0] == g["after_first_block"]["m"]
    assert close(st0[1], g["after_first_block"]["l"], g["decimals"]["l"])
    assert close(st0[2][0], g["after_first_block"]["o_tilde"], g["decimals"]["o_tilde"])
    st = orc.merge_row_states(st0, orc.block_state(s[b1], v[b1]))
    assert close(st[1], g["final"]["l"], g["decimals"]["l"])
    assert close(st[2][0], g["final"]["o_tilde"], g["decimals"]["o_tilde"])
    assert close(st[2][0] / st[1], g["o"], g["decimals"]["o"])
    if "correction" in g:
        assert close(math.exp(st0[0] - st[0]), g["correction"], g["decimals"]["correction"])
    # blockwise FA2 order with one-column blocks reproduces the same output
    for bc in (1, 2, 3):
        o, _ = orc.attention_blockwise([[1.0]], s[:, None], v, 1.0, False, 1, bc)
        assert close(o[0, 0], g["o"], g["decimals"]["o"])


def test_weights_and_lse_llm_book():
    g = GOLD["llm_book_softmax_weights_and_lse"]
    s, v = np.array(g["scores"], float), np.array(g["values"], float)[:, None]
    o, lse, _, p = orc.attention_dense([[1.0]], s[:, None], v, 1.0)
    for got, want in zip(p[0], g["weights"]):
        assert close(got, want, g["decimals"]["weights"])
    assert close(o[0, 0], g["o"], g["decimals"]["o"])
    assert close(lse[0], g["lse"], g["decimals"]["lse"])
    # the LSE merge of the two segments [1,3] | [2] gives the same O and LSE
    parts_o, parts_l = [], []
    for idx in ([0, 1], [2]):
        oo, ll, _, _ = orc.attention_dense([[1.0]], s[idx][:, None], v[idx], 1.0)
        parts_o.append(oo[0]); parts_l.append(ll[0])
    mo, ml = orc.merge_states(np.array(parts_o), np.array(parts_l))
    assert close(mo[0], g["o"], g["decimals"]["o"])
    assert close(ml, g["lse"], g["decimals"]["lse"])


def test_cuda_book_exercise_1():
    g = GOLD["cuda_book_exercise_1"]
    (s0, s1), (v0, v1) = g["blocks_scores"], g["blocks_values"]
    st0 = orc.block_state(s0, np.array(v0, float)[:, None])
    assert st0[0] == g["after_first_block"]["m"]
    assert close(st0[1], g["after_first_block"]["l"], g["decimals"]["l"])
    assert close(st0[2][0], g["after_first_block"]["o_tilde"], g["decimals"]["o_tilde"])
    st = orc.merge_row_states(st0, orc.block_state(s1, np.array(v1, float)[:, None]))
    assert st[0] == g["after_second_block"]["m"]
    assert close(st[1], g["after_second_block"]["l"], g["decimals"]["l"])
    assert close(st[2][0], g["after_second_block"]["o_tilde"], g["decimals"]["o_tilde"])
    assert close(st[2][0] / st[1], g["o"], g["decimals"]["o"])
    # direct computation printed beside it
    s = np.array(s0 + s1, float)
    assert close(np.exp(s).sum(), g["direct_weight_sum"], g["decimals"]["direct_weight_sum"])
    for got, want in zip(np.exp(s), g["direct_weights_unnormalised"]):
        assert abs(got - want) / want < 1e-3
    # the split-K merge of the two normalised segment outputs (LSE form)
    o0, l0, _, _ = orc.attention_dense([[1.0]], np.array(s0, float)[:, None], np.array(v0, float)[:, None], 1.0)
    o1, l1, _, _ = orc.attention_dense([[1.0]], np.array(s1, float)[:, None], np.array(v1, float)[:, None], 1.0)
    mo, _ = orc.merge_states(np.array([o0[0], o1[0]]), np.array([l0[0], l1[0]]))
    assert close(mo[0], g["o"], g["decimals"]["o"])


# ---------------------------------------------------------------- dense attention vs a library

def _sdpa64(q, k, v, scale, causal):
    """torch's math attention in float64 (independent code path)."""
    q, k, v = (torch.as_tensor(np.asarray(x, np.float64)) for x in (q, k, v))
    hq, hkv = q.shape[-3], k.shape[-3]
    if hq != hkv:
        k = k.repeat_interleave(hq // hkv, dim=-3)
        v = v.repeat_interleave(hq // hkv, dim=-3)
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    if causal:
        lq, lk = s.shape[-2], s.shape[-1]
        mask = torch.ones(lq, lk, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, -math.inf)
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", [(17, 17), (64, 64), (1, 9), (33, 70)])
def test_dense_matches_torch_math_attention(causal, lq, lk):
    if causal and lq != lk:
        pytest.skip("causal is defined for square problems here")
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((lq, 32)), rng.standard_normal((lk, 32)), rng.standard_normal((lk, 24))
    o, lse, s, p = orc.attention_dense(q, k, v, 0.3, causal)
    o_ref, lse_ref = _sdpa64(q[None], k[None], v[None], 0.3, causal)
    assert np.abs(o - o_ref[0]).max() < 1e-12
    assert np.abs(lse - lse_ref[0]).max() < 1e-12
    assert np.abs(lse - scipy.special.logsumexp(s, axis=1)).max() < 1e-12
    assert np.abs(p - scipy.special.softmax(s, axis=1)).max() < 1e-13


def test_prefill_gqa_matches_torch_math_attention():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 8, 40, 16))
    k = rng.standard_normal((2, 2, 40, 16))
    v = rng.standard_normal((2, 2, 40, 16))
    for causal in (False, True):
        o, lse = orc.prefill(q, k, v, 0.25, causal)
        o_ref, lse_ref = _sdpa64(q, k, v, 0.25, causal)
        assert np.abs(o - o_ref).max() < 1e-12
        assert np.abs(lse - lse_ref).max() < 1e-12
        rows = [(1, 7, 39), (0, 0, 0), (1, 3, 17), (0, 5, 1)]
        ro, rl = orc.prefill_rows(q, k, v, 0.25, causal, rows)
        for n, (b, h, i) in enumerate(rows):
            assert np.abs(ro[n] - o_ref[b, h, i]).max() < 1e-12
            assert abs(rl[n] - lse_ref[b, h, i]) < 1e-12


# ---------------------------------------------------------------- invariants and closed forms

def test_invariants_rows_sum_to_one_and_hull():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((50, 8)), rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    for causal in (False, True):
        o, lse, s, p = orc.attention_dense(q, k, v, 1.0 / math.sqrt(8), causal)
        assert np.abs(p.sum(axis=1) - 1.0).max() < 1e-14
        m = s.max(axis=1)
        l = np.exp(s - m[:, None]).sum(axis=1)
        assert np.abs(lse - (m + np.log(l))).max() < 1e-13
        assert (lse >= m - 1e-15).all()
        for i in range(50):
            vis = v[: i + 1] if causal else v
            assert (o[i] >= vis.min(axis=0) - 1e-12).all() and (o[i] <= vis.max(axis=0) + 1e-12).all()


def test_closed_forms():
    rng = np.random.default_rng(4)
    k, v = rng.standard_normal((20, 8)), rng.standard_normal((20, 8))
    # q = 0: uniform weights, O = mean of the visible values, LSE = ln(#visible)
    o, lse, _, _ = orc.attention_dense(np.zeros((20, 8)), k, v, 0.5, True)
    for i in range(20):
        assert np.abs(o[i] - v[: i + 1].mean(axis=0)).max() < 1e-13
        assert abs(lse[i] - math.log(i + 1)) < 1e-13
    # causal row 0 sees only key 0
    q = rng.standard_normal((20, 8))
    o, lse, s, _ = orc.attention_dense(q, k, v, 0.5, True)
    assert np.abs(o[0] - v[0]).max() < 1e-15 and abs(lse[0] - 0.5 * q[0] @ k[0]) < 1e-14
    # one key: O = v_0
    o, _, _, _ = orc.attention_dense(q, k[:1], v[:1], 0.5, False)
    assert np.abs(o - v[0]).max() < 1e-15
    # identical keys: O = mean(V)
    o, _, _, _ = orc.attention_dense(q, np.tile(k[:1], (20, 1)), v, 0.5, False)
    assert np.abs(o - v.mean(axis=0)).max() < 1e-13
    # no keys at all: O = 0, LSE = -inf (no NaN)
    o, lse, _, _ = orc.attention_dense(q, k[:0], v[:0], 0.5, False)
    assert (o == 0).all() and np.isneginf(lse).all()


# ---------------------------------------------------------------- orderings (brute force)

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("length", [1, 7, 64])
def test_blockwise_orders_equal_dense(causal, length):
    """[Lecture 4] 3.3: tiled and dense agree for several tile sizes."""
    rng = np.random.default_rng(length)
    q, k, v = (rng.standard_normal((length, 16)) for _ in range(3))
    o_ref, lse_ref, _, _ = orc.attention_dense(q, k, v, 0.25, causal)
    for br in (1, 3, 16, length):
        for bc in (1, 3, 16, length):
            o, lse = orc.attention_blockwise(q, k, v, 0.25, causal, br, bc)
            assert np.abs(o - o_ref).max() < 1e-13
            assert np.abs(lse - lse_ref).max() < 1e-13


@pytest.mark.parametrize("segments", [2, 8, 64])
def test_split_then_merge_equals_dense(segments):
    """[Lecture 4] 4.3: one query, 10^4 keys, 2/8/64 segments, FP64 ~1e-16."""
    rng = np.random.default_rng(segments)
    q = rng.standard_normal(64)
    k, v = rng.standard_normal((10000, 64)), rng.standard_normal((10000, 64))
    o_ref, lse_ref, _, _ = orc.attention_dense(q[None], k, v, 0.125)
    chunk = -(-10000 // segments)
    op, lp = orc.decode_split_states(q, k, v, 0.125, chunk)
    assert op.shape[0] == segments
    o, lse = orc.merge_states(op, lp)
    assert np.abs(o - o_ref[0]).max() < 1e-14
    assert abs(lse - lse_ref[0]) < 1e-12
    # commutative: reversed and shuffled orders agree in double
    o2, lse2 = orc.merge_states(op[::-1], lp[::-1])
    perm = rng.permutation(segments)
    o3, lse3 = orc.merge_states(op[perm], lp[perm])
    assert np.abs(o2 - o).max() < 1e-14 and np.abs(o3 - o).max() < 1e-14
    assert abs(lse2 - lse) < 1e-12 and abs(lse3 - lse) < 1e-12
    # associative: merging merged halves gives the same state
    h = segments // 2
    oa, la = orc.merge_states(op[:h], lp[:h])
    ob, lb = orc.merge_states(op[h:], lp[h:])
    o4, lse4 = orc.merge_states(np.array([oa, ob]), np.array([la, lb]))
    assert np.abs(o4 - o).max() < 1e-14 and abs(lse4 - lse) < 1e-12


def test_merge_skips_empty_segments():
    rng = np.random.default_rng(9)
    op, lp = rng.standard_normal((4, 8)), rng.standard_normal(4)
    lp2 = lp.copy(); lp2[2] = -math.inf
    op2 = op.copy(); op2[2] = np.nan  # contents of an empty segment must not be read
    o, lse = orc.merge_states(op2, lp2)
    o_ref, lse_ref = orc.merge_states(op[[0, 1, 3]], lp[[0, 1, 3]])
    assert np.abs(o - o_ref).max() < 1e-15 and abs(lse - lse_ref) < 1e-15
    o, lse = orc.merge_states(op, np.full(4, -math.inf))
    assert (o == 0).all() and lse == -math.inf
    assert abs(orc.merge_states(op[:1], lp[:1])[1] - lp[0]) < 1e-15


def _segment_states(scores, values, cuts):
    """(O_s, LSE_s) of one row whose score list is cut at `cuts`, each segment by
    the dense definition (d = 1, q = 1, k = the scores)."""
    s, v = np.asarray(scores, float), np.asarray(values, float)
    bounds = [0] + list(cuts) + [len(s)]
    op, lp = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        oo, ll, _, _ = orc.attention_dense([[1.0]], s[a:b, None], v[a:b, None], 1.0)
        op.append(oo[0] if b > a else np.zeros(1))
        lp.append(ll[0] if b > a else -math.inf)
    return np.array(op), np.array(lp)


def test_merge_batched_worked_examples_by_row():
    """merge_states_batched on a batch whose rows are the pages' split examples:
    [LLM book] 10.3.2's scores [1,3,2] / values [10,20,30] split [1,3]|[2]
    (O = 21.547, LSE = 3.4076), the same row split [1]|[3,2], [CUDA book]
    exercise 1 ([1,3]|[2,5] with [10,20]|[30,40], O = 36.88), a row whose
    middle segment is empty, and a row with every segment empty (O = 0,
    LSE = -inf).  Rows and segments are shuffled: each output row must be its
    own example's value."""
    g = GOLD["llm_book_softmax_weights_and_lse"]
    c = GOLD["cuda_book_exercise_1"]
    cases = [
        (_segment_states(g["scores"], g["values"], [2]), g["o"], g["lse"]),
        (_segment_states(g["scores"], g["values"], [1]), g["o"], g["lse"]),
        (_segment_states(c["blocks_scores"][0] + c["blocks_scores"][1],
                         c["blocks_values"][0] + c["blocks_values"][1], [2]), c["o"], None),
        (_segment_states(g["scores"], g["values"], [2, 2]), g["o"], g["lse"]),
    ]
    S = 3
    rows_o, rows_l, want = [], [], []
    rng = np.random.default_rng(11)
    for (op, lp), o_want, lse_want in cases:
        # pad to S segments with empty states (garbage O, LSE = -inf), then shuffle
        pad = S - len(lp)
        op = np.concatenate([op, np.full((pad, 1), np.nan)])
        lp = np.concatenate([lp, np.full(pad, -math.inf)])
        perm = rng.permutation(S)
        rows_o.append(op[perm]); rows_l.append(lp[perm]); want.append((o_want, lse_want))
    rows_o.append(np.full((S, 1), 7.0)); rows_l.append(np.full(S, -math.inf))
    want.append((0.0, -math.inf))
    order = rng.permutation(len(want))
    o, lse = orc.merge_states_batched(np.array(rows_o)[order], np.array(rows_l)[order])
    assert o.shape == (len(want), 1) and lse.shape == (len(want),)
    for out_row, src in enumerate(order):
        o_want, lse_want = want[src]
        if lse_want == -math.inf:
            assert o[out_row, 0] == 0.0 and lse[out_row] == -math.inf
            continue
        assert close(o[out_row, 0], o_want, 2), (src, o[out_row, 0], o_want)
        if lse_want is not None:
            assert close(lse[out_row], lse_want, 4)


def test_merge_batched_equals_dense_rows():
    """Split-then-merge over a batch of rows equals the dense attention of each
    row over all its keys ([Lecture 4] 4.3), with rows of different queries and
    key sets so that a transposed row or segment index shows."""
    rng = np.random.default_rng(12)
    rows, n, d, S = 6, 300, 8, 5
    q = rng.standard_normal((rows, d))
    k = rng.standard_normal((rows, n, d))
    v = rng.standard_normal((rows, n, d))
    op = np.zeros((rows, S, d)); lp = np.zeros((rows, S))
    o_ref = np.zeros((rows, d)); lse_ref = np.zeros(rows)
    for r in range(rows):
        oo, ll, _, _ = orc.attention_dense(q[r][None], k[r], v[r], 0.3)
        o_ref[r], lse_ref[r] = oo[0], ll[0]
        op[r], lp[r] = orc.decode_split_states(q[r], k[r], v[r], 0.3, 60)
    o, lse = orc.merge_states_batched(op, lp)
    assert np.abs(o - o_ref).max() < 1e-13 and np.abs(lse - lse_ref).max() < 1e-12
    # the segments of a row are an unordered set; the rows keep their order
    perm_s = rng.permutation(S)
    o2, lse2 = orc.merge_states_batched(op[:, perm_s], lp[:, perm_s])
    assert np.abs(o2 - o_ref).max() < 1e-13 and np.abs(lse2 - lse_ref).max() < 1e-12
    perm_r = rng.permutation(rows)
    o3, lse3 = orc.merge_states_batched(op[perm_r], lp[perm_r])
    assert np.abs(o3 - o_ref[perm_r]).max() < 1e-13
    assert np.abs(lse3 - lse_ref[perm_r]).max() < 1e-12


# ---------------------------------------------------------------- paging and GQA

def test_bsr_page_tables_lecture_5_2():
    g = GOLD["lecture_bsr_page_tables"]
    bs = g["block_size"]
    num_pages = max(max(t) for t in g["tables"]) + 1
    # page p, slot s of KV head 0 holds the integer 1000 * p + s (exact in float)
    pages = np.zeros((num_pages, bs, 1, 2))
    for p in range(num_pages):
        for s in range(bs):
            pages[p, s, 0] = [1000 * p + s, p]
    indices, indptr = [], [0]
    for n, table in zip(g["seq_lens"], g["tables"]):
        rows = orc.paged_gather(pages, table, n, 0)
        assert rows.shape[0] == n
        used = []
        for t in range(n):
            assert rows[t, 0] == 1000 * table[t // bs] + t % bs
            if not used or used[-1] != int(rows[t, 1]):
                used.append(int(rows[t, 1]))
        indices += used
        indptr.append(len(indices))
    assert indices == g["indices"] and indptr == g["indptr"]


def test_gqa_mapping_cuda_book_exercise_3():
    g = GOLD["gqa_head_sharing"]
    heads = [orc.kv_head_of(h, g["num_heads"], g["num_kv_heads"]) for h in range(g["num_heads"])]
    for kh in range(g["num_kv_heads"]):
        assert heads.count(kh) == g["group"]
        assert heads[kh * g["group"]: (kh + 1) * g["group"]] == [kh] * g["group"]


def test_decode_paged_equals_contiguous_attention():
    """[Lecture 4] 5.2: attention over the paged layout equals attention over
    the same keys stored contiguously (max diff 0)."""
    rng = np.random.default_rng(21)
    lens, page, hkv, hq, d = [1, 17, 40, 64], 16, 2, 8, 32
    contig_k = [rng.standard_normal((hkv, n, d)) for n in lens]
    contig_v = [rng.standard_normal((hkv, n, d)) for n in lens]
    npages = sum(-(-n // page) for n in lens)
    perm = rng.permutation(npages)
    kp = np.zeros((npages, page, hkv, d)); vp = np.zeros_like(kp)
    table = -np.ones((4, 4), dtype=np.int64)
    off = 0
    for b, n in enumerate(lens):
        for i in range(-(-n // page)):
            table[b, i] = perm[off]; off += 1
            for s in range(page):
                t = i * page + s
                if t < n:
                    kp[table[b, i], s] = contig_k[b][:, t]
                    vp[table[b, i], s] = contig_v[b][:, t]
    q = rng.standard_normal((4, hq, d))
    o, lse = orc.decode_paged(q, kp, vp, table, lens, 0.2)
    for b, n in enumerate(lens):
        o_ref, lse_ref = _sdpa64(q[b][:, None, :], contig_k[b], contig_v[b], 0.2, False)
        assert np.abs(o[b] - o_ref[:, 0]).max() < 1e-12
        assert np.abs(lse[b] - lse_ref[:, 0]).max() < 1e-12


# ---------------------------------------------------------------- split planning

def test_plan_lecture_exercise_6():
    g = GOLD["lecture_exercise_6_split_count"]
    chunk, splits = orc.plan_splits(g["seq_lens"], g["num_kv_heads"], g["slots"], 16)
    assert splits == [g["best_splits"]] * len(g["seq_lens"])


def test_plan_lecture_split_kv_speedup():
    g = GOLD["lecture_split_kv_speedup"]
    chunk, splits = orc.plan_splits(g["seq_lens"], g["num_kv_heads"], g["slots"], 16)
    units = g["num_kv_heads"] * sum(splits)
    assert units <= g["slots"]
    # lecture model: time = waves x tokens per unit; unsplit = one unit of 32K
    assert g["seq_lens"][0] // chunk[0] == g["speedup"]


def test_plan_invariants():
    rng = np.random.default_rng(2)
    for _ in range(50):
        lens = rng.integers(0, 140000, size=int(rng.integers(1, 9))).tolist()
        hkv = int(rng.choice([1, 2, 8]))
        slots = int(rng.choice([132, 152, 304, 608]))
        for forced in (0, 1, 3, 64):
            chunk, splits = orc.plan_splits(lens, hkv, slots, 16, forced)
            for n, c, s in zip(lens, chunk, splits):
                assert c % 16 == 0 and c >= 16 and s >= 1
                assert s * c >= n and (s - 1) * c < max(n, 1)
                if forced:
                    assert s <= forced
    # enough units already: nothing is split
    assert orc.plan_splits([1024] * 256, 8, 152, 16)[1] == [1] * 256


def test_plan_one_round():
    """Exercise 6's answer: the finest split whose units still fit in one
    round; one page less per chunk would need a second round."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        lens = rng.integers(0, 140000, size=int(rng.integers(1, 9))).tolist()
        hkv = int(rng.choice([1, 2, 8]))
        slots = int(rng.choice([132, 152, 456]))
        c = orc.plan_splits(lens, hkv, slots, 16)[0][0]
        units = hkv * sum(-(-n // c) for n in lens)
        if hkv * sum(1 for n in lens if n > 0) <= slots:
            assert units <= slots
            assert c == 16 or hkv * sum(-(-n // (c - 16)) for n in lens) > slots
        else:
            assert c >= max(lens)      # not split


# ---------------------------------------------------------------- cascade decode

def test_cascade_tokens_lecture_exercise_7():
    g = GOLD["lecture_exercise_7_cascade_tokens"]
    plain, cascade, saving = orc.cascade_kv_tokens(g["prefix"], [g["unique"]] * g["n_requests"])
    assert (plain, cascade) == (g["plain"], g["cascade"])
    assert round(100 * saving) == g["saving_percent"]


def test_cascade_blocks_lecture_5_3():
    """Section 5.3 prints only the totals; the unique blocks are whatever the
    plain count leaves after n x shared (76 - 4 x 15 = 16), in any split."""
    g = GOLD["lecture_5_3_composable_blocks"]
    unique_total = g["plain_blocks"] - g["n_requests"] * g["shared_blocks"]
    for split in ([4, 4, 4, 4], [1, 2, 6, 7], [16, 0, 0, 0]):
        assert sum(split) == unique_total
        plain, cascade, _ = orc.cascade_kv_tokens(g["shared_blocks"], split)
        assert (plain, cascade) == (g["plain_blocks"], g["cascade_blocks"])


def test_cascade_saving_lecture_summary():
    g = GOLD["lecture_cascade_64_requests"]
    _, _, saving = orc.cascade_kv_tokens(g["prefix"], [g["unique"]] * g["n_requests"])
    assert round(100 * saving) == g["saving_percent"]


def _cascade_case(rng, prefix_len, suffix_lens, hkv=2, hq=6, d=16, page=4):
    pk = rng.standard_normal((hkv, prefix_len, d))
    pv = rng.standard_normal((hkv, prefix_len, d))
    suf_k = [rng.standard_normal((hkv, n, d)) for n in suffix_lens]
    suf_v = [rng.standard_normal((hkv, n, d)) for n in suffix_lens]
    npages = sum(-(-n // page) for n in suffix_lens) + 1
    perm = rng.permutation(npages)
    kp = np.zeros((npages, page, hkv, d)); vp = np.zeros_like(kp)
    maxp = max(1, max(-(-n // page) for n in suffix_lens))
    table = -np.ones((len(suffix_lens), maxp), dtype=np.int64)
    off = 0
    for b, n in enumerate(suffix_lens):
        for i in range(-(-n // page)):
            table[b, i] = perm[off]; off += 1
            for s in range(page):
                t = i * page + s
                if t < n:
                    kp[table[b, i], s] = suf_k[b][:, t]
                    vp[table[b, i], s] = suf_v[b][:, t]
    q = rng.standard_normal((len(suffix_lens), hq, d))
    return q, pk, pv, suf_k, suf_v, kp, vp, table


@pytest.mark.parametrize("prefix_len,suffix_lens", [(7, [0, 1, 5, 13]), (33, [9, 0]), (1, [4])])
def test_cascade_equals_attention_over_whole_sequence(prefix_len, suffix_lens):
    """[Lecture 4] 4.4: the cascade result equals attending to prefix + suffix
    as one sequence; checked against torch's float64 math attention on the
    concatenated keys (an independent routine)."""
    rng = np.random.default_rng(prefix_len * 100 + len(suffix_lens))
    q, pk, pv, suf_k, suf_v, kp, vp, table = _cascade_case(rng, prefix_len, suffix_lens)
    o, lse = orc.decode_cascade(q, pk, pv, kp, vp, table, suffix_lens, 0.3)
    hq, hkv = q.shape[1], pk.shape[0]
    for b, n in enumerate(suffix_lens):
        kk = np.concatenate([pk, suf_k[b]], axis=1)   # [hkv, P + n, d]
        vv = np.concatenate([pv, suf_v[b]], axis=1)
        rep = hq // hkv
        o_ref, lse_ref = _sdpa64(q[b][:, None, :], np.repeat(kk, rep, axis=0),
                                 np.repeat(vv, rep, axis=0), 0.3, False)
        assert np.abs(o[b] - o_ref[:, 0]).max() < 1e-12
        assert np.abs(lse[b] - lse_ref[:, 0]).max() < 1e-12


# ---------------------------------------------------------------- varlen prefill

def test_varlen_cu_seqlens_llm_book_10_3_8():
    """The page's packing example, and sequences that never see each other:
    each packed sequence equals its own dense attention."""
    g = GOLD["llm_book_varlen_cu_seqlens"]
    cu = np.concatenate([[0], np.cumsum(g["lengths"])]).tolist()
    assert cu == g["cu_seqlens"]
    rng = np.random.default_rng(5)
    q = rng.standard_normal((cu[-1], 4, 8))
    k = rng.standard_normal((cu[-1], 2, 8))
    v = rng.standard_normal((cu[-1], 2, 8))
    for causal in (False, True):
        o, lse = orc.prefill_varlen(q, k, v, cu, cu, 0.4, causal)
        for b in range(len(g["lengths"])):
            sl = slice(cu[b], cu[b + 1])
            o_ref, lse_ref = _sdpa64(q[sl].transpose(1, 0, 2), k[sl].transpose(1, 0, 2),
                                     v[sl].transpose(1, 0, 2), 0.4, causal)
            assert np.abs(o[sl] - o_ref.transpose(1, 0, 2)).max() < 1e-12
            assert np.abs(lse[sl] - lse_ref.T).max() < 1e-12


def _sdpa64_mask(q, k, v, scale, mask):
    """torch float64 math attention with an explicit boolean mask (True = visible)."""
    q, k, v = (torch.as_tensor(np.asarray(x, np.float64)) for x in (q, k, v))
    from torch.nn.attention import SDPBackend, sdpa_kernel
    m = torch.as_tensor(mask)
    with sdpa_kernel(SDPBackend.MATH):
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    s = ((q @ k.transpose(-1, -2)) * scale).masked_fill(~m, -math.inf)
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("lq,lk", [(5, 12), (12, 12), (1, 9), (130, 300)])
def test_varlen_bottom_right_causal_matches_masked_sdpa(lq, lk):
    """Bottom-right causal (query i sees key j <= i + lk - lq) against torch's
    attention with the same explicit mask; GQA 4 query heads on 2 KV heads."""
    rng = np.random.default_rng(lq * 1000 + lk)
    q = rng.standard_normal((lq, 4, 16))
    k = rng.standard_normal((lk, 2, 16))
    v = rng.standard_normal((lk, 2, 16))
    o, lse = orc.prefill_varlen(q, k, v, [0, lq], [0, lk], 0.25, True)
    mask = np.arange(lk)[None, :] <= np.arange(lq)[:, None] + (lk - lq)
    o_ref, lse_ref = _sdpa64_mask(q.transpose(1, 0, 2), np.repeat(k, 2, 1).transpose(1, 0, 2),
                                  np.repeat(v, 2, 1).transpose(1, 0, 2), 0.25, mask)
    assert np.abs(o - o_ref.transpose(1, 0, 2)).max() < 1e-12
    assert np.abs(lse - lse_ref.T).max() < 1e-12


def test_varlen_rows_with_no_visible_key():
    """More queries than keys under bottom-right causal: the first lq - lk
    rows see nothing and give O = 0, LSE = -inf (never NaN)."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((6, 1, 8))
    k = rng.standard_normal((2, 1, 8))
    v = rng.standard_normal((2, 1, 8))
    o, lse = orc.prefill_varlen(q, k, v, [0, 6], [0, 2], 0.3, True)
    assert (o[:4] == 0).all() and np.isneginf(lse[:4]).all()
    # rows 4 and 5 see keys j <= row + (2 - 6), i.e. the square rule on the last two rows
    o_last, lse_last, _, _ = orc.attention_dense(q[4:, 0], k[:, 0], v[:, 0], 0.3, True, 0)
    assert np.isfinite(lse[4:]).all() and np.abs(o[4:, 0] - o_last).max() == 0


# ---------------------------------------------------------------- paged prefill

@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_lecture_5_2_equals_contiguous(causal):
    """[Lecture 4] section 5.2: prefill of the three requests (lengths 19,
    10, 29; block size 4; the page's shuffled block tables) over the paged
    cache equals attention over the same K/V laid out contiguously, here
    computed by torch float64 with its own masking (independent code)."""
    g = GOLD["lecture_bsr_page_tables"]
    bs, lens, tables = g["block_size"], g["seq_lens"], g["tables"]
    rng = np.random.default_rng(11)
    num_pages, hq, hkv, d = 24, 4, 2, 8
    kp = rng.standard_normal((num_pages, bs, hkv, d))
    vp = rng.standard_normal((num_pages, bs, hkv, d))
    table = np.full((3, 8), -1)
    for b, t in enumerate(tables):
        table[b, :len(t)] = t
    lq = [5, 10, 29]                      # chunks: the last 5, all 10, all 29 tokens
    cu = np.concatenate([[0], np.cumsum(lq)])
    q = rng.standard_normal((int(cu[-1]), hq, d))
    o, lse = orc.prefill_paged(q, kp, vp, table, cu, lens, 0.3, causal)
    for b in range(3):
        # contiguous K/V by direct indexing of the block table (no paged_gather)
        pages = np.asarray(tables[b])
        k = kp[pages].reshape(-1, hkv, d)[:lens[b]]
        v = vp[pages].reshape(-1, hkv, d)[:lens[b]]
        mask = np.ones((lq[b], lens[b]), bool)
        if causal:
            mask = np.arange(lens[b])[None, :] <= np.arange(lq[b])[:, None] + lens[b] - lq[b]
        qq = q[cu[b]:cu[b + 1]].transpose(1, 0, 2)
        kk = np.repeat(k, hq // hkv, 1).transpose(1, 0, 2)
        vv = np.repeat(v, hq // hkv, 1).transpose(1, 0, 2)
        o_ref, lse_ref = _sdpa64_mask(qq, kk, vv, 0.3, mask)
        assert np.abs(o[cu[b]:cu[b + 1]] - o_ref.transpose(1, 0, 2)).max() < 1e-12
        assert np.abs(lse[cu[b]:cu[b + 1]] - lse_ref.T).max() < 1e-12


def test_paged_prefill_with_whole_sequence_matches_varlen():
    """Queries covering the whole sequence: the paged prefill is the packed
    prefill of the gathered keys (the page's 'max diff 0')."""
    rng = np.random.default_rng(12)
    bs, hkv, d = 16, 1, 8
    lens = [37, 16, 1]
    pages = [[3, 0, 5], [1], [4]]
    kp = rng.standard_normal((6, bs, hkv, d))
    vp = rng.standard_normal((6, bs, hkv, d))
    table = np.full((3, 3), -1)
    for b, t in enumerate(pages):
        table[b, :len(t)] = t
    cu = np.concatenate([[0], np.cumsum(lens)])
    q = rng.standard_normal((int(cu[-1]), 2, d))
    o, lse = orc.prefill_paged(q, kp, vp, table, cu, lens, 0.5, True)
    kc = np.concatenate([kp[p].reshape(-1, hkv, d)[:n] for p, n in zip(pages, lens)])
    vc = np.concatenate([vp[p].reshape(-1, hkv, d)[:n] for p, n in zip(pages, lens)])
    o2, lse2 = orc.prefill_varlen(q, kc, vc, cu, cu, 0.5, True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    """The chain-rule gradients equal torch autograd through torch's float64
    math attention (independent code), with grouped-query heads."""
    rng = np.random.default_rng(31)
    q = rng.standard_normal((2, 4, 7, 5))
    k = rng.standard_normal((2, 2, 7, 5))
    v = rng.standard_normal((2, 2, 7, 5))
    do = rng.standard_normal((2, 4, 7, 5))
    dq, dk, dv = orc.backward(q, k, v, do, 0.4, causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(2, dim=1), tv.repeat_interleave(2, dim=1), is_causal=causal,
            scale=0.4)
    (o * torch.tensor(do)).sum().backward()
    assert np.abs(dq - tq.grad.numpy()).max() < 1e-12
    assert np.abs(dk - tk.grad.numpy()).max() < 1e-12
    assert np.abs(dv - tv.grad.numpy()).max() < 1e-12


def test_backward_finite_differences():
    """Central differences of the loss sum(dO * O) on a tiny head."""
    rng = np.random.default_rng(32)
    q, k, v, do = (rng.standard_normal((4, 3)) for _ in range(4))
    dq, dk, dv, _ = orc.attention_backward(q, k, v, do, 0.7, True)

    def loss(qq, kk, vv):
        return float((orc.attention_dense(qq, kk, vv, 0.7, True)[0] * do).sum())

    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += eps
            up = loss(*args)
            args[which][idx] -= 2 * eps
            num[idx] = (up - loss(*args)) / (2 * eps)
        assert np.abs(num - g).max() < 1e-7


def test_backward_closed_forms():
    rng = np.random.default_rng(33)
    q, do = rng.standard_normal((5, 4)), rng.standard_normal((5, 4))
    k, v = rng.standard_normal((1, 4)), rng.standard_normal((1, 4))
    # one key: P = 1 everywhere, so dV = sum of dO, and dS = P (dP - D) = 0
    dq, dk, dv, _ = orc.attention_backward(q, k, v, do, 0.5, False)
    assert np.abs(dv[0] - do.sum(0)).max() < 1e-14
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    # D_i = sum_j P_ij dP_ij equals rowsum(dO_i * O_i) (O = P V)
    k, v = rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    o = orc.attention_dense(q, k, v, 0.5, True)[0]
    _, _, _, dd = orc.attention_backward(q, k, v, do, 0.5, True)
    assert np.abs(dd - (do * o).sum(1)).max() < 1e-13
    # no keys at all: every row sees nothing, so every gradient is zero
    dq, dk, dv, _ = orc.attention_backward(q, k[:0], v[:0], do, 0.5, False)
    assert (dq == 0).all() and dk.shape == (0, 4) and dv.shape == (0, 4)


# ---------------------------------------------------------------- load-balanced schedule

def test_balanced_plan_segments_lecture_5_6():
    """Steps 2-3 of [Lecture 4] section 5.6 on a hand example: L_kv =
    ceil(150 / 4) = 38 tokens, on a 16-token page grid 48; every request is
    cut into consecutive segments of at most 48 tokens."""
    units, cta_units = orc.plan_balanced([100, 50, 0], 1, 4, 16)
    assert units == [(0, 0, 0, 48), (0, 0, 48, 96), (0, 0, 96, 100), (1, 0, 0, 48),
                     (1, 0, 48, 50), (2, 0, 0, 0)]
    assert sorted(u for c in cta_units for u in c) == list(range(len(units)))


def test_balanced_plan_covers_every_token_once():
    rng = np.random.default_rng(41)
    for _ in range(100):
        lens = rng.integers(0, 20000, size=int(rng.integers(1, 9))).tolist()
        groups, ctas = int(rng.choice([1, 2, 8])), int(rng.choice([4, 132, 456]))
        units, cta_units = orc.plan_balanced(lens, groups, ctas, 16)
        lkv = -(-max(1, -(-sum(lens) * groups // ctas)) // 16) * 16
        for b, n in enumerate(lens):
            for grp in range(groups):
                segs = [u for u in units if u[0] == b and u[1] == grp]
                assert segs[0][2] == 0 and segs[-1][3] == n
                for a, c in zip(segs, segs[1:]):
                    assert a[3] == c[2]
                assert all(u[2] % 16 == 0 and u[3] - u[2] <= lkv for u in segs)
        assert sorted(u for c in cta_units for u in c) == list(range(len(units)))


def test_balanced_plan_lpt_bound_against_brute_force():
    """Step 4 is the longest-processing-time greedy: on tiny instances its
    makespan stays within Graham's bound (4/3 - 1/(3m)) of the optimum found
    by trying every assignment."""
    import itertools
    rng = np.random.default_rng(42)
    for _ in range(40):
        lens = rng.integers(1, 200, size=int(rng.integers(2, 5))).tolist()
        m = int(rng.integers(2, 4))
        units, cta_units = orc.plan_balanced(lens, 1, m, 16, unit_cost=lambda n: n)
        if len(units) > 8:
            continue
        cost = [u[3] - u[2] for u in units]
        span = max(sum(cost[u] for u in c) for c in cta_units)
        best = min(max(sum(cost[u] for u, a in zip(range(len(cost)), assign) if a == k)
                       for k in range(m))
                   for assign in itertools.product(range(m), repeat=len(cost)))
        assert span <= (4 / 3 - 1 / (3 * m)) * best + 1e-9
        # each CTA received its units from the longest down
        for c in cta_units:
            assert all(cost[a] >= cost[b] for a, b in zip(c, c[1:]))


@pytest.mark.parametrize("causal", [False, True])
def test_bsr_prefill_lecture_5_2_example(causal):
    """[Lecture 4] section 5.2: the three requests (19, 10, 29 tokens, block
    size 4) in the page's BSR form (indptr [0, 5, 8, 16] and its indices)
    give exactly the attention of the block-table form ('max difference 0')
    and, within float64 rounding, torch's attention over the contiguous K/V."""
    g = GOLD["lecture_bsr_page_tables"]
    bs, lens = g["block_size"], g["seq_lens"]
    indptr, indices = np.array(g["indptr"]), np.array(g["indices"])
    rng = np.random.default_rng(21)
    hq, hkv, d = 4, 2, 8
    kb = rng.standard_normal((24, bs, hkv, d))
    vb = rng.standard_normal((24, bs, hkv, d))
    lq = [7, 10, 29]
    cu = np.concatenate([[0], np.cumsum(lq)])
    q = rng.standard_normal((int(cu[-1]), hq, d))
    o, lse = orc.prefill_bsr(q, kb, vb, indptr, indices, cu, lens, 0.3, causal)
    table = np.full((3, 8), -1)
    for b, t in enumerate(g["tables"]):
        table[b, :len(t)] = t
    o_t, lse_t = orc.prefill_paged(q, kb, vb, table, cu, lens, 0.3, causal)
    assert np.array_equal(o, o_t) and np.array_equal(lse, lse_t)
    for b in range(3):
        blocks = indices[indptr[b]:indptr[b + 1]]
        k = kb[blocks].reshape(-1, hkv, d)[:lens[b]]
        v = vb[blocks].reshape(-1, hkv, d)[:lens[b]]
        mask = np.ones((lq[b], lens[b]), bool)
        if causal:
            mask = np.arange(lens[b])[None, :] <= np.arange(lq[b])[:, None] + lens[b] - lq[b]
        qq = q[cu[b]:cu[b + 1]].transpose(1, 0, 2)
        kk = np.repeat(k, hq // hkv, 1).transpose(1, 0, 2)
        vv = np.repeat(v, hq // hkv, 1).transpose(1, 0, 2)
        o_ref, lse_ref = _sdpa64_mask(qq, kk, vv, 0.3, mask)
        assert np.abs(o[cu[b]:cu[b + 1]] - o_ref.transpose(1, 0, 2)).max() < 1e-12
        assert np.abs(lse[cu[b]:cu[b + 1]] - lse_ref.T).max() < 1e-12


def test_bsr_prefill_block_size_one():
    """Block size 1 (the radix-tree layout, [Lecture 4] exercise 9(a)): every
    token its own block, at a shuffled position of the pool; equals the
    attention over the tokens in logical order (torch float64)."""
    rng = np.random.default_rng(22)
    lens, hq, hkv, d = [13, 1, 30], 2, 1, 8
    pool = rng.permutation(sum(lens) + 5)
    kb = rng.standard_normal((len(pool), 1, hkv, d))
    vb = rng.standard_normal((len(pool), 1, hkv, d))
    indptr = np.concatenate([[0], np.cumsum(lens)])
    indices = pool[:sum(lens)]
    lq = [4, 1, 30]
    cu = np.concatenate([[0], np.cumsum(lq)])
    q = rng.standard_normal((int(cu[-1]), hq, d))
    o, lse = orc.prefill_bsr(q, kb, vb, indptr, indices, cu, lens, 0.35, True)
    for b in range(3):
        tok = indices[indptr[b]:indptr[b + 1]]
        k, v = kb[tok, 0], vb[tok, 0]
        mask = np.arange(lens[b])[None, :] <= np.arange(lq[b])[:, None] + lens[b] - lq[b]
        qq = q[cu[b]:cu[b + 1]].transpose(1, 0, 2)
        o_ref, lse_ref = _sdpa64_mask(qq, np.repeat(k, hq, 1).transpose(1, 0, 2),
                                      np.repeat(v, hq, 1).transpose(1, 0, 2), 0.35, mask)
        assert np.abs(o[cu[b]:cu[b + 1]] - o_ref.transpose(1, 0, 2)).max() < 1e-12
        assert np.abs(lse[cu[b]:cu[b + 1]] - lse_ref.T).max() < 1e-12
