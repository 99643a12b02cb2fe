"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU with
``torch.Generator().manual_seed(seed)`` in float32 from N(0, 1), in the order
Q, K, V (q, k_pages, v_pages for decode), then cast to the requested dtype.
"""
from __future__ import annotations

import torch

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed, device="cpu"):
    return torch.Generator(device=device).manual_seed(int(seed))


def prefill_inputs(B, Hq, Hkv, Lq, Lk, d, dtype="bf16", seed=0, device="cpu"):
    """q [B,Hq,Lq,d], k and v [B,Hkv,Lk,d], N(0,1), contiguous.

    device="cpu" (the default, used for every oracle comparison) draws with the
    CPU generator; device="cuda" draws with the CUDA generator of the same seed
    (a different stream of numbers with the same distribution, used where only
    timing matters)."""
    g = _gen(seed, device)
    q = torch.randn(B, Hq, Lq, d, generator=g, device=device)
    k = torch.randn(B, Hkv, Lk, d, generator=g, device=device)
    v = torch.randn(B, Hkv, Lk, d, generator=g, device=device)
    dt = _DT[dtype]
    return q.to(dt), k.to(dt), v.to(dt)


def sample_rows(B, Hq, Lq, n_random=4096, tile=128, seed=3):
    """Rows (b, h, i) checked on large prefill problems.

    The first ``tile`` query rows of (b=0, h=0), the last ``tile`` rows of
    (b=B-1, h=Hq-1), and ``n_random`` rows drawn by
    ``torch.randperm(B*Hq*Lq, generator=seed)``.
    """
    rows = [(0, 0, i) for i in range(min(tile, Lq))]
    rows += [(B - 1, Hq - 1, i) for i in range(max(0, Lq - tile), Lq)]
    total = B * Hq * Lq
    pick = torch.randperm(total, generator=_gen(seed))[: min(n_random, total)].tolist()
    for flat in pick:
        b, rem = divmod(flat, Hq * Lq)
        h, i = divmod(rem, Lq)
        rows.append((b, h, i))
    return rows


def decode_lengths_uniform(B, lo, hi, seed=2):
    """Per-request context lengths uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (B,), generator=_gen(seed)).tolist()


def decode_inputs(seq_lens, Hq, Hkv, d, page_size=16, dtype="bf16", seed=0, perm_seed=1,
                  extra_table_cols=0, device="cpu"):
    """Paged decode inputs with a shuffled block table.

    The pool holds exactly sum_b ceil(len_b / page_size) pages.  A random
    permutation of the pool (``torch.randperm(num_pages, generator=perm_seed)``)
    is handed out to the requests in order; table entries past a request's
    last page are -1.  Returns q [B,Hq,d], k_pages and v_pages
    [num_pages, page_size, Hkv, d], block_table int32 [B, max_pages],
    seq_lens int32 [B].  The table is always built on the CPU; device="cuda"
    draws q/k/v with the CUDA generator (timing only) and returns all five on
    the GPU.
    """
    B = len(seq_lens)
    pages_per = [-(-int(n) // page_size) for n in seq_lens]
    num_pages = max(1, sum(pages_per))
    max_pages = max(1, max(pages_per)) + int(extra_table_cols)
    perm = torch.randperm(num_pages, generator=_gen(perm_seed))
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    g = _gen(seed, device)
    q = torch.randn(B, Hq, d, generator=g, device=device)
    k_pages = torch.randn(num_pages, page_size, Hkv, d, generator=g, device=device)
    v_pages = torch.randn(num_pages, page_size, Hkv, d, generator=g, device=device)
    dt = _DT[dtype]
    lens = torch.tensor([int(n) for n in seq_lens], dtype=torch.int32)
    return (q.to(dt), k_pages.to(dt), v_pages.to(dt), table.to(device), lens.to(device))


def merge_inputs(rows, S, d, seed=0, empty_frac=0.0):
    """Random partial states: o_parts [rows,S,d] f32, lse_parts [rows,S] f32.

    A fraction ``empty_frac`` of the (row, segment) states is marked empty
    (LSE = -inf); the first row has every segment empty when empty_frac > 0.
    """
    g = _gen(seed)
    o = torch.randn(rows, S, d, generator=g)
    lse = torch.randn(rows, S, generator=g) * 4.0
    if empty_frac > 0:
        drop = torch.rand(rows, S, generator=g) < empty_frac
        lse[drop] = float("-inf")
        lse[0, :] = float("-inf")
    return o, lse


def cascade_inputs(prefix_len, suffix_lens, Hq, Hkv, d, seed=0, device="cpu"):
    """Shared-prefix decode inputs: the suffixes exactly as decode_inputs
    (q, paged cache, shuffled table) with ``seed``, then the prefix K and V
    [Hkv, prefix_len, d] bf16 ~ N(0,1) drawn from ``seed + 100``.  Returns
    (q, prefix_k, prefix_v, k_pages, v_pages, block_table, suffix_lens)."""
    q, kp, vp, table, sl = decode_inputs(suffix_lens, Hq, Hkv, d, seed=seed, perm_seed=seed + 1,
                                         device=device)
    g = _gen(seed + 100, device)
    pk = torch.randn(Hkv, prefix_len, d, generator=g, device=device).to(torch.bfloat16)
    pv = torch.randn(Hkv, prefix_len, d, generator=g, device=device).to(torch.bfloat16)
    return q, pk, pv, kp, vp, table, sl



def varlen_inputs(lens_q, lens_k, Hq, Hkv, d, seed=0, device="cpu"):
    """Packed (variable-length) prefill inputs: q [sum lens_q, Hq, d], k and v
    [sum lens_k, Hkv, d], bf16 ~ N(0,1) drawn in the order q, k, v, plus the
    int32 cumulative lengths cu_seqlens_q / cu_seqlens_k [B + 1]."""
    g = _gen(seed, device)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = torch.randn(max(tq, 1), Hq, d, generator=g, device=device)[:tq].to(torch.bfloat16)
    k = torch.randn(max(tk, 1), Hkv, d, generator=g, device=device)[:tk].to(torch.bfloat16)
    v = torch.randn(max(tk, 1), Hkv, d, generator=g, device=device)[:tk].to(torch.bfloat16)
    cu = lambda lens: torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()),
                                   dtype=torch.int32, device=device)
    return q.contiguous(), k.contiguous(), v.contiguous(), cu(lens_q), cu(lens_k)
