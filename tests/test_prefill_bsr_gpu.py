"""Prefill against a KV cache in block-sparse-row form ([Lecture 4] section
5.2), and against block tables of page sizes other than 16, on the GPU
against the float64 oracle (bf16 tolerances).

16-token blocks reach shared memory as one TMA copy each; other block
sizes (the section's block size 4, the radix tree's block size 1, 32 to
128) are gathered row by row.  Both paths must give the oracle's result."""
import json
import math
import os

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def bsr_from_table(table, lens, block):
    """indptr / indices of a block table (its rows' used entries end to end)."""
    counts = [-(-int(n) // block) for n in lens]
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    indices = np.concatenate([table[b, :c] for b, c in enumerate(counts)] +
                             [np.zeros(0, np.int32)]).astype(np.int32)
    return indptr, indices


def make_case(lens_q, lens_k, Hq, Hkv, d, block, seed=0, poison=False):
    _, kb, vb, table, sl = inputs.decode_inputs(lens_k, Hq, Hkv, d, page_size=block, seed=seed)
    q, _, _, cq, _ = inputs.varlen_inputs(lens_q, lens_q, Hq, Hkv, d, seed=seed + 50)
    if poison:  # slots of a request's last block past its length hold NaN
        for b, n in enumerate(lens_k):
            if n % block:
                last = int(table[b, -(-n // block) - 1])
                kb[last, n % block:] = float("nan")
                vb[last, n % block:] = float("nan")
    indptr, indices = bsr_from_table(table.numpy(), lens_k, block)
    return q, kb, vb, table, indptr, indices, cq, sl


def oracle(q, kb, vb, indptr, indices, cq, sl, scale, causal):
    f = lambda t: t.float().numpy()
    return orc.prefill_bsr(f(q), f(kb), f(vb), indptr, indices, cq.numpy(), sl.numpy(), scale,
                           causal)


def run_bsr(lens_q, lens_k, d, block, causal, Hq=8, Hkv=2, seed=0, poison=False):
    q, kb, vb, table, indptr, indices, cq, sl = make_case(lens_q, lens_k, Hq, Hkv, d, block, seed,
                                                          poison)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_prefill_bsr(q.cuda(), kb.cuda(), vb.cuda(), torch.from_numpy(indptr).cuda(),
                                 torch.from_numpy(indices).cuda(), cq.cuda(), sl.cuda(),
                                 causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = oracle(q, kb, vb, indptr, indices, cq, sl, scale, causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return (q, kb, vb, table, cq, sl), (o, lse)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_lecture_5_2_bsr_example(d, causal):
    """The section's three requests (19, 10, 29 tokens; block size 4) with its
    indptr [0, 5, 8, 16] and indices, the last 7 / all 10 / all 29 tokens as
    queries."""
    g = GOLD["lecture_bsr_page_tables"]
    bs, lens = g["block_size"], g["seq_lens"]
    indptr = np.array(g["indptr"], np.int32)
    indices = np.array(g["indices"], np.int32)
    num_blocks = int(indices.max()) + 1
    Hq, Hkv = 8, 2
    gen = torch.Generator().manual_seed(30)
    kb = torch.randn(num_blocks, bs, Hkv, d, generator=gen).to(torch.bfloat16)
    vb = torch.randn(num_blocks, bs, Hkv, d, generator=gen).to(torch.bfloat16)
    lq = [7, 10, 29]
    q, _, _, cq, _ = inputs.varlen_inputs(lq, lq, Hq, Hkv, d, seed=31)
    sl = torch.tensor(lens, dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_prefill_bsr(q.cuda(), kb.cuda(), vb.cuda(), torch.from_numpy(indptr).cuda(),
                                 torch.from_numpy(indices).cuda(), cq.cuda(), sl.cuda(),
                                 causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = oracle(q, kb, vb, indptr, indices, cq, sl, scale, causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    # the same blocks as a block table give the same bits ("max difference 0")
    table = torch.full((3, 8), -1, dtype=torch.int32)
    for b, t in enumerate(g["tables"]):
        table[b, :len(t)] = torch.tensor(t, dtype=torch.int32)
    o2, lse2 = ea.attn_prefill_paged(q.cuda(), kb.cuda(), vb.cuda(), table.cuda(), cq.cuda(),
                                     sl.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("block", [1, 2, 8])
def test_small_blocks_chunked(d, block):
    """Block sizes below 16 (row gathers): chunks at the end of longer
    sequences, ragged lengths, a one-token request; NaN in the unused slots
    of every last block never reaches the result."""
    run_bsr([130, 5, 1, 77], [300, 17, 1, 200], d, block, True, seed=block, poison=True)


@pytest.mark.parametrize("d", [64, 128])
def test_block_size_one_whole_sequences(d):
    """Block size 1 (every token its own block, shuffled over the pool), whole
    sequences of 1 to 400 tokens, not causal and causal."""
    lens = [400, 1, 129, 33]
    run_bsr(lens, lens, d, 1, False, seed=40)
    run_bsr(lens, lens, d, 1, True, seed=41)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("block", [16, 32, 64, 128])
def test_large_blocks(d, block):
    """Block sizes 16 (TMA copies) and 32 to 128 (row gathers), ragged tails with NaN."""
    run_bsr([200, 3, 64], [700, 3, 250], d, block, True, seed=block, poison=True)


@pytest.mark.parametrize("block", [4, 16])
def test_bsr_matches_block_table_bitwise(block):
    """The BSR form and the block-table form of the same cache take the same
    path and give the same bits."""
    (q, kb, vb, table, cq, sl), (o, lse) = run_bsr([50, 300], [500, 300], 128, block, True, seed=60)
    o2, lse2 = ea.attn_prefill_paged(q.cuda(), kb.cuda(), vb.cuda(), table.cuda(), cq.cuda(),
                                     sl.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("block", [1, 4])
def test_decode_as_one_query_per_request(block):
    """Decode through the BSR form: one query row per request, contexts up to
    3000 tokens (GQA 32 / 8, d 128)."""
    lens = [3000, 1, 777, 1024, 65]
    run_bsr([1] * len(lens), lens, 128, block, True, Hq=32, Hkv=8, seed=70 + block)


def test_serving_like_batch_block_4():
    """16 requests, contexts up to 4096 tokens, chunks of up to 256 queries,
    block size 4, Hq 32 / Hkv 8, d 128: full comparison with the oracle."""
    g = np.random.default_rng(80)
    lens_k = g.integers(1, 4097, 16)
    lens_q = np.minimum(lens_k, g.integers(1, 257, 16))
    run_bsr(lens_q.tolist(), lens_k.tolist(), 128, 4, True, Hq=32, Hkv=8, seed=81)


def test_bad_block_index_is_reported():
    """A needed block id outside the pool is reported (ATTN_ERR_BAD_INDEX) and
    never dereferenced; the call returns normally."""
    q, kb, vb, table, indptr, indices, cq, sl = make_case([20, 9], [40, 9], 4, 2, 64, 4, seed=90)
    indices = indices.copy()
    indices[2] = kb.shape[0] + 1000
    ea.attn_prefill_bsr(q.cuda(), kb.cuda(), vb.cuda(), torch.from_numpy(indptr).cuda(),
                        torch.from_numpy(indices).cuda(), cq.cuda(), sl.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
    assert ea.attn_get_device_status() == "ATTN_OK"


def test_too_few_blocks_is_reported():
    """kv_indptr giving a request fewer blocks than its length needs."""
    q, kb, vb, table, indptr, indices, cq, sl = make_case([20, 9], [40, 9], 4, 2, 64, 4, seed=91)
    sl2 = sl.clone()
    sl2[0] = 41  # 10 blocks of 4 hold 40 tokens
    ea.attn_prefill_bsr(q.cuda(), kb.cuda(), vb.cuda(), torch.from_numpy(indptr).cuda(),
                        torch.from_numpy(indices).cuda(), cq.cuda(), sl2.cuda(), causal=True,
                        max_seqlen_k=41)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
