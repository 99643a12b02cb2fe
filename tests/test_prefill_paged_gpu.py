"""Chunked prefill against a paged KV cache, bf16, against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def make_case(lens_q, lens_k, Hq, Hkv, d, seed=0, poison=False):
    """Packed queries (cu_seqlens) and a shuffled 16-token page cache; with
    `poison`, every cache slot past a sequence's length holds NaN."""
    _, kp, vp, table, sl = inputs.decode_inputs(lens_k, Hq, Hkv, d, seed=seed)
    q, _, _, cq, _ = inputs.varlen_inputs(lens_q, lens_q, Hq, Hkv, d, seed=seed + 50)
    if poison:
        for b, n in enumerate(lens_k):
            pages = -(-n // 16)
            if n % 16:
                last = int(table[b, pages - 1])
                kp[last, n % 16:] = float("nan")
                vp[last, n % 16:] = float("nan")
    return q, kp, vp, table, cq, sl


def run(lens_q, lens_k, d, causal, Hq=8, Hkv=2, seed=0, poison=False):
    q, kp, vp, table, cq, sl = make_case(lens_q, lens_k, Hq, Hkv, d, seed, poison)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_prefill_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cq.cuda(),
                                   sl.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.prefill_paged(q.float().numpy(), kp.float().numpy(), vp.float().numpy(),
                                       table.numpy(), cq.numpy(), sl.numpy(), scale, causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_chunked_prefill_mixed(d, causal):
    """Chunks of new tokens at the end of longer cached sequences, ragged
    tails, a one-token chunk and a whole-sequence chunk."""
    run([300, 5, 128, 1, 77], [300, 17, 1000, 1, 200], d, causal, seed=1)


@pytest.mark.parametrize("d", [64, 128])
def test_lecture_5_2_lengths(d):
    """The three requests of [Lecture 4] section 5.2 (19, 10, 29 tokens),
    prefilled whole from the paged cache."""
    run([19, 10, 29], [19, 10, 29], d, True, seed=2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_garbage_past_the_length_never_reaches_the_result(d, causal):
    """Slots of a last page past the sequence's length hold NaN: the result
    is finite and equals the oracle's (which never reads those slots)."""
    run([40, 3, 200], [57, 130, 213], d, causal, seed=3, poison=True)


@pytest.mark.parametrize("d", [64, 128])
def test_more_queries_than_keys(d):
    o, lse = run([100, 20], [30, 20], d, True, Hq=4, Hkv=4, seed=4)
    assert torch.isneginf(lse[:70]).all() and (o[:70] == 0).all()


@pytest.mark.parametrize("d", [64, 128])
def test_no_keys(d):
    o, lse = run([5, 9], [0, 0], d, True, seed=5)
    assert (o == 0).all() and torch.isneginf(lse).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_equals_packed_prefill_bitwise(d, causal):
    """The paged cache gathered into contiguous K/V and run through the
    packed prefill gives bitwise the same output: same tiles, same order."""
    lens_q, lens_k = [200, 64, 3], [333, 64, 150]
    q, kp, vp, table, cq, sl = make_case(lens_q, lens_k, 8, 2, d, seed=6)
    o_p, lse_p = ea.attn_prefill_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cq.cuda(),
                                       sl.cuda(), causal=causal)
    ks, vs = [], []
    for b, n in enumerate(lens_k):
        pages = table[b, : -(-n // 16)].long()
        ks.append(kp[pages].reshape(-1, 2, d)[:n])
        vs.append(vp[pages].reshape(-1, 2, d)[:n])
    ck = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    o_v, lse_v = ea.attn_fwd_varlen(q.cuda(), torch.cat(ks).cuda(), torch.cat(vs).cuda(), cq.cuda(),
                                    ck.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_v) and torch.equal(lse_p, lse_v)


@pytest.mark.parametrize("d,B", [(128, 4096), (64, 4097)])
def test_many_requests_sorted_list_and_fallback(d, B):
    """4096 work units fill the per-CTA sorted item list; 4097 keep the
    round-robin order.  Chunks of 1 to 128 tokens after up to 300 cached
    ones."""
    g = np.random.default_rng(60 + B)
    lens_q = g.integers(1, 129, B)
    lens_k = lens_q + g.integers(0, 301, B)
    run(lens_q.tolist(), lens_k.tolist(), d, True, Hq=2, Hkv=1, seed=10)


def test_long_context_chunks_sampled():
    """A serving-like batch (Hq 32, Hkv 8, d 128): 8 requests with cached
    contexts up to 8192 tokens and new chunks up to 512, checked on sampled
    (request, head, row block) triples against the oracle's attention."""
    g = torch.Generator().manual_seed(21)
    lens_k = torch.randint(1, 8193, (8,), generator=g).tolist()
    lens_q = [min(n, int(c)) for n, c in zip(lens_k, torch.randint(1, 513, (8,), generator=g))]
    q, kp, vp, table, cq, sl = make_case(lens_q, lens_k, 32, 8, 128, seed=7)
    o, lse = ea.attn_prefill_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cq.cuda(),
                                   sl.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o, lse = to_np(o), to_np(lse)
    qn, kn, vn = q.float().numpy(), kp.float().numpy(), vp.float().numpy()
    rng = np.random.default_rng(8)
    cu = cq.numpy()
    for b in range(8):
        lq, lk = lens_q[b], lens_k[b]
        for h in rng.choice(32, 2, replace=False):
            kk = orc.paged_gather(kn, table[b].numpy(), lk, h // 4)
            vv = orc.paged_gather(vn, table[b].numpy(), lk, h // 4)
            for r0 in {0, max(0, lq - 64), int(rng.integers(0, lq))}:
                r1 = min(lq, r0 + 64)
                s0 = int(cu[b])
                o_ref, lse_ref, _, _ = orc.attention_dense(qn[s0 + r0:s0 + r1, h], kk, vv,
                                                           1 / math.sqrt(128), True, r0 + lk - lq)
                check_o(o[s0 + r0:s0 + r1, h], o_ref, "bf16")
                check_lse(lse[s0 + r0:s0 + r1, h], lse_ref, "bf16")


def test_bad_table_entry_is_reported():
    q, kp, vp, table, cq, sl = make_case([10, 10], [40, 40], 4, 2, 64, seed=9)
    table[1, 1] = kp.shape[0] + 5              # needed (tokens 16..31) and out of range
    ea.attn_prefill_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cq.cuda(), sl.cuda())
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
    assert ea.attn_get_device_status() == "ATTN_OK"   # read and cleared
