"""Packed (variable-length) bf16 prefill against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_varlen(lens_q, lens_k, d, causal, Hq=4, Hkv=2, seed=0):
    q, k, v, cq, ck = inputs.varlen_inputs(lens_q, lens_k, Hq, Hkv, d, seed=seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), causal=causal,
                                scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.prefill_varlen(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                        cq.numpy(), ck.numpy(), scale, causal)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_llm_book_packing(d, causal):
    """[LLM book] 10.3.8: lengths 3, 5, 2 packed as [0, 3, 8, 10]."""
    run_varlen([3, 5, 2], [3, 5, 2], d, causal, seed=1)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_mixed_lengths_with_empty_sequences(d, causal):
    lens = [1, 129, 0, 300, 17, 256]
    run_varlen(lens, lens, d, causal, Hq=8, Hkv=2, seed=2)


@pytest.mark.parametrize("d", [64, 128])
def test_chunked_prefill_bottom_right(d):
    """Fewer queries than keys: the queries are the last tokens (bottom-right
    causal), over several K/V tiles with a diagonal that crosses tiles."""
    run_varlen([1, 100, 130, 0, 64], [300, 100, 500, 17, 64], d, True, Hq=8, Hkv=4, seed=3)


@pytest.mark.parametrize("d", [64, 128])
def test_more_queries_than_keys(d):
    """Bottom-right causal with lq > lk: the first lq - lk rows see nothing."""
    o, lse = run_varlen([200, 5], [70, 9], d, True, seed=4)
    assert torch.isneginf(lse[:130]).all() and (o[:130] == 0).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B", [4096, 4097])
def test_many_sequences_sorted_list_and_fallback(d, B):
    """Each CTA sorts at most 4096 work units (a sequence's Q-tile position)
    into its item list; one more unit keeps the round-robin order.  Chunks of
    1 to 128 queries after 0 to 300 earlier keys give units of unequal cost,
    so the sort does reorder them; every 97th sequence has no queries."""
    g = np.random.default_rng(40 + B)
    lens_q = g.integers(1, 129, B)
    lens_q[::97] = 0
    lens_k = lens_q + g.integers(0, 301, B)
    run_varlen(lens_q.tolist(), lens_k.tolist(), d, True, Hq=1, Hkv=1, seed=5)


def test_more_positions_than_the_item_list_holds():
    """More positions per CTA than the 256-entry item list holds: the batch
    keeps the round-robin order.  At d = 128 a CTA per SM takes
    ceil(sequences x 16 heads / SMs) single-pair items (chunks of at most 128
    queries), so the batch is sized from this GPU's SM count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nseq, heads, list_items = 16 * sms + 100, 16, 256
    assert -(-nseq * heads // sms) > list_items
    g = np.random.default_rng(77)
    lens_q = g.integers(1, 129, nseq)
    lens_k = lens_q + g.integers(0, 65, nseq)
    run_varlen(lens_q.tolist(), lens_k.tolist(), 128, True, Hq=heads, Hkv=2, seed=8)


@pytest.mark.parametrize("causal", [False, True])
def test_no_keys_anywhere(causal):
    """total_k = 0: every row sees no key (O = 0, LSE = -inf)."""
    o, lse = run_varlen([3, 0, 200], [0, 0, 0], 64, causal, seed=9)
    assert (o == 0).all() and torch.isneginf(lse).all()


def test_no_queries_is_a_no_op():
    q, k, v, cq, ck = inputs.varlen_inputs([0, 0], [4, 5], 4, 2, 128, seed=10)
    o, lse = ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda())
    torch.cuda.synchronize()
    assert o.shape == (0, 4, 128) and lse.shape == (0, 4)
    assert ea.attn_get_device_status() == "ATTN_OK"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_dense_bitwise(d, causal):
    """Packed equal-length sequences take the same arithmetic as the dense
    [B, H, L, d] call: the outputs are bitwise identical."""
    B, H, L = 3, 4, 300
    q, k, v = inputs.prefill_inputs(B, H, H, L, L, d, "bf16", seed=5)
    o_d, lse_d = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(B * L, H, d).contiguous().cuda()
    cu = torch.arange(0, (B + 1) * L, L, dtype=torch.int32).cuda()
    o_v, lse_v = ea.attn_fwd_varlen(pack(q), pack(k), pack(v), cu, cu, L, L, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_d.permute(0, 2, 1, 3).reshape(B * L, H, d))
    assert torch.equal(lse_v, lse_d.permute(0, 2, 1).reshape(B * L, H))


def test_long_mixed_batch_sampled():
    """A serving-like mix (Hq 32, Hkv 8, d 128): 16 lengths from a seeded
    distribution up to 4096, checked on sampled (sequence, head, row block)
    triples; a row block starting at row r0 of a sequence with lq queries and
    lk keys sees keys j <= i + r0 + lk - lq (i its row within the block)."""
    g = torch.Generator().manual_seed(11)
    lens = torch.randint(1, 4097, (16,), generator=g).tolist()
    q, k, v, cq, ck = inputs.varlen_inputs(lens, lens, 32, 8, 128, seed=6)
    o, lse = ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o, lse = to_np(o), to_np(lse)
    rng = np.random.default_rng(7)
    cu = cq.numpy()
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    for b in range(len(lens)):
        s0, n = int(cu[b]), lens[b]
        for h in rng.choice(32, 2, replace=False):
            for r0 in {0, max(0, n - 64), int(rng.integers(0, n))}:
                r1 = min(n, r0 + 64)
                kh = h // 4
                o_ref, lse_ref, _, _ = orc.attention_dense(
                    qn[s0 + r0:s0 + r1, h], kn[s0:s0 + n, kh], vn[s0:s0 + n, kh],
                    1 / math.sqrt(128), True, r0)
                check_o(o[s0 + r0:s0 + r1, h], o_ref, "bf16")
                check_lse(lse[s0 + r0:s0 + r1, h], lse_ref, "bf16")


def test_bad_cu_seqlens_reports_and_touches_nothing():
    """A length past max_seqlen is reported (ATTN_ERR_BAD_INDEX); that
    sequence is skipped, the others are still right."""
    q, k, v, cq, ck = inputs.varlen_inputs([50, 40], [50, 40], 4, 2, 64, seed=8)
    o = torch.full_like(q.cuda(), 7.0)
    ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), max_seqlen_q=45,
                       max_seqlen_k=45, out=o)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_ERR_BAD_INDEX"
    assert (o[:50] == 7.0).all()        # sequence 0 (50 > 45) left unwritten
    o_ref, _ = orc.prefill_varlen(q.float().numpy()[50:], k.float().numpy()[50:],
                                  v.float().numpy()[50:], [0, 40], [0, 40], 0.125, False)
    check_o(to_np(o[50:]), o_ref, "bf16")
