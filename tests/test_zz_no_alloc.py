"""attn_decode_paged_noalloc against the float64 oracle and attn_decode_paged.

The allocation-free entry point serves callers that may not allocate device
memory (it uses a fixed scratch array inside the library instead of a
caller-provided workspace).  Its output must match the oracle's paged decode
within the bf16 tolerances the other parity tests use, and the regular entry
point (explicit workspace) within the same tolerances, on two calls in a row:
the scratch keeps the previous call's contents, so the second call checks
that nothing stale leaks in.  This file is collected last so a failure here
cannot hide the other tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import BF16_LSE, BF16_O_MAX, BF16_O_MEAN, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_noalloc(q, kp, vp, table, sl, lens, num_splits, o, lse):
    B, Hq, d = q.shape
    num_pages, page, Hkv, _ = kp.shape
    host = (ctypes.c_int32 * B)(*lens)
    return ea.lib().attn_decode_paged_noalloc(
        _p(q), _p(kp), _p(vp), _p(table), _p(sl), ctypes.cast(host, ctypes.c_void_p), page,
        num_splits, _p(o), _p(lse), B, Hq, Hkv, d, table.shape[1], num_pages,
        1.0 / math.sqrt(d), ea.ATTN_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def close(got_o, got_l, ref_o, ref_l):
    err = (got_o.float() - ref_o.float()).abs()
    assert err.max().item() <= BF16_O_MAX and err.mean().item() <= BF16_O_MEAN
    fin = torch.isfinite(ref_l)
    assert torch.equal(torch.isneginf(got_l), torch.isneginf(ref_l))
    if fin.any():
        assert (got_l[fin] - ref_l[fin]).abs().max().item() <= BF16_LSE


@pytest.mark.parametrize("lens,num_splits", [
    ([1, 17, 1000, 4096], 0),
    ([1, 17, 1000, 4096], 5),
    ([0, 70000, 333, 123457], 0),
])
def test_noalloc_matches_workspace_entry_point(lens, num_splits):
    host = inputs.decode_inputs(lens, 32, 8, 128, seed=7)
    q, kp, vp, table, sl = (t.cuda() for t in host)
    f = lambda t: t.float().numpy()
    orc_o, orc_l = orc.decode_paged(f(host[0]), f(host[1]), f(host[2]), host[3].numpy(), lens,
                                    1.0 / math.sqrt(128))
    ref_o, ref_l = ea.attn_decode_paged(q, kp, vp, table, sl, seq_lens_host=lens,
                                        num_splits=num_splits)
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), device="cuda")
        st = call_noalloc(q, kp, vp, table, sl, lens, num_splits, o, lse)
        assert st == 0, ea.STATUS.get(st)
        torch.cuda.synchronize()
        assert ea.attn_get_device_status() == "ATTN_OK"
        check_o(to_np(o), orc_o, "bf16")
        check_lse(to_np(lse), orc_l, "bf16")
        close(o, lse, ref_o, ref_l)


def test_noalloc_rejects_plans_beyond_its_scratch():
    lens = [4096] * 64
    q, kp, vp, table, sl = (t.cuda() for t in inputs.decode_inputs(lens, 64, 8, 128, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty(64, 64, device="cuda")
    # 64 segments x 64 requests x 64 heads x 129 floats is far beyond the scratch
    assert ea.attn_decode_workspace_bytes(64, 64, 128, 64) > (8 << 20)
    assert call_noalloc(q, kp, vp, table, sl, lens, 64, o, lse) == 3
