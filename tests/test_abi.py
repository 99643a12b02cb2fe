"""CPU-only checks of the C ABI: the library loads, exports every declared
symbol, rejects invalid arguments on the host before launching anything, and
its split planner agrees bit-exactly with the oracle's reading."""
import ctypes
import os
import re

import numpy as np
import pytest

import exact_attention_sm_gb300 as ea
from oracle import attention as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ea.lib()
    names = declared_symbols()
    assert set(names) == set(ea.SIGNATURES), names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.attn_version() >= 100


def test_status_strings():
    for code, name in ea.STATUS.items():
        assert ea.lib().attn_status_string(code).decode() == name


def fwd(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Lq=8, Lk=8, d=64,
                causal=0, scale=0.125, dtype=ea.ATTN_BF16)
    args.update(kw)
    return ea.lib().attn_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                             args["Hq"], args["Hkv"], args["Lq"], args["Lk"], args["d"],
                             args["causal"], args["scale"], args["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(B=0), 1), (dict(Lk=0), 1), (dict(Hkv=3), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(dtype=7), 1),
    (dict(d=96), 2), (dict(causal=1, Lq=4), 2), (dict(q=MISALIGNED), 1),
])
def test_attn_fwd_rejects_on_host(kw, status):
    assert fwd(**kw) == status


def dec(**kw):
    lens = (ctypes.c_int32 * 2)(100, 40)
    args = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, lens=FAKE, lens_host=ctypes.cast(lens, ctypes.c_void_p),
                page=16, splits=4, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, d=128, max_pages=7,
                num_pages=14, scale=0.1, ws=None, ws_bytes=0, dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_decode_paged(a["q"], a["k"], a["v"], a["table"], a["lens"], a["lens_host"],
                                      a["page"], a["splits"], a["o"], a["lse"], a["B"], a["Hq"],
                                      a["Hkv"], a["d"], a["max_pages"], a["num_pages"], a["scale"],
                                      a["ws"], a["ws_bytes"], a["dtype"], None)


def test_decode_rejects_on_host():
    assert dec(q=None) == 1
    assert dec(table=None) == 1
    assert dec(Hkv=3) == 1
    assert dec(splits=-1) == 1
    assert dec(page=32) == 2
    assert dec(d=96) == 2
    assert dec(d=64) == 3                 # d = 64 is served; here the split plan needs a workspace
    assert dec(dtype=ea.ATTN_F32) == 2
    assert dec(max_pages=2) == 1          # a length exceeds max_pages * page_size
    assert dec() == 3                     # 4 forced segments need a workspace
    need = ea.attn_decode_workspace_bytes(2, 8, 128, 4)
    assert need >= 2 * 8 * 4 * 129 * 4
    assert dec(ws=ctypes.c_void_p(0x20000), ws_bytes=need - 1) == 3
    assert dec(ws=ctypes.c_void_p(0x20010), ws_bytes=need) == 3  # not 256-byte aligned
    assert ea.attn_decode_workspace_bytes(2, 8, 128, 1) == 0


def test_merge_rejects_on_host():
    m = ea.lib().attn_merge_states
    assert m(None, FAKE, 4, 2, 128, FAKE, None, ea.ATTN_BF16, None) == 1
    assert m(FAKE, FAKE, 4, 2, 6, FAKE, None, ea.ATTN_BF16, None) == 1
    assert m(FAKE, FAKE, 0, 2, 128, FAKE, None, ea.ATTN_BF16, None) == 1
    assert m(FAKE, FAKE, 4, 2, 1024, FAKE, None, ea.ATTN_BF16, None) == 2
    assert m(MISALIGNED, FAKE, 4, 2, 128, FAKE, None, ea.ATTN_BF16, None) == 1


def test_planner_matches_oracle_bit_exact():
    rng = np.random.default_rng(7)
    cases = [([16384, 16384], 8, 132), ([32768], 8, 132), ([1024] * 256, 8, 456),
             ([0], 8, 456), ([5, 0, 17], 1, 10)]
    for _ in range(300):
        b = int(rng.integers(1, 9))
        hi = int(rng.choice([50, 5000, 140000]))
        cases.append((rng.integers(0, hi, size=b).tolist(), int(rng.choice([1, 2, 4, 8])),
                      int(rng.choice([132, 152, 304, 456, 608]))))
    for lens, hkv, slots in cases:
        for forced in (0, 1, 2, 5, 64):
            chunk, smax = ea.attn_decode_plan(lens, hkv, 16, forced, slots)
            o_chunk, o_splits = orc.plan_splits(lens, hkv, slots, 16, forced)
            assert chunk == o_chunk[0], (lens, hkv, slots, forced)
            assert smax == max(o_splits), (lens, hkv, slots, forced)


def test_planner_config5_lengths_fill_the_gpu():
    from exact_attention_sm_gb300 import inputs
    lens = inputs.decode_lengths_uniform(4, 4096, 131072, seed=2)
    chunk, smax = ea.attn_decode_plan(lens, 8, 16, 0, 152 * 3)
    units = 8 * sum(max(1, -(-n // chunk)) for n in lens)
    assert units >= 152 and chunk % 16 == 0


def test_selftest_rejects_bad_limits_on_host():
    assert ea.lib().attn_selftest_wait_timeout(0, None) == 1
    assert ea.lib().attn_selftest_wait_timeout(20000, None) == 1


def casc(**kw):
    lens = (ctypes.c_int32 * 2)(100, 0)
    args = dict(q=FAKE, pk=FAKE, pv=FAKE, P=300, k=FAKE, v=FAKE, table=FAKE, lens=FAKE,
                lens_host=ctypes.cast(lens, ctypes.c_void_p), page=16, splits=0, o=FAKE, lse=None,
                B=2, Hq=8, Hkv=2, d=128, max_pages=7, num_pages=14, scale=0.1, ws=None, ws_bytes=0,
                dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_decode_cascade(a["q"], a["pk"], a["pv"], a["P"], a["k"], a["v"], a["table"],
                                        a["lens"], a["lens_host"], a["page"], a["splits"], a["o"],
                                        a["lse"], a["B"], a["Hq"], a["Hkv"], a["d"], a["max_pages"],
                                        a["num_pages"], a["scale"], a["ws"], a["ws_bytes"],
                                        a["dtype"], None)


def test_cascade_rejects_on_host():
    assert casc(q=None) == 1
    assert casc(pk=None) == 1
    assert casc(lens_host=None) == 1          # the host lengths fix the plan
    assert casc(P=0) == 1
    assert casc(Hkv=3) == 1
    assert casc(splits=-1) == 1
    assert casc(d=96) == 2
    assert casc(d=64) != 2                    # d = 64 is served
    assert casc(page=32) == 2
    assert casc(dtype=ea.ATTN_F32) == 2
    assert casc(pk=MISALIGNED) == 1
    assert casc(max_pages=6) == 1             # suffix length 100 > 6 * 16


def prefix_chunks_rule(P, rows, Hkv, slots):
    """The documented rule: among divisors c of P with chunks of >= 128
    tokens (or c = 1), minimise waves x (2 + tiles per chunk); ties to fewer."""
    pairs = -(-rows // 256)
    ok = [c for c in range(1, max(1, P // 128) + 1) if P % c == 0]
    cost = lambda c: -(-Hkv * pairs * c // slots) * (2 + -(-(P // c) // 128))
    return min(ok, key=lambda c: (cost(c), c))


@pytest.mark.parametrize("B,Hq,Hkv,P,slots", [(64, 32, 8, 4096, 152), (4, 32, 8, 300, 152),
                                              (2, 8, 2, 100, 152), (256, 32, 8, 1000, 16),
                                              (1, 4, 1, 131072, 152), (7, 6, 3, 2560, 152)])
def test_cascade_plan(B, Hq, Hkv, P, slots):
    lens = [0, 5, 300, 16][:B] + [17] * max(0, B - 4)
    pc, sc, ss = ea.attn_cascade_plan(B, Hq, Hkv, P, lens, 16, 0, slots, 456)
    assert pc == prefix_chunks_rule(P, B * (Hq // Hkv), Hkv, slots)
    assert P % pc == 0
    assert (sc, ss) == ea.attn_decode_plan(lens, Hkv, 16, 0, 456)
    rows = B * Hq
    r = lambda x: -(-x // 256) * 256
    for d in (64, 128):
        want = (r(rows * d * 2) + r(rows * pc * d * 2) + r(rows * pc * 4) + r(rows * ss * d * 4)
                + r(rows * ss * 4))
        assert ea.attn_cascade_workspace_bytes(B, Hq, d, pc, ss) == want


def varlen(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cq=FAKE, ck=FAKE, B=3, mq=5, mk=5, tq=10,
                tk=10, Hq=4, Hkv=2, d=64, causal=1, scale=0.125, dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"],
                                    a["B"], a["mq"], a["mk"], a["tq"], a["tk"], a["Hq"], a["Hkv"],
                                    a["d"], a["causal"], a["scale"], a["dtype"], None)


def test_varlen_rejects_on_host():
    assert varlen(q=None) == 1
    assert varlen(o=None) == 1
    assert varlen(cq=None) == 1
    assert varlen(k=None) == 1                # keys present but no k
    assert varlen(B=0) == 1
    assert varlen(Hkv=3) == 1
    assert varlen(mq=0) == 1
    assert varlen(tq=-1) == 1
    assert varlen(scale=0.0) == 1
    assert varlen(scale=float("nan")) == 1
    assert varlen(q=MISALIGNED) == 1
    assert varlen(cq=ctypes.c_void_p(0x10002)) == 1   # cu_seqlens must be 4-byte aligned
    assert varlen(d=96) == 2
    assert varlen(dtype=ea.ATTN_F32) == 2


def test_varlen_without_queries_is_a_no_op():
    """total_q = 0 (every sequence empty) succeeds without a launch, NULLs allowed."""
    assert varlen(q=None, k=None, v=None, o=None, cq=None, ck=None, tq=0, tk=0) == 0


def paged(**kw):
    args = dict(q=FAKE, kp=FAKE, vp=FAKE, table=FAKE, cq=FAKE, sk=FAKE, o=FAKE, lse=None, B=2, mq=8,
                mk=40, tq=12, Hq=4, Hkv=2, d=128, page=16, max_pages=4, num_pages=8, causal=1,
                scale=0.1, dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_prefill_paged(a["q"], a["kp"], a["vp"], a["table"], a["cq"], a["sk"],
                                       a["o"], a["lse"], a["B"], a["mq"], a["mk"], a["tq"], a["Hq"],
                                       a["Hkv"], a["d"], a["page"], a["max_pages"],
                                       a["num_pages"], a["causal"], a["scale"], a["dtype"], None)


def test_prefill_paged_rejects_on_host():
    assert paged(q=None) == 1
    assert paged(table=None) == 1
    assert paged(sk=None) == 1
    assert paged(B=0) == 1
    assert paged(Hkv=3) == 1
    assert paged(mq=0) == 1
    assert paged(mk=65) == 1                  # longer than max_pages * 16
    assert paged(num_pages=0) == 1
    assert paged(scale=-1.0) == 1
    assert paged(kp=MISALIGNED) == 1
    assert paged(table=ctypes.c_void_p(0x10002)) == 1
    assert paged(d=96) == 2
    assert paged(page=24) == 2                # pages are a power of two ...
    assert paged(page=256) == 2               # ... of at most 128 tokens
    assert paged(page=4, mk=17) == 1          # longer than max_pages * 4
    assert paged(dtype=ea.ATTN_F32) == 2
    assert paged(tq=0, q=None, o=None) == 0   # no query rows: no launch


def bsr(**kw):
    args = dict(q=FAKE, kb=FAKE, vb=FAKE, indptr=FAKE, indices=FAKE, nnz=16, cq=FAKE, sk=FAKE,
                o=FAKE, lse=None, B=3, mq=29, mk=29, tq=46, Hq=4, Hkv=2, d=64, block=4,
                num_blocks=24, causal=1, scale=0.1, dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_prefill_bsr(a["q"], a["kb"], a["vb"], a["indptr"], a["indices"], a["nnz"],
                                     a["cq"], a["sk"], a["o"], a["lse"], a["B"], a["mq"], a["mk"],
                                     a["tq"], a["Hq"], a["Hkv"], a["d"], a["block"],
                                     a["num_blocks"], a["causal"], a["scale"], a["dtype"], None)


def test_prefill_bsr_rejects_on_host():
    """[Lecture 4] 5.2 block-sparse rows: argument checks before any launch."""
    assert bsr(q=None) == 1
    assert bsr(indptr=None) == 1
    assert bsr(indices=None) == 1             # blocks listed but no indices
    assert bsr(sk=None) == 1
    assert bsr(B=0) == 1
    assert bsr(Hkv=3) == 1
    assert bsr(nnz=-1) == 1
    assert bsr(num_blocks=0) == 1
    assert bsr(scale=float("inf")) == 1
    assert bsr(kb=MISALIGNED) == 1
    assert bsr(indices=ctypes.c_void_p(0x10002)) == 1
    assert bsr(d=96) == 2
    assert bsr(block=3) == 2
    assert bsr(block=256) == 2
    assert bsr(mk=65) == 2                    # longer than all 16 blocks of 4 tokens together
    assert bsr(dtype=ea.ATTN_F32) == 2
    assert bsr(tq=0, q=None, o=None) == 0     # no query rows: no launch


def bwd(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1,
                Hq=4, Hkv=2, Lq=64, Lk=64, d=128, causal=1, scale=0.1, ws=FAKE, ws_bytes=4096,
                dtype=ea.ATTN_BF16)
    args.update(kw)
    a = args
    return ea.lib().attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                             a["dv"], a["B"], a["Hq"], a["Hkv"], a["Lq"], a["Lk"], a["d"],
                             a["causal"], a["scale"], a["ws"], a["ws_bytes"], a["dtype"], None)


def test_bwd_rejects_on_host():
    assert ea.lib().attn_bwd_workspace_bytes(2, 4, 100) == 8448   # 2 x 8 heads x 128 padded rows x 4 B, + counters
    assert bwd(q=None) == 1
    assert bwd(dv=None) == 1
    assert bwd(Hkv=3) == 1
    assert bwd(Lk=0) == 1
    assert bwd(scale=0.0) == 1
    assert bwd(dk=MISALIGNED) == 1
    assert bwd(d=96) == 2
    assert bwd(dtype=ea.ATTN_F32) == 2
    assert bwd(Lk=65) == 2                    # causal needs Lq == Lk
    assert bwd(ws=None) == 3
    assert bwd(ws_bytes=100) == 3
    assert bwd(ws=ctypes.c_void_p(0x10010)) == 3


def parse_balanced_plan(plan, B, G, ctas):
    U = ctas + B * G
    n = plan[0]
    cta_off = plan[1:1 + ctas + 1]
    cu0 = 1 + ctas + 1
    cta_units = plan[cu0:cu0 + U]
    u0 = cu0 + U
    units = [tuple(plan[u0 + 4 * u:u0 + 4 * u + 4]) for u in range(n)]
    per_cta = [cta_units[cta_off[c]:cta_off[c + 1]] for c in range(ctas)]
    s0 = u0 + 4 * U
    seg_off = plan[s0:s0 + B * G + 1]
    return units, per_cta, seg_off


def test_balanced_schedule_matches_oracle_bit_exact():
    rng = np.random.default_rng(43)
    cases = [([16384, 16384], 32, 8, 132), ([0, 5, 17], 8, 2, 10), ([1024] * 256, 32, 8, 456)]
    for _ in range(60):
        b = int(rng.integers(1, 9))
        hkv = int(rng.choice([1, 2, 8]))
        hq = hkv * int(rng.choice([1, 4, 6, 8]))
        cases.append((rng.integers(0, 140000, size=b).tolist(), hq, hkv,
                      int(rng.choice([8, 132, 456]))))
    for lens, hq, hkv, ctas in cases:
        G = hkv * ((hq // hkv + 3) // 4)
        plan = ea.attn_decode_schedule_host(lens, hq, hkv, ctas)
        units, per_cta, seg_off = parse_balanced_plan(plan, len(lens), G, ctas)
        o_units, o_cta = orc.plan_balanced(lens, G, ctas, 16)
        assert units == o_units, (lens, hq, hkv, ctas)
        assert per_cta == o_cta
        # the units of (request, group) i are seg_off[i] .. seg_off[i + 1] - 1, in token order
        for i in range(len(lens) * G):
            segs = units[seg_off[i]:seg_off[i + 1]]
            assert all(s[:2] == (i // G, i % G) for s in segs)


def test_balanced_rejects_on_host():
    lens = (ctypes.c_int32 * 2)(100, 0)
    lh = ctypes.cast(lens, ctypes.c_void_p)
    assert ea.lib().attn_decode_schedule(None, 2, 8, 2, 16, 10, FAKE, 1 << 20, None) == 1
    assert ea.lib().attn_decode_schedule(lh, 2, 8, 3, 16, 10, FAKE, 1 << 20, None) == 1
    assert ea.lib().attn_decode_schedule(lh, 2, 8, 2, 16, 10, None, 0, None) == 3
    assert ea.lib().attn_decode_schedule(lh, 2, 8, 2, 16, 10, FAKE, 64, None) == 3
    bad = (ctypes.c_int32 * 2)(100, -1)
    assert ea.lib().attn_decode_schedule(ctypes.cast(bad, ctypes.c_void_p), 2, 8, 2, 16, 10, FAKE,
                                         1 << 20, None) == 1
    bd = lambda **kw: ea.lib().attn_decode_paged_balanced(
        kw.get("q", FAKE), FAKE, FAKE, FAKE, FAKE, kw.get("page", 16), FAKE, None, 2, 8, 2,
        kw.get("d", 128), 7, 14, 0.1, 10, kw.get("ws", FAKE), kw.get("wsb", 1 << 20),
        kw.get("dtype", ea.ATTN_BF16), None)
    assert bd(q=None) == 1
    assert bd(q=MISALIGNED) == 1
    assert bd(d=64) == 2
    assert bd(page=32) == 2
    assert bd(dtype=ea.ATTN_F32) == 2
    assert bd(ws=None) == 3
    assert bd(wsb=100) == 3
    assert ea.lib().attn_decode_sched_workspace_bytes(2, 8, 2, 128, 10) > 0
