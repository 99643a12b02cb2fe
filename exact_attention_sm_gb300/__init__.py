"""GB300 (sm_103a) exact attention: thin Python binding over libattn.so.

Every function below only marshals arguments (torch tensors -> device
pointers and sizes) and calls the C ABI declared in ``include/attn.h``; all
arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_F32, ATTN_BF16 = 0, 1
STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
    4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_DEVICE_TIMEOUT", 6: "ATTN_ERR_BAD_INDEX",
}

# Every symbol include/attn.h declares, with its ctypes signature.
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                             _I, _P]),
    "attn_prefill_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                _I, _I, _I, _F, _I, _P]),
    "attn_prefill_bsr": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                              _I, _I, _I, _F, _I, _P]),
    "attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ,
                      _I, _P]),
    "attn_decode_sched_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_decode_schedule": (_I, [_P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "attn_decode_schedule_host": (_I, [_P, _I, _I, _I, _I, _I, _P, _SZ]),
    "attn_decode_paged_balanced": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                                        _I, _P, _SZ, _I, _P]),
    "attn_decode_plan": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "attn_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                               _P, _SZ, _I, _P]),
    "attn_decode_paged_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I,
                                       _I, _F, _I, _P]),
    "attn_merge_states": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _P]),
    "attn_cascade_plan": (_I, [_I, _I, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P]),
    "attn_cascade_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_decode_cascade": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I,
                                 _I, _I, _I, _F, _P, _SZ, _I, _P]),
    "attn_get_device_status": (_I, [_P]),
    "attn_selftest_wait_timeout": (_I, [_I, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_version": (_I, []),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def lib():
    """The loaded libattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m exact_attention_sm_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype, fn.argtypes = res, args
        _lib = h
    return _lib


def _check(status, where):
    if status != 0:
        raise AttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name):
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def attn_fwd(q, k, v, causal=False, scale=None, out=None, lse=None, want_lse=True, stream=None):
    """Prefill attention. q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] -> (o [B,Hq,Lq,d], lse [B,Hq,Lq] fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Lq, Lk, d,
                        int(bool(causal)), float(scale), _dtype_code(q), _stream(stream))
    _check(st, "attn_fwd")
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=None, max_seqlen_k=None,
                    causal=False, scale=None, out=None, lse=None, want_lse=True, stream=None):
    """Packed prefill. q [total_q,Hq,d], k/v [total_k,Hkv,d] bf16; cu_seqlens_q/k int32 [B+1] on
    the device. Causal is aligned bottom-right. Returns (o [total_q,Hq,d], lse [total_q,Hq])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cu_seqlens_q, "cu_seqlens_q"),
                 (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, n)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if max_seqlen_q is None or max_seqlen_k is None:
        cq, ck = cu_seqlens_q.cpu(), cu_seqlens_k.cpu()
        max_seqlen_q = int((cq[1:] - cq[:-1]).max()) if max_seqlen_q is None else max_seqlen_q
        max_seqlen_k = int((ck[1:] - ck[:-1]).max()) if max_seqlen_k is None else max_seqlen_k
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(total_q, Hq, dtype=torch.float32, device=q.device)
    st = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                               _ptr(cu_seqlens_k), B, max(1, int(max_seqlen_q)),
                               max(1, int(max_seqlen_k)), total_q, total_k, Hq, Hkv, d,
                               1 if causal else 0, float(scale), _dtype_code(q), _stream(stream))
    _check(st, "attn_fwd_varlen")
    return out, lse


def attn_prefill_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seq_lens_k,
                       max_seqlen_q=None, max_seqlen_k=None, causal=False, scale=None, out=None,
                       lse=None, want_lse=True, stream=None):
    """Chunked prefill against a paged cache. q [total_q,Hq,d] bf16 packed by cu_seqlens_q
    (int32 [B+1], device); k_pages/v_pages [num_pages,page_size,Hkv,d] bf16 (page_size a
    power of two, 1..128); block_table int32 [B,max_pages]; seq_lens_k int32 [B] (device).
    Causal is aligned bottom-right. Returns (o [total_q,Hq,d], lse [total_q,Hq])."""
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"), (block_table, "block_table"),
                 (cu_seqlens_q, "cu_seqlens_q"), (seq_lens_k, "seq_lens_k")):
        _need(t, n)
    for t in (block_table, cu_seqlens_q, seq_lens_k):
        if t.dtype != torch.int32:
            raise TypeError("block_table, cu_seqlens_q and seq_lens_k must be int32")
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    B = cu_seqlens_q.numel() - 1
    if max_seqlen_q is None:
        cq = cu_seqlens_q.cpu()
        max_seqlen_q = int((cq[1:] - cq[:-1]).max()) if B > 0 else 1
    if max_seqlen_k is None:
        max_seqlen_k = int(seq_lens_k.max()) if B > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(total_q, Hq, dtype=torch.float32, device=q.device)
    st = lib().attn_prefill_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                  _ptr(cu_seqlens_q), _ptr(seq_lens_k), _ptr(out), _ptr(lse), B,
                                  max(1, int(max_seqlen_q)), int(max_seqlen_k), total_q, Hq, Hkv, d,
                                  page_size, block_table.shape[1], num_pages, 1 if causal else 0,
                                  float(scale), _dtype_code(q), _stream(stream))
    _check(st, "attn_prefill_paged")
    return out, lse


def attn_prefill_bsr(q, k_blocks, v_blocks, kv_indptr, kv_indices, cu_seqlens_q, seq_lens_k,
                     max_seqlen_q=None, max_seqlen_k=None, causal=False, scale=None, out=None,
                     lse=None, want_lse=True, stream=None):
    """Prefill against a KV cache in block-sparse-row form. q [total_q,Hq,d] bf16 packed by
    cu_seqlens_q; k_blocks/v_blocks [num_blocks,block_size,Hkv,d] bf16; request b's blocks
    are kv_indices[kv_indptr[b]:kv_indptr[b+1]] (int32, device); seq_lens_k int32 [B].
    Returns (o [total_q,Hq,d], lse [total_q,Hq])."""
    for t, n in ((q, "q"), (k_blocks, "k_blocks"), (v_blocks, "v_blocks"),
                 (kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"),
                 (cu_seqlens_q, "cu_seqlens_q"), (seq_lens_k, "seq_lens_k")):
        _need(t, n)
    for t in (kv_indptr, kv_indices, cu_seqlens_q, seq_lens_k):
        if t.dtype != torch.int32:
            raise TypeError("kv_indptr, kv_indices, cu_seqlens_q and seq_lens_k must be int32")
    total_q, Hq, d = q.shape
    num_blocks, block_size, Hkv, _ = k_blocks.shape
    B = cu_seqlens_q.numel() - 1
    if max_seqlen_q is None:
        cq = cu_seqlens_q.cpu()
        max_seqlen_q = int((cq[1:] - cq[:-1]).max()) if B > 0 else 1
    if max_seqlen_k is None:
        max_seqlen_k = int(seq_lens_k.max()) if B > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(total_q, Hq, dtype=torch.float32, device=q.device)
    st = lib().attn_prefill_bsr(_ptr(q), _ptr(k_blocks), _ptr(v_blocks), _ptr(kv_indptr),
                                _ptr(kv_indices), kv_indices.numel(), _ptr(cu_seqlens_q),
                                _ptr(seq_lens_k), _ptr(out), _ptr(lse), B,
                                max(1, int(max_seqlen_q)), int(max_seqlen_k), total_q, Hq, Hkv, d,
                                block_size, num_blocks, 1 if causal else 0, float(scale),
                                _dtype_code(q), _stream(stream))
    _check(st, "attn_prefill_bsr")
    return out, lse


def attn_bwd(q, k, v, o, lse, d_o, causal=False, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Backward of attn_fwd: q, o, d_o [B,Hq,Lq,d], k, v [B,Hkv,Lk,d] bf16, lse [B,Hq,Lq] fp32.
    Returns (dq, dk, dv) in bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (d_o, "d_o")):
        _need(t, n)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(lib().attn_bwd_workspace_bytes(B, Hq, Lq), dtype=torch.uint8,
                                device=q.device)
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, d, 1 if causal else 0,
                        float(scale), _ptr(workspace), workspace.numel(), _dtype_code(q),
                        _stream(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_decode_schedule(seq_lens_host, num_heads, num_kv_heads, workspace, page_size=16,
                         num_ctas=0, stream=None):
    """Load-balanced plan for attn_decode_paged_balanced, written into `workspace`."""
    lens = (ctypes.c_int32 * len(seq_lens_host))(*[int(x) for x in seq_lens_host])
    st = lib().attn_decode_schedule(ctypes.cast(lens, ctypes.c_void_p), len(seq_lens_host),
                                    int(num_heads), int(num_kv_heads), int(page_size),
                                    int(num_ctas), _ptr(workspace), workspace.numel(),
                                    _stream(stream))
    _check(st, "attn_decode_schedule")


def attn_decode_schedule_host(seq_lens_host, num_heads, num_kv_heads, num_ctas, page_size=16):
    """The same plan on the host: a list of int32 (layout documented in attn.h / api.cpp)."""
    B = len(seq_lens_host)
    G = num_kv_heads * ((num_heads // num_kv_heads + 3) // 4)
    U = num_ctas + B * G
    n = 1 + (num_ctas + 1) + U + 4 * U + (B * G + 1) + U
    lens = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens_host])
    out = (ctypes.c_int32 * n)()
    st = lib().attn_decode_schedule_host(ctypes.cast(lens, ctypes.c_void_p), B, int(num_heads),
                                         int(num_kv_heads), int(page_size), int(num_ctas),
                                         ctypes.cast(out, ctypes.c_void_p), n)
    _check(st, "attn_decode_schedule_host")
    return list(out)


def attn_decode_paged_balanced(q, k_pages, v_pages, block_table, seq_lens, workspace, out=None,
                               lse=None, want_lse=True, scale=None, num_ctas=0, stream=None):
    """Fixed-grid decode following the plan in `workspace` (attn_decode_schedule)."""
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"),
                 (block_table, "block_table"), (seq_lens, "seq_lens"), (workspace, "workspace")):
        _need(t, n)
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    st = lib().attn_decode_paged_balanced(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                          _ptr(seq_lens), page_size, _ptr(out), _ptr(lse), B, Hq,
                                          Hkv, d, block_table.shape[1], num_pages, float(scale),
                                          int(num_ctas), _ptr(workspace), workspace.numel(),
                                          _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_paged_balanced")
    return out, lse


def attn_decode_plan(seq_lens_host, num_kv_heads, page_size=16, num_splits=0, slots=0):
    """Host planner: returns (chunk, max_splits) for the given context lengths."""
    lens = (ctypes.c_int32 * len(seq_lens_host))(*[int(x) for x in seq_lens_host])
    chunk, smax = ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().attn_decode_plan(ctypes.cast(lens, ctypes.c_void_p), len(seq_lens_host),
                                int(num_kv_heads), int(page_size), int(num_splits), int(slots),
                                ctypes.byref(chunk), ctypes.byref(smax))
    _check(st, "attn_decode_plan")
    return chunk.value, smax.value


def attn_decode_workspace_bytes(B, Hq, d, max_splits):
    return int(lib().attn_decode_workspace_bytes(int(B), int(Hq), int(d), int(max_splits)))


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, seq_lens_host=None,
                      num_splits=0, scale=None, out=None, lse=None, workspace=None,
                      want_lse=True, stream=None):
    """Paged GQA decode. q [B,Hq,d]; k/v_pages [num_pages,page,Hkv,d]; block_table int32
    [B,max_pages]; seq_lens int32 [B] on the device; seq_lens_host: list/array or None.
    Allocates the split workspace when none is given. Returns (o [B,Hq,d], lse [B,Hq])."""
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"),
                 (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    host_arr = None
    if seq_lens_host is not None:
        host_arr = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens_host])
    if workspace is None and num_splits != 1:
        if seq_lens_host is None:
            seq_lens_host = seq_lens.cpu().tolist()
        _, smax = attn_decode_plan(seq_lens_host, Hkv, page_size, num_splits)
        nbytes = attn_decode_workspace_bytes(B, Hq, d, smax)
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
        None if host_arr is None else ctypes.cast(host_arr, ctypes.c_void_p), page_size,
        int(num_splits), _ptr(out), _ptr(lse), B, Hq, Hkv, d, block_table.shape[1], num_pages,
        float(scale), _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_paged")
    return out, lse


def attn_cascade_plan(B, Hq, Hkv, prefix_len, suffix_lens_host, page_size=16, num_splits=0,
                      prefix_slots=0, suffix_slots=0):
    """Cascade plan: (prefix_chunks, suffix_chunk, suffix_splits); slots <= 0 query the device."""
    arr = (ctypes.c_int32 * B)(*[int(x) for x in suffix_lens_host])
    pc, sc, ss = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().attn_cascade_plan(B, Hq, Hkv, int(prefix_len), ctypes.cast(arr, ctypes.c_void_p),
                                 page_size, int(num_splits), int(prefix_slots), int(suffix_slots),
                                 ctypes.byref(pc), ctypes.byref(sc), ctypes.byref(ss))
    _check(st, "attn_cascade_plan")
    return pc.value, sc.value, ss.value


def attn_cascade_workspace_bytes(B, Hq, d, prefix_chunks, suffix_splits):
    return lib().attn_cascade_workspace_bytes(B, Hq, d, prefix_chunks, suffix_splits)


def attn_decode_cascade(q, prefix_k, prefix_v, k_pages, v_pages, block_table, seq_lens,
                        seq_lens_host=None, num_splits=0, scale=None, out=None, lse=None,
                        workspace=None, want_lse=True, stream=None):
    """Shared-prefix decode. q [B,Hq,d]; prefix_k/v [Hkv,P,d]; the suffixes in the paged cache
    (seq_lens = suffix lengths). Allocates the workspace when none is given.
    Returns (o [B,Hq,d], lse [B,Hq])."""
    for t, n in ((q, "q"), (prefix_k, "prefix_k"), (prefix_v, "prefix_v"), (k_pages, "k_pages"),
                 (v_pages, "v_pages"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    prefix_len = prefix_k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if seq_lens_host is None:
        seq_lens_host = seq_lens.cpu().tolist()
    if workspace is None:
        pc, _, ss = attn_cascade_plan(B, Hq, Hkv, prefix_len, seq_lens_host, page_size, num_splits)
        workspace = torch.empty(attn_cascade_workspace_bytes(B, Hq, d, pc, ss), dtype=torch.uint8,
                                device=q.device)
    host_arr = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens_host])
    st = lib().attn_decode_cascade(
        _ptr(q), _ptr(prefix_k), _ptr(prefix_v), prefix_len, _ptr(k_pages), _ptr(v_pages),
        _ptr(block_table), _ptr(seq_lens), ctypes.cast(host_arr, ctypes.c_void_p), page_size,
        int(num_splits), _ptr(out), _ptr(lse), B, Hq, Hkv, d, block_table.shape[1], num_pages,
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_cascade")
    return out, lse


def attn_merge_states(o_parts, lse_parts, out_dtype=torch.bfloat16, out=None, lse=None,
                      want_lse=True, stream=None):
    """LSE merge. o_parts [rows,S,d] fp32, lse_parts [rows,S] fp32 -> (o [rows,d], lse [rows])."""
    _need(o_parts, "o_parts")
    _need(lse_parts, "lse_parts")
    rows, S, d = o_parts.shape
    if out is None:
        out = torch.empty(rows, d, dtype=out_dtype, device=o_parts.device)
    if lse is None and want_lse:
        lse = torch.empty(rows, dtype=torch.float32, device=o_parts.device)
    st = lib().attn_merge_states(_ptr(o_parts), _ptr(lse_parts), rows, S, d, _ptr(out), _ptr(lse),
                                 _dtype_code(out), _stream(stream))
    _check(st, "attn_merge_states")
    return out, lse


def attn_get_device_status(stream=None):
    """Reads and clears the device status word; returns the status name."""
    return STATUS.get(lib().attn_get_device_status(_stream(stream)), "?")


def attn_selftest_wait_timeout(limit_ms=200, stream=None):
    """Runs the bounded-wait self-test kernel (see include/attn.h)."""
    _check(lib().attn_selftest_wait_timeout(int(limit_ms), _stream(stream)),
           "attn_selftest_wait_timeout")
