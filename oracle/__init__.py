"""fp64 CPU oracle for paged KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links
or calls it, and it never imports the CUDA library: the two share no code.
The only thing both sides consume is the seeded input generator
(``paged_kv_attention_14_gb300.workloads``), which holds none of the
method's arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain loops, fp64); this module
compiles it with gcc on first use and wraps it for numpy arrays.  What each
function computes and which passage of the source pages it follows is stated
in ``pa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_FP8_E5M2 = 2
KV_F16 = 3


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``libpa_oracle.so`` (gcc, -O2, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        lib.pa_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_e4m3_decode.restype = ctypes.c_double
        lib.pa_oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.pa_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.pa_oracle_e5m2_decode.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_e5m2_decode.restype = ctypes.c_double
        lib.pa_oracle_e5m2_encode.argtypes = [ctypes.c_double]
        lib.pa_oracle_e5m2_encode.restype = ctypes.c_uint8
        lib.pa_oracle_f16_decode.argtypes = [ctypes.c_uint16]
        lib.pa_oracle_f16_decode.restype = ctypes.c_double
        lib.pa_oracle_cache_write.argtypes = [I, I, I, I, P, P, P, I, F, F, P, P, P, P]
        lib.pa_oracle_cache_write.restype = None
        lib.pa_oracle_attend_range.argtypes = [I, I, I, I, P, P, P, P, I, I, I, F, F, F, P, P]
        lib.pa_oracle_attend_range.restype = None
        lib.pa_oracle_decode.argtypes = [I, I, I, I, I, P, P, P, P, I, P, I, F, F, F, P, P, I, I, P, I, P, P]
        lib.pa_oracle_decode.restype = None
        lib.pa_oracle_prefill.argtypes = [I, I, I, I, I, P, P, P, P, P, I, P, I, F, F, F, P, P, I, I, P, I, P, P]
        lib.pa_oracle_prefill.restype = None
        lib.pa_oracle_prefix.argtypes = [I, I, I, I, I, P, P, P, P, P, I, P, I, F, F, F, P, P, P, I, P, P]
        lib.pa_oracle_prefix.restype = None
        lib.pa_oracle_copy_blocks.argtypes = [I, I, I, I, P, P, I, P, P]
        lib.pa_oracle_copy_blocks.restype = None
        lib.pa_oracle_merge.argtypes = [P, P, I, I, P, P]
        lib.pa_oracle_merge.restype = None
        lib.pa_oracle_bind_blocks.argtypes = [P, I, P, P, P, I, P, I, P]
        lib.pa_oracle_bind_blocks.restype = None
        lib.pa_oracle_release_blocks.argtypes = [P, I, P, P, I, P, I, P, P, P]
        lib.pa_oracle_release_blocks.restype = None
        _lib = lib
        return lib


def _np(a, dtype):
    """Contiguous numpy array of ``dtype`` from a numpy array or CPU torch tensor.
    16-bit float tensors (bf16) are passed as their bit patterns."""
    if hasattr(a, "detach"):
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        elif t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
            t = t.view(torch.uint8)
        a = t.numpy()
    a = np.ascontiguousarray(a)
    want = np.dtype(dtype)
    if a.dtype != want:
        if a.dtype.kind in "iu" and want.kind in "iu" and a.dtype.itemsize == want.itemsize:
            a = a.view(want)
        else:
            a = a.astype(want)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _cache_np(cache, kv_dtype):
    return _np(cache, np.uint16 if kv_dtype in (KV_BF16, KV_F16) else np.uint8)


def e4m3_decode(byte: int) -> float:
    return _load().pa_oracle_e4m3_decode(int(byte) & 0xFF)


def e4m3_encode(x: float) -> int:
    return int(_load().pa_oracle_e4m3_encode(float(x)))


def e5m2_decode(byte: int) -> float:
    return _load().pa_oracle_e5m2_decode(int(byte) & 0xFF)


def e5m2_encode(x: float) -> int:
    return int(_load().pa_oracle_e5m2_encode(float(x)))


def f16_decode(bits: int) -> float:
    return _load().pa_oracle_f16_decode(int(bits) & 0xFFFF)


def _scales(a):
    """Optional per-kv-head fp32 scales -> (keep-alive array or None, pointer or None)."""
    if a is None:
        return None, None
    arr = _np(a, np.float32)
    return arr, _ptr(arr)


def cache_write(kv_dtype, block_size, num_kv_heads, head_dim, k, v, slot_mapping,
                k_cache, v_cache, k_scale=1.0, v_scale=1.0, k_scales=None, v_scales=None):
    """Scatter new K/V rows into copies of the caches; returns (k_cache, v_cache).
    ``k_scales`` / ``v_scales``: optional per-kv-head scales of an 8-bit cache."""
    lib = _load()
    ksa, ksp = _scales(k_scales)
    vsa, vsp = _scales(v_scales)
    k = _np(k, np.uint16)
    v = _np(v, np.uint16)
    sm = _np(slot_mapping, np.int64)
    kc = _cache_np(k_cache, kv_dtype).copy()
    vc = _cache_np(v_cache, kv_dtype).copy()
    lib.pa_oracle_cache_write(kv_dtype, block_size, num_kv_heads, head_dim, _ptr(k), _ptr(v),
                              _ptr(sm), int(sm.shape[0]), float(k_scale), float(v_scale), ksp, vsp,
                              _ptr(kc), _ptr(vc))
    return kc, vc


def attend_range(kv_dtype, block_size, num_kv_heads, head_dim, q_vec, k_cache, v_cache,
                 table_row, kv_head, t_begin, t_end, scale, k_scale=1.0, v_scale=1.0):
    """Attention of one bf16 query over logical keys [t_begin, t_end); returns (out, lse)."""
    lib = _load()
    qv = _np(q_vec, np.uint16)
    kc = _cache_np(k_cache, kv_dtype)
    vc = _cache_np(v_cache, kv_dtype)
    tr = _np(table_row, np.int32)
    out = np.zeros(head_dim, np.float64)
    lse = np.zeros(1, np.float64)
    lib.pa_oracle_attend_range(kv_dtype, block_size, num_kv_heads, head_dim, _ptr(qv), _ptr(kc),
                               _ptr(vc), _ptr(tr), int(kv_head), int(t_begin), int(t_end),
                               float(scale), float(k_scale), float(v_scale), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def decode(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, q, k_cache, v_cache,
           block_tables, context_lens, scale, k_scale=1.0, v_scale=1.0, pairs=None, window=0, chunk=0,
           k_scales=None, v_scales=None):
    """Decode attention.  Returns (out [n, D], lse [n]) in fp64 for the (s, h)
    pairs given (default: all, row-major over (s, h)).  ``window`` / ``chunk``:
    sliding-window / chunked-local attention (0: off); ``k_scales`` /
    ``v_scales``: per-kv-head scales of an 8-bit cache."""
    lib = _load()
    ksa, ksp = _scales(k_scales)
    vsa, vsp = _scales(v_scales)
    qn = _np(q, np.uint16)
    kc = _cache_np(k_cache, kv_dtype)
    vc = _cache_np(v_cache, kv_dtype)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    S = int(cl.shape[0])
    if pairs is None:
        n, pp = S * num_q_heads, None
    else:
        pp = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
        n = int(pp.shape[0])
    out = np.zeros((n, head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    lib.pa_oracle_decode(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, _ptr(qn),
                         _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(cl), S,
                         float(scale), float(k_scale), float(v_scale), ksp, vsp, int(window), int(chunk),
                         None if pp is None else _ptr(pp), n, _ptr(out), _ptr(lse))
    return out, lse


def prefill(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, q, query_start_loc,
            k_cache, v_cache, block_tables, context_lens, scale, k_scale=1.0, v_scale=1.0,
            pairs=None, window=0, chunk=0, k_scales=None, v_scales=None):
    """Causal chunked-prefill attention.  Returns (out [n, D], lse [n]) in fp64
    for the (token row, head) pairs given (default: all rows x heads).
    ``window`` / ``chunk``: sliding-window / chunked-local attention (0: off);
    ``k_scales`` / ``v_scales``: per-kv-head scales of an 8-bit cache."""
    lib = _load()
    ksa, ksp = _scales(k_scales)
    vsa, vsp = _scales(v_scales)
    qn = _np(q, np.uint16)
    qsl = _np(query_start_loc, np.int32)
    kc = _cache_np(k_cache, kv_dtype)
    vc = _cache_np(v_cache, kv_dtype)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    S = int(cl.shape[0])
    if pairs is None:
        n, pp = int(qsl[S]) * num_q_heads, None
    else:
        pp = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
        n = int(pp.shape[0])
    out = np.zeros((n, head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    lib.pa_oracle_prefill(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, _ptr(qn),
                          _ptr(qsl), _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(cl), S,
                          float(scale), float(k_scale), float(v_scale), ksp, vsp, int(window), int(chunk),
                          None if pp is None else _ptr(pp), n, _ptr(out), _ptr(lse))
    return out, lse


def prefix(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, q, query_start_loc, k_cache, v_cache,
           block_tables, prefix_lens, scale, k_scale=1.0, v_scale=1.0, pairs=None, k_scales=None, v_scales=None):
    """Shared-prefix attention of query groups (group j: rows
    [query_start_loc[j], query_start_loc[j+1]) over the prefix_lens[j] tokens
    of block_tables[j], no causal mask).  Returns (out [n, D], lse [n])."""
    lib = _load()
    ksa, ksp = _scales(k_scales)
    vsa, vsp = _scales(v_scales)
    qn = _np(q, np.uint16)
    qsl = _np(query_start_loc, np.int32)
    kc = _cache_np(k_cache, kv_dtype)
    vc = _cache_np(v_cache, kv_dtype)
    bt = _np(block_tables, np.int32)
    pl = _np(prefix_lens, np.int32)
    G = int(pl.shape[0])
    if pairs is None:
        n, pp = int(qsl[G]) * num_q_heads, None
    else:
        pp = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
        n = int(pp.shape[0])
    out = np.zeros((n, head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    lib.pa_oracle_prefix(kv_dtype, block_size, num_kv_heads, num_q_heads, head_dim, _ptr(qn), _ptr(qsl),
                         _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(pl), G, float(scale),
                         float(k_scale), float(v_scale), ksp, vsp, None if pp is None else _ptr(pp), n,
                         _ptr(out), _ptr(lse))
    return out, lse


def copy_blocks(kv_dtype, block_size, num_kv_heads, head_dim, src_blocks, dst_blocks, k_cache, v_cache):
    """Copy-on-write of whole blocks into copies of the caches; returns (k_cache, v_cache)."""
    lib = _load()
    kc = _cache_np(k_cache, kv_dtype).copy()
    vc = _cache_np(v_cache, kv_dtype).copy()
    src = _np(src_blocks, np.int32)
    dst = _np(dst_blocks, np.int32)
    lib.pa_oracle_copy_blocks(2 if kv_dtype in (KV_BF16, KV_F16) else 1, block_size, num_kv_heads, head_dim,
                              _ptr(src), _ptr(dst), int(src.shape[0]), _ptr(kc), _ptr(vc))
    return kc, vc


def bind_blocks(block_tables, seq_rows, hit_start, hit_blocks, refcounts):
    """Zero-copy prefix hit: binds each new sequence's table row to its hit's
    pages and counts one more owner per page.  Returns (block_tables,
    refcounts, errors) as new arrays."""
    lib = _load()
    bt = _np(block_tables, np.int32).copy()
    rc = _np(refcounts, np.int32).copy()
    rows = _np(seq_rows, np.int32)
    hs = _np(hit_start, np.int32)
    hb = _np(hit_blocks, np.int32) if len(hit_blocks) else np.zeros(1, np.int32)
    err = np.zeros(1, np.int32)
    lib.pa_oracle_bind_blocks(_ptr(bt), int(bt.shape[1]), _ptr(rows), _ptr(hs), _ptr(hb), int(rows.shape[0]),
                              _ptr(rc), int(rc.shape[0]), _ptr(err))
    return bt, rc, int(err[0])


def release_blocks(block_tables, seq_rows, block_counts, refcounts):
    """Release of finished sequences (or evicted entries): one owner less for
    each page of the given rows, entries set to -1, pages left without an
    owner returned to the pool.  Returns (block_tables, refcounts, free_list,
    errors) as new arrays."""
    lib = _load()
    bt = _np(block_tables, np.int32).copy()
    rc = _np(refcounts, np.int32).copy()
    rows = _np(seq_rows, np.int32)
    cnt = _np(block_counts, np.int32)
    free = np.zeros(max(1, rc.shape[0]), np.int32)
    nfree = np.zeros(1, np.int32)
    err = np.zeros(1, np.int32)
    lib.pa_oracle_release_blocks(_ptr(bt), int(bt.shape[1]), _ptr(rows), _ptr(cnt), int(rows.shape[0]), _ptr(rc),
                                 int(rc.shape[0]), _ptr(free), _ptr(nfree), _ptr(err))
    return bt, rc, free[:int(nfree[0])].copy(), int(err[0])


def merge(part_o, part_lse):
    """Log-sum-exp merge of partial results: part_o [P, D], part_lse [P] -> (out [D], lse)."""
    lib = _load()
    po = np.ascontiguousarray(np.asarray(part_o, np.float64))
    pl = np.ascontiguousarray(np.asarray(part_lse, np.float64))
    D = int(po.shape[1])
    out = np.zeros(D, np.float64)
    lse = np.zeros(1, np.float64)
    lib.pa_oracle_merge(_ptr(po), _ptr(pl), int(po.shape[0]), D, _ptr(out), _ptr(lse))
    return out, float(lse[0])
