"""Shared helpers of the GPU tests: run the CUDA library through its C ABI and
the fp64 oracle on the same seeded inputs.  Nothing here computes attention:
the expected values come from ``oracle`` only."""
from __future__ import annotations

import concurrent.futures as cf
import math
import os

import numpy as np
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W

#: max-abs tolerance of fp32 outputs against the fp64 oracle (16-bit KV: 2e-3,
#: FP8 KV: 2e-2; the fp16 cache takes the bf16 bound, its type being finer)
TOL = {W.KV_BF16: 2e-3, W.KV_F16: 2e-3, W.KV_FP8: 2e-2, W.KV_FP8_E5M2: 2e-2}
#: tolerance of the natural-log log-sum-exp outputs
LSE_TOL = {W.KV_BF16: 2e-3, W.KV_F16: 2e-3, W.KV_FP8: 2e-2, W.KV_FP8_E5M2: 2e-2}
#: generator cache type -> (library code, oracle code)
_CODES = {W.KV_BF16: (B.PA_KV_BF16, oracle.KV_BF16), W.KV_F16: (B.PA_KV_F16, oracle.KV_F16),
          W.KV_FP8: (B.PA_KV_FP8_E4M3, oracle.KV_FP8_E4M3), W.KV_FP8_E5M2: (B.PA_KV_FP8_E5M2, oracle.KV_FP8_E5M2)}
#: cache types stored as 16-bit values (the pool itself is the cache)
KV16 = (W.KV_BF16, W.KV_F16)


def tcgen05_takes(impl: int, kv: str, head_dim: int) -> bool:
    """Whether the prefill kernel ``impl`` takes this cache type and head_dim:
    the mma.sync kernel every one; the tcgen05 kernel 16-bit caches, and
    8-bit caches at head_dim 128 outside its pair mode."""
    if impl == B.PA_PREFILL_MMA_SYNC or kv in KV16:
        return True
    return impl == B.PA_PREFILL_TCGEN05 and head_dim == 128


def _cpu(t):
    return None if t is None else t.cpu()


def kv_code(b: W.PagedBatch) -> int:
    return _CODES[b.kv_dtype][0]


def desc_of(b: W.PagedBatch, decode_impl: int = B.PA_DECODE_AUTO,
            prefill_impl: int = B.PA_PREFILL_AUTO, window: int = 0, chunk: int = 0) -> B.PaKvDesc:
    return B.make_desc(b.num_blocks, b.num_kv_heads, b.num_q_heads, b.head_dim, kv_code(b),
                       b.k_scale if b.kv_dtype not in KV16 else 0.0,
                       b.v_scale if b.kv_dtype not in KV16 else 0.0, decode_impl=decode_impl,
                       prefill_impl=prefill_impl, sliding_window=window, attention_chunk=chunk,
                       k_scales=b.k_scales, v_scales=b.v_scales)


def gpu_caches(b: W.PagedBatch):
    """The caches as the CUDA path holds them: the bf16 / fp16 pool itself, or
    the 8-bit pool written by the library's own cache write."""
    if b.kv_dtype in KV16:
        return b.k_pool, b.v_pool
    k, v, slots = b.pool_tokens_as_rows()
    kc = torch.zeros(tuple(b.k_pool.shape), dtype=torch.uint8, device=b.k_pool.device)
    vc = torch.zeros_like(kc)
    B.pa_cache_write(desc_of(b), k, v, kc, vc, slots)
    return kc, vc


def oracle_caches(b: W.PagedBatch):
    """The caches as the oracle sees them (CPU numpy): the bf16 / fp16 pool, or
    the oracle's own 8-bit encoding of it."""
    if b.kv_dtype in KV16:
        return _CODES[b.kv_dtype][1], b.k_pool.cpu(), b.v_pool.cpu()
    code = _CODES[b.kv_dtype][1]
    k, v, slots = b.pool_tokens_as_rows()
    z = np.zeros(tuple(b.k_pool.shape), np.uint8)
    kc, vc = oracle.cache_write(code, b.block_size, b.num_kv_heads, b.head_dim,
                                k.cpu(), v.cpu(), slots.cpu(), z, z, b.k_scale, b.v_scale,
                                k_scales=_cpu(b.k_scales), v_scales=_cpu(b.v_scales))
    return code, kc, vc


def gpu_decode(b: W.PagedBatch, caches=None, decode_impl: int = B.PA_DECODE_AUTO, workspace=None, window=0,
               chunk=0):
    kc, vc = caches if caches is not None else gpu_caches(b)
    S = b.context_lens_decode.shape[0]
    out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=kc.device)
    lse = torch.full((S, b.num_q_heads), float("nan"), device=kc.device)
    d = desc_of(b, decode_impl, window=window, chunk=chunk)
    maxL = b.max_context_len_decode()
    ws = workspace if workspace is not None else B.decode_workspace(d, S, maxL, kc.device)
    B.pa_decode(d, out, b.q_decode, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL, b.scale, ws,
                lse=lse)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0, "decode kernel reported a wait timeout"
    return out, lse


def _threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def oracle_in_parallel(call, pairs, num_rows: int, num_heads: int):
    """Runs ``call(pairs_chunk) -> (out [n, D], lse [n])`` of the oracle over
    the (row, head) pairs given (None: every row x head, row-major), in
    chunks on a thread per host core.  The oracle is a C library called
    through ctypes, which releases the GIL, so the chunks run in parallel;
    each pair is computed exactly as in a single call, and the results are
    put back in order."""
    if pairs is None:
        i = np.arange(num_rows * num_heads, dtype=np.int64)
        pairs = np.stack([i // num_heads, i % num_heads], axis=1)
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    n = pairs.shape[0]
    if n == 0:
        return call(pairs)
    bounds = np.linspace(0, n, min(n, 8 * _threads()) + 1).astype(np.int64)
    chunks = [pairs[bounds[i]:bounds[i + 1]] for i in range(len(bounds) - 1) if bounds[i + 1] > bounds[i]]
    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        parts = list(ex.map(call, chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def oracle_decode(b: W.PagedBatch, ocaches=None, pairs=None, window=0, chunk=0):
    kd, kc, vc = ocaches if ocaches is not None else oracle_caches(b)
    q, bt, cl = b.q_decode.cpu(), b.block_tables_decode.cpu(), b.context_lens_decode.cpu()
    ks, vs = _cpu(b.k_scales), _cpu(b.v_scales)

    def call(pp):
        return oracle.decode(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, q, kc, vc, bt, cl,
                             b.scale, b.k_scale, b.v_scale, pairs=pp, window=window, chunk=chunk, k_scales=ks,
                             v_scales=vs)

    return oracle_in_parallel(call, pairs, int(cl.shape[0]), b.num_q_heads)


def gpu_prefill(b: W.PagedBatch, caches=None, prefill_impl: int = B.PA_PREFILL_AUTO, window=0, chunk=0,
                workspace=None):
    """pa_prefill_chunk, or pa_prefill_chunk_balanced with ``workspace``."""
    kc, vc = caches if caches is not None else gpu_caches(b)
    Tq = b.q_prefill.shape[0]
    out = torch.full((Tq, b.num_q_heads, b.head_dim), float("nan"), device=kc.device)
    lse = torch.full((Tq, b.num_q_heads), float("nan"), device=kc.device)
    qsl = b.query_start_loc
    max_q = int((qsl[1:] - qsl[:-1]).max())
    maxL = int(b.context_lens_prefill.max())
    d = desc_of(b, prefill_impl=prefill_impl, window=window, chunk=chunk)
    if workspace is None:
        B.pa_prefill_chunk(d, out, b.q_prefill, qsl, kc, vc, b.block_tables_prefill, b.context_lens_prefill, max_q,
                           maxL, b.scale, lse=lse)
    else:
        B.pa_prefill_chunk_balanced(d, out, b.q_prefill, qsl, kc, vc, b.block_tables_prefill, b.context_lens_prefill,
                                    max_q, maxL, b.scale, workspace, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def prefill_workspace(b: W.PagedBatch, prefill_impl: int = B.PA_PREFILL_AUTO):
    """A zeroed workspace for pa_prefill_chunk_balanced on the batch."""
    qsl = b.query_start_loc
    max_q = int((qsl[1:] - qsl[:-1]).max())
    return B.prefill_workspace(desc_of(b, prefill_impl=prefill_impl), int(b.context_lens_prefill.shape[0]), max_q,
                               b.q_prefill.device)


def oracle_prefill(b: W.PagedBatch, ocaches=None, pairs=None, window=0, chunk=0):
    kd, kc, vc = ocaches if ocaches is not None else oracle_caches(b)
    q, qsl = b.q_prefill.cpu(), b.query_start_loc.cpu()
    bt, cl = b.block_tables_prefill.cpu(), b.context_lens_prefill.cpu()
    ks, vs = _cpu(b.k_scales), _cpu(b.v_scales)

    def call(pp):
        return oracle.prefill(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, q, qsl, kc, vc, bt, cl,
                              b.scale, b.k_scale, b.v_scale, pairs=pp, window=window, chunk=chunk, k_scales=ks,
                              v_scales=vs)

    return oracle_in_parallel(call, pairs, int(q.shape[0]), b.num_q_heads)


def assert_close(got: torch.Tensor, want: np.ndarray, tol: float, what: str = ""):
    g = got.detach().double().cpu().numpy().reshape(want.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - want)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max abs err {worst:.3e} > {tol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst
