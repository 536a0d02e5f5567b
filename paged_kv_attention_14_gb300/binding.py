"""Thin Python binding of the C ABI in ``include/pa.h``.

Argument marshalling only: each function takes torch tensors, checks that they
have the dtype, device and contiguity the C ABI expects, and passes their
device pointers and the current CUDA stream to the library function of the
same name.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback.  If ``libpa_gb300.so`` has not been built, loading it
raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_gb300.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4

PA_KV_BF16 = 0
PA_KV_FP8_E4M3 = 1
PA_KV_FP8_E5M2 = 2
PA_KV_F16 = 3

PA_DECODE_AUTO = 0
PA_DECODE_SIMT = 1
PA_DECODE_MMA = 2

PA_PREFILL_AUTO = 0
PA_PREFILL_MMA_SYNC = 1
PA_PREFILL_TCGEN05 = 2
PA_PREFILL_TCGEN05_PAIR = 3

PA_DEVERR_WAIT_TIMEOUT = 1
PA_DEVERR_BAD_INDEX = 2
PA_DEVERR_FP16_RANGE = 4
PA_DEVERR_REFCOUNT = 8

#: every symbol include/pa.h declares
#: PA_ABI_VERSION this binding is written against (pa_kv_desc layout, entry points)
ABI_VERSION = 4
EXPORTED = ("pa_abi_version", "pa_last_error", "pa_cache_write", "pa_decode_workspace_size",
            "pa_decode", "pa_prefill_chunk", "pa_merge_partials", "pa_decode_static", "pa_prefix_attention",
            "pa_copy_blocks", "pa_test_stall_pipelines", "pa_bind_blocks", "pa_release_blocks",
            "pa_mixed_workspace_size", "pa_mixed_attention", "pa_prefill_workspace_size",
            "pa_prefill_chunk_balanced", "pa_test_prefill_schedule", "pa_prefill_balanced_chosen",
            "pa_decode_append", "pa_mixed_attention_append")


class PaKvDesc(ctypes.Structure):
    """``pa_kv_desc`` of include/pa.h (field order and types must match)."""
    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("decode_impl", ctypes.c_int32),
        ("prefill_impl", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32),
        ("attention_chunk", ctypes.c_int32),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("error_word", ctypes.c_void_p),
        ("check_indices", ctypes.c_int32),
    ]


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load the library (once).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with paged_kv_attention_14_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, I32, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        D = ctypes.POINTER(PaKvDesc)
        lib.pa_abi_version.argtypes = []
        lib.pa_abi_version.restype = ctypes.c_int
        lib.pa_last_error.argtypes = []
        lib.pa_last_error.restype = ctypes.c_char_p
        lib.pa_cache_write.argtypes = [D, P, P, P, P, P, I32, P]
        lib.pa_cache_write.restype = ctypes.c_int
        lib.pa_decode_workspace_size.argtypes = [D, I32, I32]
        lib.pa_decode_workspace_size.restype = SZ
        lib.pa_decode.argtypes = [D, P, P, P, P, P, P, I32, P, I32, I32, F, P, SZ, P]
        lib.pa_decode.restype = ctypes.c_int
        lib.pa_decode_append.argtypes = [D, P, P, P, P, P, P, P, P, I32, P, I32, I32, F, P, SZ, P]
        lib.pa_decode_append.restype = ctypes.c_int
        lib.pa_prefill_chunk.argtypes = [D, P, P, P, P, P, P, P, I32, P, I32, I32, I32, F, P]
        lib.pa_prefill_chunk.restype = ctypes.c_int
        lib.pa_prefill_workspace_size.argtypes = [D, I32, I32]
        lib.pa_prefill_workspace_size.restype = SZ
        lib.pa_prefill_chunk_balanced.argtypes = [D, P, P, P, P, P, P, P, I32, P, I32, I32, I32, F, P, SZ, P]
        lib.pa_prefill_chunk_balanced.restype = ctypes.c_int
        lib.pa_prefill_balanced_chosen.argtypes = [D, I32, I32, I32, I32]
        lib.pa_prefill_balanced_chosen.restype = I32
        lib.pa_prefix_attention.argtypes = [D, P, P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, F, P]
        lib.pa_prefix_attention.restype = ctypes.c_int
        lib.pa_copy_blocks.argtypes = [D, P, P, P, P, I32, P]
        lib.pa_copy_blocks.restype = ctypes.c_int
        lib.pa_merge_partials.argtypes = [P, P, P, P, P, I32, I32, I32, I32, P]
        lib.pa_merge_partials.restype = ctypes.c_int
        lib.pa_decode_static.argtypes = [D, P, P, P, P, P, P, I32, P, I32, I32, F, P]
        lib.pa_decode_static.restype = ctypes.c_int
        lib.pa_mixed_workspace_size.argtypes = [D, I32, I32]
        lib.pa_mixed_workspace_size.restype = SZ
        lib.pa_mixed_attention.argtypes = [D, P, P, P, P, I32, P, I32, I32, P, P, P, P, P, I32, P, I32, I32, I32,
                                           P, P, F, P, SZ, P]
        lib.pa_mixed_attention.restype = ctypes.c_int
        lib.pa_mixed_attention_append.argtypes = [D, P, P, P, P, I32, P, I32, I32, P, P, P, P, P, I32, P, I32, I32,
                                                  I32, P, P, ctypes.c_int64, P, P, F, P, SZ, P]
        lib.pa_mixed_attention_append.restype = ctypes.c_int
        lib.pa_bind_blocks.argtypes = [D, P, I32, I32, P, P, P, I32, P, P]
        lib.pa_bind_blocks.restype = ctypes.c_int
        lib.pa_release_blocks.argtypes = [D, P, I32, I32, P, P, I32, P, P, P, P]
        lib.pa_release_blocks.restype = ctypes.c_int
        lib.pa_test_stall_pipelines.argtypes = [I32, ctypes.c_int64]
        lib.pa_test_stall_pipelines.restype = ctypes.c_int
        lib.pa_test_prefill_schedule.argtypes = [I32]
        lib.pa_test_prefill_schedule.restype = ctypes.c_int
        if lib.pa_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{p} has ABI version {lib.pa_abi_version()}, this binding expects {ABI_VERSION}: "
                               "rebuild it")
        if path is None:
            _lib = lib
        return lib


def make_desc(num_blocks: int, num_kv_heads: int, num_q_heads: int, head_dim: int,
              kv_dtype: int = PA_KV_BF16, k_scale: float = 0.0, v_scale: float = 0.0,
              block_size: int = 16, decode_impl: int = PA_DECODE_AUTO,
              prefill_impl: int = PA_PREFILL_AUTO, sliding_window: int = 0,
              attention_chunk: int = 0, k_scales: Optional[torch.Tensor] = None,
              v_scales: Optional[torch.Tensor] = None, error_word: Optional[torch.Tensor] = None,
              check_indices: bool = False) -> PaKvDesc:
    """``k_scales`` / ``v_scales``: optional per-kv-head fp32 scales of an
    8-bit cache, CUDA tensors of num_kv_heads elements; ``error_word``: an
    optional CUDA int32 tensor (one element) that the kernels OR their
    PA_DEVERR_* bits into; the descriptor keeps a reference to these (the
    kernels use them at run time).  ``check_indices``: range-check the
    device arrays' block ids, lengths and slots on the device."""
    for t, name in ((k_scales, "k_scales"), (v_scales, "v_scales")):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()
                              or t.numel() != num_kv_heads):
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of num_kv_heads elements")
    if error_word is not None and (error_word.dtype != torch.int32 or not error_word.is_cuda
                                   or error_word.numel() < 1):
        raise ValueError("error_word must be a CUDA int32 tensor")
    d = PaKvDesc(num_blocks, block_size, num_kv_heads, num_q_heads, head_dim, kv_dtype,
                 k_scale, v_scale, decode_impl, prefill_impl, sliding_window, attention_chunk,
                 k_scales.data_ptr() if k_scales is not None else None,
                 v_scales.data_ptr() if v_scales is not None else None,
                 error_word.data_ptr() if error_word is not None else None, 1 if check_indices else 0)
    d._keep = (k_scales, v_scales, error_word)
    return d


def abi_version() -> int:
    return load().pa_abi_version()


def last_error() -> str:
    return load().pa_last_error().decode()


def _check(status: int):
    if status != PA_OK:
        raise PaError(status, last_error())


def _ptr(t: Optional[torch.Tensor], dtypes, name: str, allow_none: bool = False, host_ok: bool = False):
    """The tensor's address.  ``host_ok``: a pinned CPU tensor is taken too
    (unified addressing maps pinned host memory at the same address)."""
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_cuda and not (host_ok and t.device.type == "cpu" and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or a pinned CPU tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_CACHE = (torch.bfloat16, torch.float16, torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)
_BF16 = (torch.bfloat16,)
_F16 = (torch.float16,)


def _act(desc) -> tuple:
    """Element type of q and of new K/V rows: fp16 with an fp16 cache, else bf16."""
    return _F16 if desc.kv_dtype == PA_KV_F16 else _BF16
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_I64 = (torch.int64,)


def pa_cache_write(desc: PaKvDesc, k, v, k_cache, v_cache, slot_mapping, stream=None):
    """Scatter k, v ``[T, Hkv, D]`` bf16 into the caches at ``slot_mapping`` (int64 [T])."""
    T = int(slot_mapping.shape[0])
    _check(load().pa_cache_write(ctypes.byref(desc), _ptr(k, _act(desc), "k"), _ptr(v, _act(desc), "v"),
                                 _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                 _ptr(slot_mapping, _I64, "slot_mapping"), T, _stream(stream)))


def pa_decode_workspace_size(desc: PaKvDesc, num_seqs: int, max_context_len: int) -> int:
    n = load().pa_decode_workspace_size(ctypes.byref(desc), int(num_seqs), int(max_context_len))
    if n == 0 and num_seqs > 0:
        raise PaError(PA_ERR_UNSUPPORTED, last_error())
    return int(n)


def decode_workspace(desc: PaKvDesc, num_seqs: int, max_context_len: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor of the size pa_decode needs."""
    n = pa_decode_workspace_size(desc, num_seqs, max_context_len)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def pa_decode(desc: PaKvDesc, out, q, k_cache, v_cache, block_tables, context_lens,
              max_context_len: int, scale: float, workspace, lse=None, stream=None):
    """Decode attention: q ``[S, Hq, D]`` bf16 -> out ``[S, Hq, D]`` fp32 (lse ``[S, Hq]``).
    ``out`` / ``lse`` may be pinned CPU tensors: the kernel stores the result
    straight into host memory."""
    S = int(context_lens.shape[0])
    _check(load().pa_decode(ctypes.byref(desc), _ptr(out, _F32, "out", host_ok=True),
                            _ptr(lse, _F32, "lse", allow_none=True, host_ok=True), _ptr(q, _act(desc), "q"),
                            _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                            _ptr(block_tables, _I32, "block_tables"), int(block_tables.shape[1]),
                            _ptr(context_lens, _I32, "context_lens"), S, int(max_context_len),
                            float(scale), _ptr(workspace, (torch.uint8,), "workspace"),
                            workspace.numel(), _stream(stream)))


def pa_decode_append(desc: PaKvDesc, out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                     max_context_len: int, scale: float, workspace, lse=None, stream=None):
    """One decode step in one launch: sequence s's new token (k_new[s], v_new[s],
    ``[S, Hkv, D]``) goes into the caches at position context_lens[s] - 1, and the
    decode attends over all context_lens[s] tokens."""
    S = int(context_lens.shape[0])
    _check(load().pa_decode_append(ctypes.byref(desc), _ptr(out, _F32, "out", host_ok=True),
                                   _ptr(lse, _F32, "lse", allow_none=True, host_ok=True), _ptr(q, _act(desc), "q"),
                                   _ptr(k_new, _act(desc), "k_new"), _ptr(v_new, _act(desc), "v_new"),
                                   _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                   _ptr(block_tables, _I32, "block_tables"), int(block_tables.shape[1]),
                                   _ptr(context_lens, _I32, "context_lens"), S, int(max_context_len),
                                   float(scale), _ptr(workspace, (torch.uint8,), "workspace"),
                                   workspace.numel(), _stream(stream)))


def pa_decode_static(desc: PaKvDesc, out, q, k_cache, v_cache, block_tables, context_lens,
                     max_context_len: int, scale: float, lse=None, stream=None):
    """pa_decode on the library's own fixed-size scratch (no workspace argument,
    for callers that cannot allocate device memory where they decode)."""
    S = int(context_lens.shape[0])
    _check(load().pa_decode_static(ctypes.byref(desc), _ptr(out, _F32, "out", host_ok=True),
                                   _ptr(lse, _F32, "lse", allow_none=True, host_ok=True), _ptr(q, _act(desc), "q"),
                                   _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                   _ptr(block_tables, _I32, "block_tables"), int(block_tables.shape[1]),
                                   _ptr(context_lens, _I32, "context_lens"), S, int(max_context_len),
                                   float(scale), _stream(stream)))


def mixed_workspace(desc: PaKvDesc, num_dec_seqs: int, max_context_len: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor of the size pa_mixed_attention needs."""
    n = load().pa_mixed_workspace_size(ctypes.byref(desc), int(num_dec_seqs), int(max_context_len))
    if n == 0:
        raise PaError(PA_ERR_UNSUPPORTED, last_error())
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _mixed_args(desc: PaKvDesc, dec, pf):
    """The dec_* and pf_* arguments of the mixed entry points."""
    if dec is not None:
        d_out, d_q, d_bt, d_cl, d_maxL = dec[:5]
        d_lse = dec[5] if len(dec) > 5 else None
        dargs = (_ptr(d_out, _F32, "dec out"), _ptr(d_lse, _F32, "dec lse", allow_none=True), _ptr(d_q, _act(desc), "dec q"),
                 _ptr(d_bt, _I32, "dec block_tables"), int(d_bt.shape[1]), _ptr(d_cl, _I32, "dec context_lens"),
                 int(d_cl.shape[0]), int(d_maxL))
    else:
        dargs = (None, None, None, None, 1, None, 0, 0)
    if pf is not None:
        p_out, p_q, p_qsl, p_bt, p_cl, p_maxq, p_maxL = pf[:7]
        p_lse = pf[7] if len(pf) > 7 else None
        pargs = (_ptr(p_out, _F32, "prefill out"), _ptr(p_lse, _F32, "prefill lse", allow_none=True),
                 _ptr(p_q, _act(desc), "prefill q"), _ptr(p_qsl, _I32, "query_start_loc"),
                 _ptr(p_bt, _I32, "prefill block_tables"), int(p_bt.shape[1]), _ptr(p_cl, _I32, "prefill context_lens"),
                 int(p_cl.shape[0]), int(p_maxq), int(p_maxL))
    else:
        pargs = (None, None, None, None, None, 1, None, 0, 0, 0)
    return dargs, pargs


def pa_mixed_attention(desc: PaKvDesc, k_cache, v_cache, scale: float, workspace, dec=None, pf=None, stream=None):
    """Decode and prefill attention of one step in one launch.  ``dec``:
    (out, q, block_tables, context_lens, max_context_len[, lse]) or None;
    ``pf``: (out, q, query_start_loc, block_tables, context_lens, max_q_len,
    max_context_len[, lse]) or None.  ``workspace``: mixed_workspace() for
    the decode part's batch."""
    dargs, pargs = _mixed_args(desc, dec, pf)
    _check(load().pa_mixed_attention(ctypes.byref(desc), *dargs, *pargs, _ptr(k_cache, _CACHE, "k_cache"),
                                     _ptr(v_cache, _CACHE, "v_cache"), float(scale),
                                     _ptr(workspace, (torch.uint8,), "workspace"), workspace.numel(),
                                     _stream(stream)))


def pa_mixed_attention_append(desc: PaKvDesc, k_new, v_new, k_cache, v_cache, scale: float, workspace, dec=None,
                              pf=None, stream=None):
    """pa_mixed_attention with the step's cache write in the same launch.
    ``k_new`` / ``v_new``: ``[T, Hkv, D]``, the decode sequences' new tokens
    first, then the prefill chunks' tokens in query order; every chunk
    starts at a block boundary."""
    dargs, pargs = _mixed_args(desc, dec, pf)
    _check(load().pa_mixed_attention_append(ctypes.byref(desc), *dargs, *pargs, _ptr(k_new, _act(desc), "k_new"),
                                            _ptr(v_new, _act(desc), "v_new"), int(k_new.shape[0]),
                                            _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                            float(scale), _ptr(workspace, (torch.uint8,), "workspace"),
                                            workspace.numel(), _stream(stream)))


def pa_prefill_chunk(desc: PaKvDesc, out, q, query_start_loc, k_cache, v_cache, block_tables,
                     context_lens, max_q_len: int, max_context_len: int, scale: float, lse=None,
                     stream=None):
    """Causal chunked prefill: q ``[Tq, Hq, D]`` bf16 -> out ``[Tq, Hq, D]`` fp32."""
    S = int(context_lens.shape[0])
    _check(load().pa_prefill_chunk(ctypes.byref(desc), _ptr(out, _F32, "out"),
                                   _ptr(lse, _F32, "lse", allow_none=True), _ptr(q, _act(desc), "q"),
                                   _ptr(query_start_loc, _I32, "query_start_loc"),
                                   _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                   _ptr(block_tables, _I32, "block_tables"), int(block_tables.shape[1]),
                                   _ptr(context_lens, _I32, "context_lens"), S, int(max_q_len),
                                   int(max_context_len), float(scale), _stream(stream)))


def pa_prefill_workspace_size(desc: PaKvDesc, num_seqs: int, max_q_len: int) -> int:
    n = load().pa_prefill_workspace_size(ctypes.byref(desc), int(num_seqs), int(max_q_len))
    if n == 0:
        raise PaError(PA_ERR_INVALID_ARG, last_error())
    return n


def pa_prefill_balanced_chosen(desc: PaKvDesc, num_seqs: int, max_q_len: int, max_context_len: int,
                               max_blocks_per_seq: int) -> bool:
    """Whether pa_prefill_chunk_balanced runs the balanced kernel for such a batch."""
    r = load().pa_prefill_balanced_chosen(ctypes.byref(desc), int(num_seqs), int(max_q_len), int(max_context_len),
                                          int(max_blocks_per_seq))
    if r < 0:
        raise PaError(PA_ERR_INVALID_ARG, "invalid descriptor or batch shape")
    return bool(r)


def prefill_workspace(desc: PaKvDesc, num_seqs: int, max_q_len: int, device=None) -> torch.Tensor:
    """A zero-filled workspace of pa_prefill_workspace_size bytes."""
    return torch.zeros(pa_prefill_workspace_size(desc, num_seqs, max_q_len), dtype=torch.uint8, device=device or "cuda")


def pa_prefill_chunk_balanced(desc: PaKvDesc, out, q, query_start_loc, k_cache, v_cache, block_tables,
                              context_lens, max_q_len: int, max_context_len: int, scale: float, workspace,
                              lse=None, stream=None):
    """pa_prefill_chunk with the KV work spread evenly over the SMs (``workspace``:
    a uint8 CUDA tensor of pa_prefill_workspace_size bytes, zero-filled once)."""
    S = int(context_lens.shape[0])
    _check(load().pa_prefill_chunk_balanced(ctypes.byref(desc), _ptr(out, _F32, "out"),
                                            _ptr(lse, _F32, "lse", allow_none=True), _ptr(q, _act(desc), "q"),
                                            _ptr(query_start_loc, _I32, "query_start_loc"),
                                            _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                            _ptr(block_tables, _I32, "block_tables"), int(block_tables.shape[1]),
                                            _ptr(context_lens, _I32, "context_lens"), S, int(max_q_len),
                                            int(max_context_len), float(scale), _ptr(workspace, (torch.uint8,), "workspace"),
                                            workspace.numel(), _stream(stream)))


def pa_prefix_attention(desc: PaKvDesc, out, lse, q, query_start_loc, k_cache, v_cache, prefix_tables,
                        prefix_lens, max_q_len: int, max_prefix_len: int, scale: float, num_splits: int = 1,
                        out_slots: int = 0, stream=None):
    """Shared-prefix (cascade) attention of query groups: q ``[Nq, Hq, D]`` ->
    out ``[Nq, Hq, out_slots, D]`` fp32 and lse ``[Nq, Hq, out_slots]``, split
    i of the prefix keys in slot i (group j: rows query_start_loc[j] ..
    query_start_loc[j+1] over its prefix, no mask).  With one split and
    out_slots 0 the outputs may be ``[Nq, Hq, D]`` / ``[Nq, Hq]``."""
    G = int(prefix_lens.shape[0])
    _check(load().pa_prefix_attention(ctypes.byref(desc), _ptr(out, _F32, "out"), _ptr(lse, _F32, "lse"),
                                      _ptr(q, _act(desc), "q"), _ptr(query_start_loc, _I32, "query_start_loc"),
                                      _ptr(k_cache, _CACHE, "k_cache"), _ptr(v_cache, _CACHE, "v_cache"),
                                      _ptr(prefix_tables, _I32, "prefix_tables"), int(prefix_tables.shape[1]),
                                      _ptr(prefix_lens, _I32, "prefix_lens"), G, int(max_q_len),
                                      int(max_prefix_len), int(num_splits), int(out_slots), float(scale),
                                      _stream(stream)))


def prefix_splits(num_groups: int, num_kv_heads: int, q_tiles: int, max_prefix_len: int, sm_count: int) -> int:
    """A key-split count for pa_prefix_attention that gives about one CTA per
    SM: groups x kv heads x query tiles x splits ~ sm_count, each split at
    least 512 keys."""
    base = max(1, num_groups * num_kv_heads * q_tiles)
    return max(1, min(sm_count // base if base < sm_count else 1, max(1, max_prefix_len // 512)))


def pa_copy_blocks(desc: PaKvDesc, k_cache, v_cache, src_blocks, dst_blocks, stream=None):
    """Copy-on-write: block dst_blocks[i] of both caches gets block src_blocks[i]."""
    _check(load().pa_copy_blocks(ctypes.byref(desc), _ptr(k_cache, _CACHE, "k_cache"),
                                 _ptr(v_cache, _CACHE, "v_cache"), _ptr(src_blocks, _I32, "src_blocks"),
                                 _ptr(dst_blocks, _I32, "dst_blocks"), int(src_blocks.shape[0]),
                                 _stream(stream)))


def pa_bind_blocks(desc: PaKvDesc, block_tables, seq_rows, hit_start, hit_blocks, refcounts, stream=None):
    """Zero-copy prefix hits: row seq_rows[i] of block_tables gets the pages
    hit_blocks[hit_start[i]:hit_start[i+1]]; each page gains an owner in refcounts."""
    _check(load().pa_bind_blocks(ctypes.byref(desc), _ptr(block_tables, _I32, "block_tables"),
                                 int(block_tables.shape[1]), int(block_tables.shape[0]),
                                 _ptr(seq_rows, _I32, "seq_rows"), _ptr(hit_start, _I32, "hit_start"),
                                 _ptr(hit_blocks, _I32, "hit_blocks"), int(seq_rows.shape[0]),
                                 _ptr(refcounts, _I32, "refcounts"), _stream(stream)))


def pa_release_blocks(desc: PaKvDesc, block_tables, seq_rows, block_counts, refcounts, free_list, free_count,
                      stream=None):
    """Release: the first block_counts[i] pages of row seq_rows[i] lose an owner
    (entries set to -1); pages left without owners are appended to free_list at
    free_count."""
    _check(load().pa_release_blocks(ctypes.byref(desc), _ptr(block_tables, _I32, "block_tables"),
                                    int(block_tables.shape[1]), int(block_tables.shape[0]),
                                    _ptr(seq_rows, _I32, "seq_rows"), _ptr(block_counts, _I32, "block_counts"),
                                    int(seq_rows.shape[0]), _ptr(refcounts, _I32, "refcounts"),
                                    _ptr(free_list, _I32, "free_list"), _ptr(free_count, _I32, "free_count"),
                                    _stream(stream)))


def pa_test_stall_pipelines(enable: bool, wait_limit_ns: int = 20_000_000):
    """Test hook of the failure path: while enabled, the decode and tcgen05
    prefill kernels issue no copies and their bounded waits (limited to
    ``wait_limit_ns``) run out; they report PA_DEVERR_WAIT_TIMEOUT and return."""
    _check(load().pa_test_stall_pipelines(1 if enable else 0, int(wait_limit_ns)))


def pa_test_prefill_schedule(schedule: int):
    """Test hook: 0 the library's choice, 1 the balanced kernel wherever it
    applies, 2 pa_prefill_chunk's grid (for pa_prefill_chunk_balanced)."""
    _check(load().pa_test_prefill_schedule(int(schedule)))


def pa_merge_partials(out, part_o, part_lse, num_parts=None, lse_out=None, stream=None):
    """Merge part_o ``[S, H, P, D]`` / part_lse ``[S, H, P]`` into out ``[S, H, D]``."""
    S, H, P, D = (int(x) for x in part_o.shape)
    _check(load().pa_merge_partials(_ptr(out, _F32, "out"), _ptr(lse_out, _F32, "lse_out", allow_none=True),
                                    _ptr(part_o, _F32, "part_o"), _ptr(part_lse, _F32, "part_lse"),
                                    _ptr(num_parts, _I32, "num_parts", allow_none=True), S, H, P, D,
                                    _stream(stream)))
