"""Failure detection on the GPU, without a fault.

* Bounded waits: with the library's test hook the producers of the decode and
  tcgen05 prefill kernels issue no copies, so every wait on them runs out
  after a short limit.  The kernels must report PA_DEVERR_WAIT_TIMEOUT in
  the caller's error word (and the decode workspace's), free what they hold
  and return; a normal call afterwards must be correct.  Nothing is in
  flight when a wait gives up, because nothing was issued.
* Checked indices: with ``check_indices`` the kernels range-check block ids,
  lengths and slots before using them.  Corrupt tables, lengths and slots
  made on the host are reported as PA_DEVERR_BAD_INDEX and redirected into
  the cache, so no access leaves the buffers.  Corrupt inputs are only ever
  passed with checking on.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import (LSE_TOL, TOL, assert_close, desc_of, gpu_caches, gpu_decode, gpu_prefill, oracle_decode,
                        oracle_prefill)

pytestmark = pytest.mark.gpu
DEV = "cuda"
STALL_NS = 20_000_000  # 20 ms


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _with_error_word(b, decode_impl=B.PA_DECODE_AUTO, prefill_impl=B.PA_PREFILL_AUTO, check=False):
    """The batch's descriptor with a fresh zeroed error word (and checking on or off)."""
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = desc_of(b, decode_impl, prefill_impl)
    d2 = B.make_desc(d.num_blocks, d.num_kv_heads, d.num_q_heads, d.head_dim, d.kv_dtype, d.k_scale, d.v_scale,
                     decode_impl=decode_impl, prefill_impl=prefill_impl, k_scales=b.k_scales, v_scales=b.v_scales,
                     error_word=ew, check_indices=check)
    return d2, ew


def _decode(b, d, caches, ws=None, static=False):
    kc, vc = caches
    S = b.context_lens_decode.shape[0]
    out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    maxL = b.max_context_len_decode()
    if static:
        B.pa_decode_static(d, out, b.q_decode, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL, b.scale,
                           lse=lse)
    else:
        B.pa_decode(d, out, b.q_decode, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL, b.scale, ws,
                    lse=lse)
    torch.cuda.synchronize()
    return out, lse


def _stalled(fn):
    B.pa_test_stall_pipelines(True, STALL_NS)
    try:
        return fn()
    finally:
        torch.cuda.synchronize()
        B.pa_test_stall_pipelines(False)


# --------------------------------------------------------------- bounded waits

@pytest.mark.parametrize("impl", [B.PA_DECODE_SIMT, B.PA_DECODE_MMA])
def test_decode_wait_timeout_is_reported_and_the_next_call_is_correct(impl):
    b = W.random_decode(501, [1, 40, 300, 2000, 17], 8, 2, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    d, ew = _with_error_word(b, decode_impl=impl)
    ws = B.decode_workspace(d, 5, b.max_context_len_decode(), DEV)
    _stalled(lambda: _decode(b, d, caches, ws))
    assert int(ew[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    assert int(ws[:4].view(torch.int32)[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    # after an error the workspace is zero-filled again (its contract); the
    # next call runs normally
    ws.zero_()
    ew.zero_()
    out, lse = _decode(b, d, caches, ws)
    assert int(ew[0]) == 0 and int(ws[:4].view(torch.int32)[0]) == 0
    o_ref, l_ref = oracle_decode(b)
    assert_close(out, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")


@pytest.mark.parametrize("impl", [B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR])
@pytest.mark.parametrize("prefix_mode", [False, True])
def test_tcgen05_prefill_wait_timeout_frees_tensor_memory(prefix_mode, impl):
    """The stalled kernel gives up, frees its tensor memory and returns: the
    next launches (which allocate tensor memory on the same SMs) run and are
    correct."""
    b = W.random_prefill(502, [300, 64, 1, 200], [700, 64, 129, 530], 8, 2, 128, device=DEV, poison=True,
                         shared_prefix_blocks=2)
    d, ew = _with_error_word(b, prefill_impl=impl)
    kc, vc = b.k_pool, b.v_pool
    Tq = b.q_prefill.shape[0]
    out = torch.full((Tq, 8, 128), float("nan"), device=DEV)
    lse = torch.full((Tq, 8), float("nan"), device=DEV)
    qsl = b.query_start_loc

    def call():
        if prefix_mode:
            B.pa_prefix_attention(d, out, lse, b.q_prefill, qsl, kc, vc, b.block_tables_prefill,
                                  b.context_lens_prefill, 300, int(b.context_lens_prefill.max()), b.scale)
        else:
            B.pa_prefill_chunk(d, out, b.q_prefill, qsl, kc, vc, b.block_tables_prefill, b.context_lens_prefill, 300,
                               int(b.context_lens_prefill.max()), b.scale, lse=lse)

    _stalled(call)
    assert int(ew[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    ew.zero_()
    for _ in range(3):
        o2, l2 = gpu_prefill(b, prefill_impl=impl, caches=(kc, vc))
    o_ref, l_ref = oracle_prefill(b)
    assert_close(o2, o_ref, TOL[b.kv_dtype], "out")
    assert_close(l2, l_ref, LSE_TOL[b.kv_dtype], "lse")
    assert int(ew[0]) == 0


def test_mixed_attention_wait_timeout_frees_tensor_memory():
    """The single-launch step stalled: every decode partition and prefill tile
    gives up and reports; the counters are back at zero and the next step
    is correct."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.workload(5, device=DEV, poison=True)
    d, ew = _with_error_word(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, b.k_new, b.v_new, kc, vc, b.slot_mapping)
    S = b.context_lens_decode.shape[0]
    ws = B.mixed_workspace(d, S, b.max_context_len_decode(), DEV)
    dec_out = torch.full((S, 32, 128), float("nan"), device=DEV)
    pf_out = torch.full((b.q_prefill.shape[0], 32, 128), float("nan"), device=DEV)
    qsl = b.query_start_loc
    ms = MixedStep(d, kc, vc, b.scale, decode_out=dec_out, workspace=ws, max_context_len_decode=b.max_context_len_decode(),
                   prefill_out=pf_out, max_q_len=512, max_context_len_prefill=2560, mode="fused")
    args = ((b.q_decode, b.block_tables_decode, b.context_lens_decode), (b.q_prefill, qsl, b.block_tables_prefill,
                                                                           b.context_lens_prefill))
    _stalled(lambda: ms.attend(*args))
    assert int(ew[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    assert ws[4:12].view(torch.int32).tolist() == [0, 0], "work counters reset"
    ws.zero_()
    ew.zero_()
    ms.attend(*args)
    torch.cuda.synchronize()
    assert int(ew[0]) == 0
    ok, ov = oracle.cache_write(oracle.KV_BF16, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    rows = [0, 511, 512 + 300, 2047]
    pairs = [(r, h) for r in rows for h in range(32)]
    o_ref, _ = oracle_prefill(b, ocaches=(oracle.KV_BF16, ok, ov), pairs=pairs)
    idx = torch.tensor([r * 32 + h for r, h in pairs])
    assert_close(pf_out.reshape(-1, 128)[idx], o_ref, TOL[W.KV_BF16], "prefill out")
    o_ref, _ = oracle_decode(b, ocaches=(oracle.KV_BF16, ok, ov))
    assert_close(dec_out, o_ref, TOL[W.KV_BF16], "decode out")


def test_static_decode_reports_through_the_callers_error_word():
    b = W.random_decode(503, [5, 1000, 77], 8, 2, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    d, ew = _with_error_word(b)
    _stalled(lambda: _decode(b, d, caches, static=True))
    assert int(ew[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    ew.zero_()
    out, lse = _decode(b, d, caches, static=True)
    ws = B.decode_workspace(d, 3, b.max_context_len_decode(), DEV)
    ref, ref_lse = _decode(b, d, caches, ws)
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    assert int(ew[0]) == 0


# ------------------------------------------------------------- checked indices

@pytest.mark.parametrize("impl", [B.PA_DECODE_SIMT, B.PA_DECODE_MMA])
def test_checked_decode_equals_unchecked_on_valid_inputs(impl):
    b = W.workload(3, device=DEV, poison=True)
    o1, l1 = gpu_decode(b, decode_impl=impl)
    d, ew = _with_error_word(b, decode_impl=impl, check=True)
    ws = B.decode_workspace(d, b.context_lens_decode.shape[0], b.max_context_len_decode(), DEV)
    o2, l2 = _decode(b, d, (b.k_pool, b.v_pool), ws)
    assert int(ew[0]) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("impl", [B.PA_DECODE_SIMT, B.PA_DECODE_MMA])
@pytest.mark.parametrize("corrupt", ["block_id_high", "block_id_negative", "length_too_long", "length_negative"])
def test_checked_decode_reports_corrupt_tables_and_lengths(impl, corrupt):
    b = W.random_decode(504, [33, 200, 1000, 16], 8, 2, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    t = b.block_tables_decode.clone()
    L = b.context_lens_decode.clone()
    if corrupt == "block_id_high":
        t[2, 10] = b.num_blocks + 7
    elif corrupt == "block_id_negative":
        t[1, 3] = -5
    elif corrupt == "length_too_long":
        L[0] = t.shape[1] * 16 + 100
    else:
        L[3] = -4
    b.block_tables_decode, b.context_lens_decode = t, L
    d, ew = _with_error_word(b, decode_impl=impl, check=True)
    ws = B.decode_workspace(d, 4, 1000, DEV)
    kc, vc = caches
    out = torch.empty(4, 8, 128, device=DEV)
    B.pa_decode(d, out, b.q_decode, kc, vc, t, L, 1000, b.scale, ws)
    torch.cuda.synchronize()
    assert int(ew[0]) & B.PA_DEVERR_BAD_INDEX
    assert int(ws[:4].view(torch.int32)[0]) & B.PA_DEVERR_BAD_INDEX


@pytest.mark.parametrize("impl", [B.PA_PREFILL_MMA_SYNC, B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR])
@pytest.mark.parametrize("corrupt", ["none", "block_id", "chunk_longer_than_context", "length_too_long"])
def test_checked_prefill(impl, corrupt):
    b = W.random_prefill(505, [100, 37], [300, 37], 8, 2, 128, device=DEV, poison=True, shared_prefix_blocks=1)
    t = b.block_tables_prefill.clone()
    L = b.context_lens_prefill.clone()
    if corrupt == "block_id":
        t[0, 5] = b.num_blocks
    elif corrupt == "chunk_longer_than_context":
        L[1] = 20  # 37 queries over 20 keys
    elif corrupt == "length_too_long":
        L[0] = t.shape[1] * 16 + 1
    d, ew = _with_error_word(b, prefill_impl=impl, check=True)
    Tq = b.q_prefill.shape[0]
    out = torch.full((Tq, 8, 128), float("nan"), device=DEV)
    lse = torch.full((Tq, 8), float("nan"), device=DEV)
    B.pa_prefill_chunk(d, out, b.q_prefill, b.query_start_loc, b.k_pool, b.v_pool, t, L, 100,
                       int(t.shape[1]) * 16, b.scale, lse=lse)
    torch.cuda.synchronize()
    if corrupt == "none":
        assert int(ew[0]) == 0
        o_ref, l_ref = oracle_prefill(b)
        assert_close(out, o_ref, TOL[b.kv_dtype], "out")
        assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")
    else:
        assert int(ew[0]) == B.PA_DEVERR_BAD_INDEX


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8])
def test_checked_cache_write_skips_slots_past_the_pool(kv):
    g = torch.Generator().manual_seed(506)
    NB, H, D, T = 20, 2, 64, 40
    k = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[3] = NB * 16  # one past the pool
    slots[7] = NB * 16 + 1000
    slots[9] = -1  # skipped, not an error
    code = B.PA_KV_BF16 if kv == W.KV_BF16 else B.PA_KV_FP8_E4M3
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(NB, H, 2 * H, D, code, 0.0 if kv == W.KV_BF16 else 0.02, 0.0 if kv == W.KV_BF16 else 0.03,
                    error_word=ew, check_indices=True)
    shape = (NB, H, 16, D)
    kc = torch.zeros(shape, dtype=torch.bfloat16 if kv == W.KV_BF16 else torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    B.pa_cache_write(d, k.to(DEV), v.to(DEV), kc, vc, slots.to(DEV))
    torch.cuda.synchronize()
    assert int(ew[0]) == B.PA_DEVERR_BAD_INDEX
    # every valid slot is written exactly as the oracle writes it; the rest untouched
    valid = slots.clone()
    valid[valid >= NB * 16] = -1
    ocode = oracle.KV_BF16 if kv == W.KV_BF16 else oracle.KV_FP8_E4M3
    z = np.zeros(shape, np.uint16 if kv == W.KV_BF16 else np.uint8)
    ok, ov = oracle.cache_write(ocode, 16, H, D, k, v, valid, z, z, d.k_scale or 1.0, d.v_scale or 1.0)
    assert np.array_equal(_bits(kc), ok) and np.array_equal(_bits(vc), ov)


def test_checked_block_copy_skips_pairs_outside_the_cache():
    NB, H, D = 12, 2, 64
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(NB, H, 2 * H, D, error_word=ew, check_indices=True)
    kc = torch.randn(NB, H, 16, D, device=DEV).to(torch.bfloat16)
    vc = torch.randn(NB, H, 16, D, device=DEV).to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    src = torch.tensor([1, 2, NB + 3, 4], dtype=torch.int32, device=DEV)
    dst = torch.tensor([5, -1, 7, 8], dtype=torch.int32, device=DEV)
    B.pa_copy_blocks(d, kc, vc, src, dst)
    torch.cuda.synchronize()
    assert int(ew[0]) == B.PA_DEVERR_BAD_INDEX
    want_k, want_v = k0.clone(), v0.clone()
    for s_, d_ in ((1, 5), (4, 8)):
        want_k[d_], want_v[d_] = k0[s_], v0[s_]
    assert torch.equal(kc, want_k) and torch.equal(vc, want_v)
