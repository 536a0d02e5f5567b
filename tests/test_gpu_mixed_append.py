"""pa_mixed_attention_append (a continuous-batch step's cache write, decode
and chunked prefill in one launch) against the fp64 oracle's cache write
followed by its decode and prefill.

The rows the step writes hold NaN in the cache before the call (the pools
are poisoned there): a kernel that read a new token from the cache instead
of from the step's new rows would show NaN or a wrong output.  The caches
must come out bit for bit equal to the oracle's write, the outputs within
2e-3, and caches and outputs bit for bit equal to pa_cache_write followed by
pa_mixed_attention.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
import pa_helpers as H
from pa_helpers import LSE_TOL, TOL, assert_close, desc_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _same_bits(x, y):
    return torch.equal(x.view(torch.int16), y.view(torch.int16))


def _parts(b):
    S = b.context_lens_decode.shape[0]
    qsl = b.query_start_loc
    maxq = int((qsl[1:] - qsl[:-1]).max())
    maxLp = int(b.context_lens_prefill.max())
    maxLd = b.max_context_len_decode()
    d_out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    d_lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    p_out = torch.full(tuple(b.q_prefill.shape), float("nan"), device=DEV)
    p_lse = torch.full((b.q_prefill.shape[0], b.num_q_heads), float("nan"), device=DEV)
    dec = (d_out, b.q_decode, b.block_tables_decode, b.context_lens_decode, maxLd, d_lse)
    pf = (p_out, b.q_prefill, qsl, b.block_tables_prefill, b.context_lens_prefill, maxq, maxLp, p_lse)
    return dec, pf, S, maxLd


def _run(b):
    """The fused step against the two calls and the oracle (every row)."""
    d = desc_of(b)
    dec, pf, S, maxLd = _parts(b)
    ws = B.mixed_workspace(d, S, maxLd, DEV)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_mixed_attention_append(d, b.k_new, b.v_new, kc, vc, b.scale, ws, dec=dec, pf=pf)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0
    # the same step as two calls
    dec2, pf2, _, _ = _parts(b)
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, b.k_new, b.v_new, kc2, vc2, b.slot_mapping)
    B.pa_mixed_attention(d, kc2, vc2, b.scale, B.mixed_workspace(d, S, maxLd, DEV), dec=dec2, pf=pf2)
    torch.cuda.synchronize()
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)
    for x, y in ((dec[0], dec2[0]), (dec[5], dec2[5]), (pf[0], pf2[0]), (pf[7], pf2[7])):
        assert torch.equal(x, y)
    # the oracle: its cache write of the step's rows, then decode and prefill
    code = oracle.KV_F16 if b.kv_dtype == W.KV_F16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, b.num_kv_heads, b.head_dim, b.k_new.cpu(), b.v_new.cpu(),
                                b.slot_mapping.cpu(), b.k_pool.cpu(), b.v_pool.cpu())
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)
    o_ref, l_ref = H.oracle_decode(b, ocaches=(code, ok, ov))
    assert_close(dec[0], o_ref, TOL[b.kv_dtype], "decode out")
    assert_close(dec[5], l_ref, LSE_TOL[b.kv_dtype], "decode lse")
    p_ref, pl_ref = H.oracle_prefill(b, ocaches=(code, ok, ov))
    assert_close(pf[0], p_ref, TOL[b.kv_dtype], "prefill out")
    assert_close(pf[7], pl_ref, LSE_TOL[b.kv_dtype], "prefill lse")


def test_fused_step_on_the_mixed_workload():
    """Workload 5 in full: 16 decode sequences and 4 chunks of 512 on
    2048-token prefixes (1024 shared), every output row against the oracle."""
    _run(W.workload(5, device=DEV, poison=True))


@pytest.mark.parametrize("fp16", [False, True])
@pytest.mark.parametrize("n_dec,n_pf,prefix,chunk,shared", [
    (3, 2, 64, 100, 32),     # chunks ending inside a block; the next chunk's rows follow in k_new
    (1, 1, 0, 33, 0),        # a fresh prompt: every key is a new row
    (5, 3, 160, 257, 160),   # the whole prefix shared
    (0, 2, 48, 16, 16),      # no decode part
    (4, 1, 1024, 700, 512),  # a long chunk over many tiles
])
def test_fused_step_random_batches(fp16, n_dec, n_pf, prefix, chunk, shared):
    b = W.mixed_batch(1300 + n_dec + prefix + chunk, device=DEV, poison=True,
                      kv_dtype=W.KV_F16 if fp16 else W.KV_BF16, n_dec=max(n_dec, 1), dec_range=(1, 700),
                      n_pf=n_pf, prefix=prefix, chunk=chunk, shared=shared)
    if n_dec == 0:
        _run_no_decode(b)
    else:
        _run(b)


def _run_no_decode(b):
    """Only a prefill part: the step's rows are the chunks' rows alone."""
    d = desc_of(b)
    n_dec = b.context_lens_decode.shape[0]
    k_new, v_new = b.k_new[n_dec:].contiguous(), b.v_new[n_dec:].contiguous()
    slots = b.slot_mapping[n_dec:].contiguous()
    _, pf, _, _ = _parts(b)
    ws = B.mixed_workspace(d, 0, 0, DEV)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_mixed_attention_append(d, k_new, v_new, kc, vc, b.scale, ws, dec=None, pf=pf)
    _, pf2, _, _ = _parts(b)
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, k_new, v_new, kc2, vc2, slots)
    B.pa_mixed_attention(d, kc2, vc2, b.scale, B.mixed_workspace(d, 0, 0, DEV), dec=None, pf=pf2)
    torch.cuda.synchronize()
    # the decode sequences' last rows were not written by either call
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)
    assert torch.equal(pf[0], pf2[0]) and torch.equal(pf[7], pf2[7])
    code = oracle.KV_F16 if b.kv_dtype == W.KV_F16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, b.num_kv_heads, b.head_dim, k_new.cpu(), v_new.cpu(), slots.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    p_ref, pl_ref = H.oracle_prefill(b, ocaches=(code, ok, ov))
    assert_close(pf[0], p_ref, TOL[b.kv_dtype], "prefill out")
    assert_close(pf[7], pl_ref, LSE_TOL[b.kv_dtype], "prefill lse")


def test_chunk_not_at_a_block_boundary_is_reported():
    """A chunk whose first position is not a multiple of 16: the step reports
    PA_DEVERR_BAD_INDEX (its outputs are meaningless); nothing leaves the
    buffers."""
    b = W.mixed_batch(1350, device=DEV, poison=False, n_dec=2, dec_range=(10, 100), n_pf=2, prefix=40, chunk=88,
                      shared=32)
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(b.num_blocks, b.num_kv_heads, b.num_q_heads, b.head_dim, error_word=ew)
    dec, pf, S, maxLd = _parts(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_mixed_attention_append(d, b.k_new, b.v_new, kc, vc, b.scale, B.mixed_workspace(d, S, maxLd, DEV),
                                dec=dec, pf=pf)
    torch.cuda.synchronize()
    assert int(ew[0]) & B.PA_DEVERR_BAD_INDEX
    # the decode part is unaffected, and the rows were still written where the slots say
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, b.k_new, b.v_new, kc2, vc2, b.slot_mapping)
    torch.cuda.synchronize()
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)


def test_fused_step_argument_errors():
    b = W.mixed_batch(1360, device=DEV, poison=False, n_dec=2, dec_range=(10, 100), n_pf=1, prefix=32, chunk=16,
                      shared=16)
    d = desc_of(b)
    dec, pf, S, maxLd = _parts(b)
    ws = B.mixed_workspace(d, S, maxLd, DEV)
    with pytest.raises(B.PaError) as e:  # too few rows for the prefill part
        B.pa_mixed_attention_append(d, b.k_new[:2].contiguous(), b.v_new[:2].contiguous(), b.k_pool, b.v_pool,
                                    b.scale, ws, dec=dec, pf=pf)
    assert e.value.status == B.PA_ERR_INVALID_ARG
    d8 = B.make_desc(b.num_blocks, b.num_kv_heads, b.num_q_heads, b.head_dim, B.PA_KV_FP8_E4M3, 1.0, 1.0)
    kc8 = torch.zeros(tuple(b.k_pool.shape), dtype=torch.uint8, device=DEV)
    with pytest.raises(B.PaError) as e:  # the single launch takes 16-bit caches
        B.pa_mixed_attention_append(d8, b.k_new, b.v_new, kc8, kc8.clone(), b.scale, ws, dec=dec, pf=pf)
    assert e.value.status == B.PA_ERR_UNSUPPORTED


def test_mixed_step_writes_in_the_launch():
    """MixedStep(write_in_step=True) on workload 5: one launch per step, the
    same bits as the cache write and pa_mixed_attention."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.workload(5, device=DEV, poison=False)
    d = desc_of(b)
    res = []
    for fused_write in (True, False):
        dec, pf, S, maxLd = _parts(b)
        kc, vc = b.k_pool.clone(), b.v_pool.clone()
        ms = MixedStep(d, kc, vc, b.scale, decode_out=dec[0], decode_lse=dec[5],
                       workspace=B.mixed_workspace(d, S, maxLd, DEV), max_context_len_decode=maxLd,
                       prefill_out=pf[0], prefill_lse=pf[7], max_q_len=pf[5], max_context_len_prefill=pf[6],
                       write_in_step=fused_write)
        ms(b.k_new, b.v_new, b.slot_mapping, dec[1:4], pf[1:5])
        torch.cuda.synchronize()
        res.append((dec[0], dec[5], pf[0], pf[7], kc, vc))
    for x, y in zip(res[0][:4], res[1][:4]):
        assert torch.equal(x, y)
    assert _same_bits(res[0][4], res[1][4]) and _same_bits(res[0][5], res[1][5])


def test_rows_past_the_declared_count_are_reported():
    """num_new_rows short of the chunks' rows: the rows past it are neither
    read nor written, and the step reports PA_DEVERR_BAD_INDEX."""
    b = W.mixed_batch(1370, device=DEV, poison=False, n_dec=2, dec_range=(10, 100), n_pf=2, prefix=32, chunk=40,
                      shared=16)
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(b.num_blocks, b.num_kv_heads, b.num_q_heads, b.head_dim, error_word=ew)
    dec, pf, S, maxLd = _parts(b)
    short = 2 + 40 + 8  # the decode rows, the first chunk and 8 rows of the second
    k_new, v_new = b.k_new[:short].contiguous(), b.v_new[:short].contiguous()
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_mixed_attention_append(d, k_new, v_new, kc, vc, b.scale, B.mixed_workspace(d, S, maxLd, DEV),
                                dec=dec, pf=pf)
    torch.cuda.synchronize()
    assert int(ew[0]) & B.PA_DEVERR_BAD_INDEX
    # the rows up to the count went where the slots say; the others are untouched
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, k_new, v_new, kc2, vc2, b.slot_mapping[:short].contiguous())
    torch.cuda.synchronize()
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)


@pytest.mark.parametrize("window,chunk", [(96, 0), (0, 64)])
def test_fused_step_with_local_attention(window, chunk):
    """Sliding-window and chunked-local attention: pages below every window
    are skipped, the chunk's own keys still come from the new rows."""
    b = W.mixed_batch(1380 + window + chunk, device=DEV, poison=True, n_dec=3, dec_range=(50, 600), n_pf=2,
                      prefix=256, chunk=200, shared=128)
    d = desc_of(b, window=window, chunk=chunk)
    dec, pf, S, maxLd = _parts(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_mixed_attention_append(d, b.k_new, b.v_new, kc, vc, b.scale, B.mixed_workspace(d, S, maxLd, DEV),
                                dec=dec, pf=pf)
    dec2, pf2, _, _ = _parts(b)
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, b.k_new, b.v_new, kc2, vc2, b.slot_mapping)
    B.pa_mixed_attention(d, kc2, vc2, b.scale, B.mixed_workspace(d, S, maxLd, DEV), dec=dec2, pf=pf2)
    torch.cuda.synchronize()
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)
    for x, y in ((dec[0], dec2[0]), (dec[5], dec2[5]), (pf[0], pf2[0]), (pf[7], pf2[7])):
        assert torch.equal(x, y)
    ok, ov = oracle.cache_write(oracle.KV_BF16, 16, b.num_kv_heads, b.head_dim, b.k_new.cpu(), b.v_new.cpu(),
                                b.slot_mapping.cpu(), b.k_pool.cpu(), b.v_pool.cpu())
    o_ref, l_ref = H.oracle_decode(b, ocaches=(oracle.KV_BF16, ok, ov), window=window, chunk=chunk)
    assert_close(dec[0], o_ref, TOL[b.kv_dtype], "decode out")
    p_ref, pl_ref = H.oracle_prefill(b, ocaches=(oracle.KV_BF16, ok, ov), window=window, chunk=chunk)
    assert_close(pf[0], p_ref, TOL[b.kv_dtype], "prefill out")
    assert_close(pf[7], pl_ref, LSE_TOL[b.kv_dtype], "prefill lse")
