"""pa_prefill_chunk_balanced's balanced kernel (the KV work of all items dealt
out evenly over one CTA per SM, items cut between CTAs merged by log-sum-exp
in the launch) against the fp64 oracle, and the library's choice between it
and pa_prefill_chunk's grid.

Bars as everywhere: max-abs 2e-3 (16-bit caches) and 2e-2 (8-bit caches) on
the output and on the log-sum-exp.  The cases cover items cut into two
pieces (the usual case), into many pieces (long contexts, few items),
launches with fewer units than SMs, local attention (items whose first KV
tile is not tile 0), every cache type, and the reuse of one workspace by
consecutive calls (its piece counters back at zero after each call).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import (LSE_TOL, TOL, assert_close, desc_of, gpu_caches, gpu_prefill, oracle_prefill,
                        prefill_workspace, tcgen05_takes)
from test_gpu_parity import PREFILL_CASES, PREFILL_IMPLS

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


@pytest.fixture(autouse=True)
def _balanced():
    """Every test here runs the balanced kernel wherever it applies (the
    library would pick the grid for some of these batches)."""
    B.pa_test_prefill_schedule(1)
    yield
    B.pa_test_prefill_schedule(0)


def _counters_clear(ws, b):
    """The error word and every item's piece counter are zero (the layout:
    error word, then one int32 per (sequence, query tile, kv head) from byte
    256 on)."""
    g = b.num_q_heads // b.num_kv_heads
    qt = 256 // g
    qsl = b.query_start_loc
    max_q = int((qsl[1:] - qsl[:-1]).max())
    items = int(b.context_lens_prefill.shape[0]) * ((max_q + qt - 1) // qt) * b.num_kv_heads
    words = ws.view(torch.int32)
    return int(words[0]) == 0 and int(words[64:64 + items].abs().sum()) == 0


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
@pytest.mark.parametrize("D,Hq,Hkv,kv,q_lens,ctx,shared", PREFILL_CASES)
def test_balanced_prefill_random_shapes(D, Hq, Hkv, kv, q_lens, ctx, shared, impl):
    """Small batches (fewer units than four per SM: the launch shares them
    among fewer CTAs) of every cache type; with the mma.sync kernel selected
    the call runs pa_prefill_chunk's grid."""
    if not tcgen05_takes(impl, kv, D):
        pytest.skip("the tcgen05 prefill takes 16-bit caches, and 8-bit ones at head_dim 128 outside the pair mode")
    b = W.random_prefill(200 + D + Hq + len(q_lens), q_lens, ctx, Hq, Hkv, D, kv_dtype=kv, device=DEV,
                         poison=True, shared_prefix_blocks=shared)
    ws = prefill_workspace(b, impl)
    caches = gpu_caches(b)
    out, lse = gpu_prefill(b, caches=caches, prefill_impl=impl, workspace=ws)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")
    assert _counters_clear(ws, b)


@pytest.mark.parametrize("fp16", [False, True])
def test_balanced_prefill_every_row_of_the_mixed_step_chunks(fp16):
    """Workload 5's prefill (4 chunks of 512 queries on 2048-token prefixes,
    32 q / 8 kv heads): 256 items of 17-20 KV tiles over the SMs, so most
    CTAs hold pieces of two items.  Every query row x head against the
    oracle."""
    b = W.workload(5, device=DEV, poison=True, fp16=fp16)
    kv = b.kv_dtype
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(desc_of(b), b.k_new, b.v_new, kc, vc, b.slot_mapping)  # the chunks' own K/V
    ws = prefill_workspace(b)
    out, lse = gpu_prefill(b, caches=(kc, vc), workspace=ws)
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    o_ref, l_ref = oracle_prefill(b, ocaches=(code, ok, ov))
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")
    assert _counters_clear(ws, b)


@pytest.mark.parametrize("Hq,Hkv,q_lens,ctx", [
    (32, 8, [100], [8000]),          # 2 query tiles x 8 kv heads, 63 KV tiles each
    (8, 8, [300, 5], [6000, 4000]),  # g = 1: 256 queries per item
    (16, 2, [64, 64, 64], [12000, 3000, 64]),
])
def test_balanced_prefill_long_items_cut_into_many_pieces(Hq, Hkv, q_lens, ctx):
    """Few, long items: each is cut between many CTAs, and the last piece to
    finish merges all of them."""
    b = W.random_prefill(700 + Hq + len(q_lens), q_lens, ctx, Hq, Hkv, 128, device=DEV, poison=True,
                         shared_prefix_blocks=0)
    ws = prefill_workspace(b)
    out, lse = gpu_prefill(b, workspace=ws)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(out, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")
    assert _counters_clear(ws, b)


@pytest.mark.parametrize("window,chunk", [(300, 0), (0, 1024), (700, 512)])
def test_balanced_prefill_local_attention(window, chunk):
    """Sliding window / chunked local attention: an item's first KV tile is
    where its earliest query's window starts, so pieces start at any tile."""
    b = W.random_prefill(750 + window + chunk, [400, 130, 7], [3000, 1500, 600], 32, 8, 128, device=DEV,
                         poison=True, shared_prefix_blocks=0)
    ws = prefill_workspace(b)
    out, lse = gpu_prefill(b, window=window, chunk=chunk, workspace=ws)
    o_ref, l_ref = oracle_prefill(b, window=window, chunk=chunk)
    assert_close(out, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")
    assert _counters_clear(ws, b)


def test_balanced_prefill_reuses_its_workspace_and_equals_itself():
    """Consecutive calls on one workspace give bit-identical outputs (the
    schedule and the merge order are fixed by the inputs), each leaving the
    counters at zero; a fresh workspace gives the same bits."""
    b = W.random_prefill(777, [512, 200, 64], [2600, 900, 64], 32, 8, 128, device=DEV, poison=True,
                         shared_prefix_blocks=2)
    caches = gpu_caches(b)
    ws = prefill_workspace(b)
    o1, l1 = gpu_prefill(b, caches=caches, workspace=ws)
    for _ in range(3):
        o2, l2 = gpu_prefill(b, caches=caches, workspace=ws)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        assert _counters_clear(ws, b)
    o3, l3 = gpu_prefill(b, caches=caches, workspace=prefill_workspace(b))
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(o1, o_ref, TOL[b.kv_dtype], "out")


def test_balanced_prefill_rejects_a_small_workspace():
    b = W.random_prefill(778, [100, 37], [300, 37], 32, 8, 128, device=DEV, poison=False)
    ws = prefill_workspace(b)
    with pytest.raises(B.PaError) as e:
        gpu_prefill(b, workspace=ws[: ws.numel() - 16])
    assert e.value.status == B.PA_ERR_WORKSPACE


def test_library_picks_the_grid_for_a_full_batch_and_the_balanced_kernel_for_a_long_chunk():
    """Schedule 0 (the library's choice): workload 5's prefill (256 items on
    the SMs: more than one wave) runs pa_prefill_chunk's grid, bit for bit;
    a single 100-query chunk over 16000 keys (16 items) runs the balanced
    kernel (bits of the forced balanced run, not the grid's); both against
    the oracle."""
    B.pa_test_prefill_schedule(0)
    b = W.workload(5, device=DEV, poison=True)
    caches = (b.k_pool.clone(), b.v_pool.clone())
    B.pa_cache_write(desc_of(b), b.k_new, b.v_new, caches[0], caches[1], b.slot_mapping)  # the chunks' own K/V
    grid, _ = gpu_prefill(b, caches=caches)
    assert bool(torch.isfinite(grid).all())
    auto, _ = gpu_prefill(b, caches=caches, workspace=prefill_workspace(b))
    assert torch.equal(grid, auto)
    b = W.random_prefill(790, [100], [16000], 32, 8, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    grid, _ = gpu_prefill(b, caches=caches)
    auto, lse = gpu_prefill(b, caches=caches, workspace=prefill_workspace(b))
    B.pa_test_prefill_schedule(1)
    forced, _ = gpu_prefill(b, caches=caches, workspace=prefill_workspace(b))
    assert torch.equal(auto, forced) and not torch.equal(auto, grid)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(auto, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")


def test_balanced_prefill_wait_timeout_reports_and_the_next_call_is_correct():
    """With the producer stalled (test hook), every bounded wait of the
    balanced kernel runs out: PA_DEVERR_WAIT_TIMEOUT in the caller's error
    word and the workspace's, tensor memory freed; after the workspace is
    zeroed again, a normal call is correct."""
    b = W.random_prefill(791, [300, 64, 200], [2000, 64, 530], 32, 8, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d0 = desc_of(b)
    d = B.make_desc(d0.num_blocks, d0.num_kv_heads, d0.num_q_heads, d0.head_dim, error_word=ew)
    ws = prefill_workspace(b)
    qsl = b.query_start_loc
    out = torch.full((b.q_prefill.shape[0], 32, 128), float("nan"), device=DEV)
    B.pa_test_stall_pipelines(True, 20_000_000)
    try:
        B.pa_prefill_chunk_balanced(d, out, b.q_prefill, qsl, caches[0], caches[1], b.block_tables_prefill,
                                    b.context_lens_prefill, 300, 2000, b.scale, ws)
    finally:
        torch.cuda.synchronize()
        B.pa_test_stall_pipelines(False)
    assert int(ew[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    assert int(ws.view(torch.int32)[0]) == B.PA_DEVERR_WAIT_TIMEOUT
    ws.zero_()
    ew.zero_()
    o2, l2 = gpu_prefill(b, caches=caches, workspace=ws)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(o2, o_ref, TOL[b.kv_dtype], "out")
    assert_close(l2, l_ref, LSE_TOL[b.kv_dtype], "lse")
    assert _counters_clear(ws, b)


@pytest.mark.parametrize("corrupt", ["none", "block_id", "length_too_long"])
def test_balanced_prefill_checked_indices(corrupt):
    """check_indices on the balanced kernel: valid inputs give the unchecked
    result; a corrupt block id or length is reported in the caller's error
    word and the workspace's, with no access outside the buffers."""
    b = W.random_prefill(792, [100, 37], [3000, 37], 32, 8, 128, device=DEV, poison=True, shared_prefix_blocks=1)
    t = b.block_tables_prefill.clone()
    L = b.context_lens_prefill.clone()
    if corrupt == "block_id":
        t[0, 100] = b.num_blocks
    elif corrupt == "length_too_long":
        L[0] = t.shape[1] * 16 + 1
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(b.num_blocks, 8, 32, 128, error_word=ew, check_indices=True)
    ws = prefill_workspace(b)
    out = torch.full((b.q_prefill.shape[0], 32, 128), float("nan"), device=DEV)
    lse = torch.full((b.q_prefill.shape[0], 32), float("nan"), device=DEV)
    B.pa_prefill_chunk_balanced(d, out, b.q_prefill, b.query_start_loc, b.k_pool, b.v_pool, t, L, 100,
                                int(t.shape[1]) * 16, b.scale, ws, lse=lse)
    torch.cuda.synchronize()
    if corrupt == "none":
        assert int(ew[0]) == 0 and _counters_clear(ws, b)
        o_ref, l_ref = oracle_prefill(b)
        assert_close(out, o_ref, TOL[b.kv_dtype], "out")
        assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")
    else:
        assert int(ew[0]) == B.PA_DEVERR_BAD_INDEX
        assert int(ws.view(torch.int32)[0]) == B.PA_DEVERR_BAD_INDEX


def test_mixed_step_with_a_long_chunk_runs_the_balanced_prefill():
    """A continuous-batch step whose prefill is one chunk of 512 new tokens on
    a 7680-token prefix (64 items, fewer than the SMs) beside 8 decode
    sequences: MixedStep "fused" with a prefill workspace runs the decode and
    then the balanced prefill (the library's choice), and both parts match
    the oracle; the cache write bit for bit."""
    from paged_kv_attention_14_gb300.step import MixedStep
    B.pa_test_prefill_schedule(0)
    b = W.mixed_batch(801, device=DEV, poison=True, n_dec=8, dec_range=(256, 2048), n_pf=1, prefix=7680,
                      chunk=512, shared=0)
    d = desc_of(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    ws = B.mixed_workspace(d, S, maxL, DEV)
    pws = B.prefill_workspace(d, 1, 512, DEV)
    dec_out = torch.full((S, 32, 128), float("nan"), device=DEV)
    pf_out = torch.full((512, 32, 128), float("nan"), device=DEV)
    pf_lse = torch.full((512, 32), float("nan"), device=DEV)
    qsl = b.query_start_loc
    ms = MixedStep(d, kc, vc, b.scale, decode_out=dec_out, workspace=ws, max_context_len_decode=maxL,
                   prefill_out=pf_out, prefill_lse=pf_lse, max_q_len=512, max_context_len_prefill=8192,
                   mode="fused", prefill_workspace=pws)
    pf_args = (b.q_prefill, qsl, b.block_tables_prefill, b.context_lens_prefill)
    assert ms.mode == "fused" and ms.prefill_balanced(pf_args)
    ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode), pf_args)
    torch.cuda.synchronize()
    ok, ov = oracle.cache_write(oracle.KV_BF16, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    assert np.array_equal(kc.view(torch.int16).cpu().numpy().view(np.uint16), ok)
    oc = (oracle.KV_BF16, ok, ov)
    from pa_helpers import oracle_decode
    o_ref, _ = oracle_decode(b, ocaches=oc)
    assert_close(dec_out, o_ref, TOL[b.kv_dtype], "decode out")
    o_ref, l_ref = oracle_prefill(b, ocaches=oc)
    assert_close(pf_out, o_ref, TOL[b.kv_dtype], "prefill out")
    assert_close(pf_lse, l_ref, LSE_TOL[b.kv_dtype], "prefill lse")
    assert _counters_clear(pws, b)
