"""pa_decode_append (a decode step's cache write and decode in one launch)
against the fp64 oracle's cache write followed by its decode.

The appended rows are fresh values, not the pool's, and the cache rows they
go to hold NaN before the call: a kernel that read any appended token from
the cache instead of from k_new / v_new would show NaN or a wrong output.
The caches must come out bit for bit equal to the oracle's write, the outputs
within the usual 2e-3, and bit for bit equal to pa_cache_write followed by
pa_decode on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
import pa_helpers as H
from pa_helpers import LSE_TOL, TOL, assert_close, desc_of, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _same_bits(x, y):
    """Bit-for-bit equality (the poisoned pools hold NaN, which torch.equal
    counts as different from itself)."""
    return torch.equal(x.view(torch.int16), y.view(torch.int16))


def _run(b, seed, window=0, chunk=0):
    g = torch.Generator().manual_seed(seed)
    act = b.k_new.dtype
    k_new = torch.randn(b.k_new.shape, generator=g).to(act).to(DEV)
    v_new = torch.randn(b.v_new.shape, generator=g).to(act).to(DEV)
    d = desc_of(b, decode_impl=B.PA_DECODE_MMA, window=window, chunk=chunk)
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    slots = b.slot_mapping
    live = slots >= 0
    blk, off = slots[live] // 16, slots[live] % 16
    # the step writes these rows: NaN in the cache until then
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    kc[blk, :, off, :] = float("nan")
    vc[blk, :, off, :] = float("nan")
    out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    ws = B.decode_workspace(d, S, maxL, DEV)
    B.pa_decode_append(d, out, b.q_decode, k_new, v_new, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL,
                       b.scale, ws, lse=lse)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0
    # the same step as two calls
    kc2, vc2 = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, k_new, v_new, kc2, vc2, slots)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    B.pa_decode(d, out2, b.q_decode, kc2, vc2, b.block_tables_decode, b.context_lens_decode, maxL, b.scale,
                B.decode_workspace(d, S, maxL, DEV), lse=lse2)
    torch.cuda.synchronize()
    assert _same_bits(kc, kc2) and _same_bits(vc, vc2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # the oracle: its own cache write of the same rows, then its decode
    code = oracle.KV_F16 if b.kv_dtype == W.KV_F16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, b.num_kv_heads, b.head_dim, k_new.cpu(), v_new.cpu(), slots.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    assert np.array_equal(_bits(kc), ok) and np.array_equal(_bits(vc), ov)
    o_ref, l_ref = oracle_decode(b, ocaches=(code, ok, ov), window=window, chunk=chunk)
    Hq, D = b.num_q_heads, b.head_dim
    ne = (b.context_lens_decode > 0).cpu()
    assert_close(out.cpu()[ne], o_ref.reshape(S, Hq, D)[ne.numpy()], TOL[b.kv_dtype], "out")
    assert_close(lse.cpu()[ne], l_ref.reshape(S, Hq)[ne.numpy()], LSE_TOL[b.kv_dtype], "lse")
    # an empty sequence appends nothing and attends to nothing
    assert torch.all(out.cpu()[~ne] == 0) and torch.all(lse.cpu()[~ne] == float("-inf"))


@pytest.mark.parametrize("fp16", [False, True])
def test_decode_append_on_the_qwen3_8b_decode_step(fp16):
    """Workload 2 in full: 32 sequences, lengths U[512, 4096], 32 q / 8 kv heads."""
    b = W.workload(2, device=DEV, poison=True, fp16=fp16)
    _run(b, 11 + fp16)


@pytest.mark.parametrize("D,Hq,Hkv,lens", [
    (128, 32, 8, [1, 15, 16, 17, 31, 32, 33, 100, 2049]),   # every position of the last row in a block
    (128, 40, 8, [5, 64, 513, 1000]),                        # g = 5
    (128, 16, 1, [16, 300, 47]),                             # g = 16
    (64, 4, 2, [1, 7, 16, 33]),                              # D 64, g 2
    (128, 32, 8, [0, 40, 0, 17]),                            # empty sequences append nothing
])
@pytest.mark.parametrize("fp16", [False, True])
def test_decode_append_random_shapes(D, Hq, Hkv, lens, fp16):
    b = W.random_decode(900 + D + Hq + len(lens), lens, Hq, Hkv, D, kv_dtype=W.KV_F16 if fp16 else W.KV_BF16,
                        device=DEV, poison=True)
    _run(b, 21 + len(lens))


@pytest.mark.parametrize("window,chunk", [(256, 0), (0, 512)])
def test_decode_append_with_local_attention(window, chunk):
    b = W.random_decode(950 + window + chunk, [100, 700, 1500, 33], 32, 8, 128, device=DEV, poison=True)
    _run(b, 31, window=window, chunk=chunk)


def _run8(b, seed):
    """The same check for an 8-bit cache: the appended rows are encoded in the
    kernel exactly as pa_cache_write and the oracle encode them."""
    g = torch.Generator().manual_seed(seed)
    k_new = (2 * torch.randn(b.k_new.shape, generator=g)).to(torch.bfloat16).to(DEV)
    v_new = (2 * torch.randn(b.v_new.shape, generator=g)).to(torch.bfloat16).to(DEV)
    d = desc_of(b, decode_impl=B.PA_DECODE_MMA)
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    slots = b.slot_mapping
    live = slots >= 0
    blk, off = slots[live] // 16, slots[live] % 16
    kc0, vc0 = H.gpu_caches(b)
    kc, vc = kc0.clone(), vc0.clone()
    kc[blk, :, off, :] = 0x7F  # NaN codes until the step writes the rows
    vc[blk, :, off, :] = 0x7F
    out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    ws = B.decode_workspace(d, S, maxL, DEV)
    B.pa_decode_append(d, out, b.q_decode, k_new, v_new, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL,
                       b.scale, ws, lse=lse)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0
    kc2, vc2 = kc0.clone(), vc0.clone()
    B.pa_cache_write(d, k_new, v_new, kc2, vc2, slots)
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    B.pa_decode(d, out2, b.q_decode, kc2, vc2, b.block_tables_decode, b.context_lens_decode, maxL, b.scale,
                B.decode_workspace(d, S, maxL, DEV), lse=lse2)
    torch.cuda.synchronize()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    code, okc, ovc = H.oracle_caches(b)
    ok, ov = oracle.cache_write(code, 16, b.num_kv_heads, b.head_dim, k_new.cpu(), v_new.cpu(), slots.cpu(), okc,
                                ovc, b.k_scale, b.v_scale, k_scales=H._cpu(b.k_scales), v_scales=H._cpu(b.v_scales))
    assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)
    o_ref, l_ref = oracle_decode(b, ocaches=(code, ok, ov))
    assert_close(out, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")


def test_decode_append_on_the_fp8_decode_step():
    """Workload 4 in full: 128 sequences, 40 q / 8 kv heads, E4M3 cache."""
    _run8(W.workload(4, device=DEV, poison=False), 41)


@pytest.mark.parametrize("kv", [W.KV_FP8, W.KV_FP8_E5M2])
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("D,Hq,Hkv,lens", [
    (128, 32, 8, [1, 15, 16, 17, 100, 2049]),
    (128, 40, 8, [5, 64, 513]),
    (64, 4, 2, [1, 7, 16, 33]),
])
def test_decode_append_8bit_random_shapes(kv, per_head, D, Hq, Hkv, lens):
    b = W.random_decode(980 + D + Hq + len(lens), lens, Hq, Hkv, D, kv_dtype=kv, device=DEV, poison=False,
                        per_head_scales=per_head)
    _run8(b, 51 + len(lens))


def test_decode_append_refuses_the_cuda_core_kernel():
    """decode_impl PA_DECODE_SIMT: PA_ERR_UNSUPPORTED, nothing enqueued (the
    caller makes the two calls)."""
    b = W.random_decode(960, [40, 17], 8, 2, 128, device=DEV, poison=False)
    S, maxL = 2, 40
    out = torch.empty(S, 8, 128, device=DEV)
    d = desc_of(b, decode_impl=B.PA_DECODE_SIMT)
    ws = B.decode_workspace(d, S, maxL, DEV)
    kc = b.k_pool.clone()
    with pytest.raises(B.PaError) as e:
        B.pa_decode_append(d, out, b.q_decode, b.k_new, b.v_new, kc, kc.clone(), b.block_tables_decode,
                           b.context_lens_decode, maxL, b.scale, ws)
    assert e.value.status == B.PA_ERR_UNSUPPORTED
    assert torch.equal(kc.view(torch.int16), b.k_pool.view(torch.int16))


def test_decode_append_checked_skips_an_out_of_range_last_block():
    """check_indices: a last block whose id lies outside the pool is reported
    and its row is not written (the rest of the cache is unchanged)."""
    b = W.random_decode(970, [40, 17, 64], 32, 8, 128, device=DEV, poison=False)
    t = b.block_tables_decode.clone()
    t[1, 1] = b.num_blocks + 3  # sequence 1's last block (tokens 16..16)
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(b.num_blocks, 8, 32, 128, decode_impl=B.PA_DECODE_MMA, error_word=ew, check_indices=True)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    ws = B.decode_workspace(d, 3, 64, DEV)
    out = torch.empty(3, 32, 128, device=DEV)
    k_new = torch.randn(b.k_new.shape, device=DEV).to(torch.bfloat16)
    B.pa_decode_append(d, out, b.q_decode, k_new, k_new, kc, vc, t, b.context_lens_decode, 64, b.scale, ws)
    torch.cuda.synchronize()
    assert int(ew[0]) & B.PA_DEVERR_BAD_INDEX
    # sequences 0 and 2 appended, sequence 1's row went nowhere
    slots = b.slot_mapping.cpu()
    for s in (0, 2):
        blk, off = int(slots[s]) // 16, int(slots[s]) % 16
        assert _same_bits(kc[blk, :, off, :], k_new[s])
    blk, off = int(slots[1]) // 16, int(slots[1]) % 16
    assert _same_bits(kc[blk, :, off, :], b.k_pool[blk, :, off, :])


def test_mixed_step_appends_a_decode_only_step():
    """MixedStep(decode_append=True), as bench.py runs a decode workload: one
    pa_decode_append launch per step, the same bits as the two calls."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.workload(2, device=DEV, poison=False)
    d = desc_of(b)
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    outs = []
    for append in (True, False):
        kc, vc = b.k_pool.clone(), b.v_pool.clone()
        out = torch.empty(S, 32, 128, device=DEV)
        ms = MixedStep(d, kc, vc, b.scale, decode_out=out, workspace=B.decode_workspace(d, S, maxL, DEV),
                       max_context_len_decode=maxL, decode_append=append)
        ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode))
        torch.cuda.synchronize()
        assert ms.decode_append == append
        outs.append((out, kc, vc))
    assert torch.equal(outs[0][0], outs[1][0])
    assert _same_bits(outs[0][1], outs[1][1]) and _same_bits(outs[0][2], outs[1][2])


def test_mixed_step_appends_an_8bit_decode_step():
    """MixedStep(decode_append=True) with an E4M3 cache: one launch, the same
    bytes and outputs as pa_cache_write + pa_decode."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.random_decode(990, [100, 2049, 17, 512, 1], 40, 8, 128, kv_dtype=W.KV_FP8, device=DEV, poison=False)
    d = desc_of(b)
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    kc0, vc0 = H.gpu_caches(b)
    g = torch.Generator().manual_seed(3)
    k_new = torch.randn(tuple(b.k_new.shape), generator=g).to(torch.bfloat16).to(DEV)
    v_new = torch.randn(tuple(b.v_new.shape), generator=g).to(torch.bfloat16).to(DEV)
    outs = []
    for append in (True, False):
        kc, vc = kc0.clone(), vc0.clone()
        out = torch.empty(S, 40, 128, device=DEV)
        ms = MixedStep(d, kc, vc, b.scale, decode_out=out, workspace=B.decode_workspace(d, S, maxL, DEV),
                       max_context_len_decode=maxL, decode_append=append)
        ms(k_new, v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode))
        torch.cuda.synchronize()
        assert ms.decode_append == append
        outs.append((out, kc, vc))
    assert all(torch.equal(x, y) for x, y in zip(outs[0], outs[1]))
