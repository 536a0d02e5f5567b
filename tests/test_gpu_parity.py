"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bars: cache writes and block indexing bit-exact; fp32 attention outputs within
max-abs 2e-3 of the oracle for bf16 / fp16 KV and 2e-2 for E4M3 / E5M2 KV.  Every input is
seeded and synthetic; pool slots that no sequence may read hold NaN, so a
stray read shows up as a non-finite output.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import (TOL, LSE_TOL, assert_close, desc_of, tcgen05_takes, gpu_caches, gpu_decode,
                        gpu_prefill, oracle_caches, oracle_decode, oracle_prefill)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


# ------------------------------------------------------------------ cache write

def _bits(t):
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("fp16", [False, True])
def test_cache_write_16bit_bit_exact_on_mixed_step(fp16):
    b = W.workload(5, device=DEV, poison=True, fp16=fp16)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(desc_of(b), b.k_new, b.v_new, kc, vc, b.slot_mapping)
    torch.cuda.synchronize()
    ok, ov = oracle.cache_write(oracle.KV_F16 if fp16 else oracle.KV_BF16, 16, b.num_kv_heads, b.head_dim,
                                b.k_new.cpu(), b.v_new.cpu(),
                                b.slot_mapping.cpu(), b.k_pool.cpu(), b.v_pool.cpu())
    assert np.array_equal(_bits(kc), ok) and np.array_equal(_bits(vc), ov)


def _adversarial_bf16(n_random, g):
    special = [1.0625, -1.0625, 1.1875, 464.0, -464.0, 480.0, 1e30, -1e30, float("inf"), float("-inf"),
               2.0 ** -10, 3 * 2.0 ** -10, -2.0 ** -10, 2.0 ** -12, 0.0, -0.0, float("nan"), 448.0, 449.0,
               2.0 ** -6, 2.0 ** -7 * 1.5, 240.0, 248.0, 232.0,
               # E5M2 ties, saturation and subnormals
               1.125, 1.375, 57344.0, 61440.0, 65536.0, -61440.0, 2.0 ** -16, 3 * 2.0 ** -17, 2.0 ** -17,
               2.0 ** -14, 5 * 2.0 ** -16, 28672.0, 30720.0]
    x = torch.randn(n_random, generator=g) * 3
    return torch.cat([torch.tensor(special), x]).to(torch.bfloat16)


_FP8_CODES = {"e4m3": (B.PA_KV_FP8_E4M3, oracle.KV_FP8_E4M3), "e5m2": (B.PA_KV_FP8_E5M2, oracle.KV_FP8_E5M2)}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.5])
def test_cache_write_fp8_bit_exact_with_ties_saturation_and_nan(scale, fmt):
    lib_code, oracle_code = _FP8_CODES[fmt]
    g = torch.Generator().manual_seed(7)
    H, D = 2, 64
    vals = _adversarial_bf16(H * D * 40, g)
    T = vals.numel() // (H * D)
    k = vals[: T * H * D].reshape(T, H, D)
    v = k.flip(0).contiguous()
    NB = (T + 15) // 16 + 3
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[5] = -1
    d = B.make_desc(NB, H, 2 * H, D, lib_code, scale, scale * 2)
    kc = torch.full((NB, H, 16, D), 0xAB, dtype=torch.uint8, device=DEV)
    vc = kc.clone()
    B.pa_cache_write(d, k.to(DEV), v.to(DEV), kc, vc, slots.to(DEV))
    torch.cuda.synchronize()
    z = np.full((NB, H, 16, D), 0xAB, np.uint8)
    ok, ov = oracle.cache_write(oracle_code, 16, H, D, k, v, slots, z, z, scale, scale * 2)
    assert np.array_equal(kc.cpu().numpy(), ok), np.argwhere(kc.cpu().numpy() != ok)[:5]
    assert np.array_equal(vc.cpu().numpy(), ov)


def test_cache_write_fp8_bit_exact_on_fp8_workload_rows():
    b = W.workload(4, device=DEV, poison=False)
    # 4096 rows of the workload's source values, written at random slots
    k, v, _ = b.pool_tokens_as_rows()
    rows = torch.randperm(k.shape[0], generator=torch.Generator().manual_seed(3))[:4096].to(DEV)
    k, v = k[rows].contiguous(), v[rows].contiguous()
    NB = 300
    slots = torch.randperm(NB * 16, generator=torch.Generator().manual_seed(4))[:4096].to(torch.int64)
    d = B.make_desc(NB, 8, 40, 128, B.PA_KV_FP8_E4M3, b.k_scale, b.v_scale)
    kc = torch.zeros((NB, 8, 16, 128), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    B.pa_cache_write(d, k, v, kc, vc, slots.to(DEV))
    torch.cuda.synchronize()
    z = np.zeros((NB, 8, 16, 128), np.uint8)
    ok, ov = oracle.cache_write(oracle.KV_FP8_E4M3, 16, 8, 128, k.cpu(), v.cpu(), slots, z, z, b.k_scale, b.v_scale)
    assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)


# ---------------------------------------------------------------------- decode

def _check_decode(b, impl=B.PA_DECODE_AUTO, pairs=None, caches=None, ocaches=None):
    out, lse = gpu_decode(b, caches=caches, decode_impl=impl)
    o_ref, l_ref = oracle_decode(b, ocaches=ocaches, pairs=pairs)
    if pairs is not None:
        idx = torch.tensor([s * b.num_q_heads + h for s, h in pairs])
        out = out.reshape(-1, b.head_dim)[idx]
        lse = lse.reshape(-1)[idx]
    e = assert_close(out, o_ref, TOL[b.kv_dtype], "out")
    assert_close(lse, l_ref, LSE_TOL[b.kv_dtype], "lse")
    return e


IMPLS = [B.PA_DECODE_SIMT, B.PA_DECODE_MMA]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("n,fp16", [(1, False), (2, False), (3, False), (1, True), (2, True)])
def test_decode_matches_oracle_on_workload(n, fp16, impl):
    b = W.workload(n, device=DEV, poison=True, fp16=fp16)
    _check_decode(b, impl=impl)


def test_decode_matches_oracle_on_fp8_workload():
    """Workload 4 in full: the library's E4M3 cache write of the whole pool is
    bit-exact against the oracle's encoding, and decode of all 128 sequences
    x 40 heads is within the FP8 tolerance of the oracle over that cache."""
    b = W.workload(4, device=DEV, poison=True)
    caches = gpu_caches(b)
    out, lse = gpu_decode(b, caches=caches)
    code, okc, ovc = oracle_caches(b)
    assert np.array_equal(caches[0].cpu().numpy(), okc), "E4M3 K cache differs from the oracle's encoding"
    assert np.array_equal(caches[1].cpu().numpy(), ovc), "E4M3 V cache differs from the oracle's encoding"
    o_ref, l_ref = oracle_decode(b, ocaches=(code, okc, ovc))
    assert_close(out, o_ref, TOL[W.KV_FP8], "out")
    assert_close(lse, l_ref, LSE_TOL[W.KV_FP8], "lse")


CASES = [
    # (D, Hq, Hkv, kv dtype, lengths)
    (64, 4, 2, W.KV_BF16, [1, 7, 16, 33]),
    (128, 8, 2, W.KV_BF16, [1, 15, 16, 17, 100, 1000, 2049]),
    (128, 3, 1, W.KV_BF16, [5, 64, 300]),
    (64, 1, 1, W.KV_BF16, [1, 2, 31, 500]),
    (128, 16, 16, W.KV_BF16, [40, 41, 700]),
    (128, 10, 2, W.KV_BF16, [1, 17, 333]),
    (128, 16, 1, W.KV_BF16, [9, 250, 1031]),
    (64, 12, 1, W.KV_BF16, [3, 77]),
    (64, 4, 2, W.KV_FP8, [1, 7, 16, 33, 250]),
    (128, 8, 2, W.KV_FP8, [1, 15, 17, 1000, 1600]),
    (128, 2, 1, W.KV_FP8, [3, 129]),
    (128, 40, 8, W.KV_FP8, [1, 100, 1025]),
    (64, 12, 1, W.KV_FP8, [5, 300]),
    (128, 16, 1, W.KV_FP8, [64, 65]),
    (64, 4, 2, W.KV_FP8_E5M2, [1, 7, 16, 33, 250]),
    (128, 8, 2, W.KV_FP8_E5M2, [1, 15, 17, 1000, 1600]),
    (128, 40, 8, W.KV_FP8_E5M2, [1, 100, 1025]),
    (128, 16, 1, W.KV_FP8_E5M2, [64, 65]),
    (64, 4, 2, W.KV_F16, [1, 7, 16, 33, 250]),
    (128, 8, 2, W.KV_F16, [1, 15, 16, 17, 100, 1000, 2049]),
    (128, 32, 8, W.KV_F16, [1, 100, 1025]),
    (128, 16, 1, W.KV_F16, [64, 65, 700]),
    (64, 12, 1, W.KV_F16, [3, 77]),
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("D,Hq,Hkv,kv,lens", CASES)
def test_decode_random_shapes(D, Hq, Hkv, kv, lens, impl):
    if impl == B.PA_DECODE_SIMT and Hq // Hkv > 4:
        pytest.skip("the CUDA-core kernel takes group sizes up to 4")
    b = W.random_decode(100 + D + Hq + len(lens), lens, Hq, Hkv, D, kv_dtype=kv, device=DEV, poison=True)
    _check_decode(b, impl=impl)


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_many_short_sequences_cross_cta_boundaries(impl):
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(1, 200, (300,), generator=g).tolist()
    b = W.random_decode(77, lens, 8, 2, 128, device=DEV, poison=True)
    _check_decode(b, impl=impl)


def test_simt_and_mma_decode_agree():
    b = W.workload(2, device=DEV, poison=True)
    o1, l1 = gpu_decode(b, decode_impl=B.PA_DECODE_SIMT)
    o2, l2 = gpu_decode(b, decode_impl=B.PA_DECODE_MMA)
    assert (o1 - o2).abs().max().item() < 1e-3
    assert (l1 - l2).abs().max().item() < 1e-3


@pytest.mark.parametrize("fp16", [False, True])
@pytest.mark.parametrize("impl", IMPLS)
def test_decode_context_length_one_returns_v_bit_exactly(impl, fp16):
    b = W.workload(1, device=DEV, poison=True, fp16=fp16)
    out, _ = gpu_decode(b, decode_impl=impl)
    blk = int(b.block_tables_decode[0, 0])
    for h in range(4):
        v0 = b.v_pool[blk, h // 2, 0].float()
        assert torch.equal(out[0, h], v0)


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_empty_sequence_gives_zeros_and_minus_inf(impl):
    b = W.random_decode(88, [9, 1, 40], 4, 2, 64, device=DEV, poison=True)
    b.context_lens_decode = torch.tensor([9, 0, 40], dtype=torch.int32, device=DEV)
    out, lse = gpu_decode(b, decode_impl=impl)
    assert torch.all(out[1] == 0) and torch.all(lse[1] == -math.inf)
    o_ref, l_ref = oracle_decode(b)
    keep = [0, 1, 2, 3, 8, 9, 10, 11]
    assert_close(out.reshape(-1, 64)[keep], o_ref[keep], TOL[W.KV_BF16])


@pytest.mark.parametrize("impl", IMPLS)
def test_decode_is_bit_identical_under_physical_block_permutation(impl):
    b = W.workload(3, device=DEV, poison=True)
    out1, lse1 = gpu_decode(b, decode_impl=impl)
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(9)).to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks, device=DEV)
    b.k_pool = b.k_pool[inv].contiguous()
    b.v_pool = b.v_pool[inv].contiguous()
    t = b.block_tables_decode.long()
    b.block_tables_decode = torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32)
    out2, lse2 = gpu_decode(b, decode_impl=impl)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_decode_is_deterministic_and_workspace_reusable():
    b = W.workload(3, device=DEV, poison=True)
    d = desc_of(b)
    ws = B.decode_workspace(d, b.context_lens_decode.shape[0], b.max_context_len_decode(), DEV)
    o1, l1 = gpu_decode(b, workspace=ws)
    assert int(ws[:4].view(torch.int32)[0]) == 0, "error word must stay zero"
    o2, l2 = gpu_decode(b, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_workspace_too_small_is_rejected():
    b = W.workload(1, device=DEV)
    d = desc_of(b)
    n = B.pa_decode_workspace_size(d, 4, 33)
    ws = torch.zeros(n - 256, dtype=torch.uint8, device=DEV)
    out = torch.empty(4, 4, 64, device=DEV)
    with pytest.raises(B.PaError) as ei:
        B.pa_decode(d, out, b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode, b.context_lens_decode, 33,
                    b.scale, ws)
    assert ei.value.status == B.PA_ERR_WORKSPACE


# ---------------------------------------------------------------------- merge

def test_merge_partials_matches_oracle():
    g = torch.Generator().manual_seed(11)
    S, H, P, D = 5, 6, 7, 128
    po = torch.randn(S, H, P, D, generator=g, dtype=torch.float32)
    pl = torch.randn(S, H, P, generator=g, dtype=torch.float32) * 5
    pl[0, 0, 3] = -math.inf
    pl[1, 2, :] = -math.inf
    nparts = torch.tensor([7, 3, 1, 0, 5], dtype=torch.int32)
    out = torch.full((S, H, D), float("nan"), device=DEV)
    lse = torch.full((S, H), float("nan"), device=DEV)
    B.pa_merge_partials(out, po.to(DEV), pl.to(DEV), num_parts=nparts.to(DEV), lse_out=lse)
    torch.cuda.synchronize()
    for s in range(S):
        for h in range(H):
            n = int(nparts[s])
            ro, rl = oracle.merge(po[s, h, :n].double().numpy().reshape(n, D), pl[s, h, :n].double().numpy())
            if n == 0 or rl == -math.inf:
                assert torch.all(out[s, h] == 0) and lse[s, h] == -math.inf
            else:
                assert_close(out[s, h], ro, 1e-5)
                assert abs(float(lse[s, h]) - rl) < 1e-5


def test_merge_of_gpu_split_decode_equals_unsplit():
    """Two half-range decodes merged by pa_merge_partials equal the full decode."""
    b = W.random_decode(55, [300, 161], 4, 2, 128, device=DEV, poison=True)
    full, lfull = gpu_decode(b)
    kc, vc = b.k_pool, b.v_pool
    # first part: the first 160 tokens (ten whole blocks) of each sequence
    first = W.random_decode(55, [300, 161], 4, 2, 128, device=DEV, poison=True)
    first.context_lens_decode = torch.tensor([160, 160], dtype=torch.int32, device=DEV)
    o1, l1 = gpu_decode(first, caches=(kc, vc))
    # second part: the remaining tokens, via a table that starts at block 10
    second = W.random_decode(55, [300, 161], 4, 2, 128, device=DEV, poison=True)
    t = b.block_tables_decode[:, 10:].contiguous()
    second.block_tables_decode = t
    second.context_lens_decode = torch.tensor([140, 1], dtype=torch.int32, device=DEV)
    o2, l2 = gpu_decode(second, caches=(kc, vc))
    po = torch.stack([o1, o2], dim=2).contiguous()
    pl = torch.stack([l1, l2], dim=2).contiguous()
    out = torch.empty_like(full)
    lse = torch.empty_like(lfull)
    B.pa_merge_partials(out, po, pl, lse_out=lse)
    torch.cuda.synchronize()
    assert (out - full).abs().max().item() < 1e-5
    assert (lse - lfull).abs().max().item() < 1e-5


# ---------------------------------------------------------------------- prefill

PREFILL_CASES = [
    # (D, Hq, Hkv, kv, q_lens, ctx_lens, shared prefix blocks)
    (64, 4, 2, W.KV_BF16, [5, 16, 1, 23], [5, 40, 33, 64], 1),
    (128, 32, 8, W.KV_BF16, [100, 37], [300, 37], 0),
    (128, 8, 2, W.KV_BF16, [200, 64, 1], [530, 64, 129], 2),
    (128, 10, 2, W.KV_BF16, [70, 3], [150, 90], 0),
    (128, 1, 1, W.KV_BF16, [129], [129], 0),
    (128, 4, 1, W.KV_BF16, [300, 64], [1000, 65], 3),
    (64, 16, 1, W.KV_BF16, [40, 8], [200, 8], 0),
    (64, 4, 2, W.KV_FP8, [5, 16, 1, 23], [5, 40, 33, 64], 1),
    (128, 8, 2, W.KV_FP8, [90, 20], [300, 20], 1),
    (64, 4, 2, W.KV_FP8_E5M2, [5, 16, 1, 23], [5, 40, 33, 64], 1),
    (128, 8, 2, W.KV_FP8_E5M2, [90, 20], [300, 20], 1),
    (64, 4, 2, W.KV_F16, [5, 16, 1, 23], [5, 40, 33, 64], 1),
    (128, 32, 8, W.KV_F16, [100, 37], [300, 37], 0),
    (128, 8, 2, W.KV_F16, [200, 64, 1], [530, 64, 129], 2),
    (128, 10, 2, W.KV_F16, [70, 3], [150, 90], 0),
]
PREFILL_IMPLS = [B.PA_PREFILL_MMA_SYNC, B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR]
TC_IMPLS = (B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
@pytest.mark.parametrize("D,Hq,Hkv,kv,q_lens,ctx,shared", PREFILL_CASES)
def test_prefill_random_shapes(D, Hq, Hkv, kv, q_lens, ctx, shared, impl):
    if not tcgen05_takes(impl, kv, D):
        pytest.skip("the tcgen05 prefill takes 16-bit caches, and 8-bit ones at head_dim 128 outside the pair mode")
    b = W.random_prefill(200 + D + Hq + len(q_lens), q_lens, ctx, Hq, Hkv, D, kv_dtype=kv, device=DEV,
                         poison=True, shared_prefix_blocks=shared)
    out, lse = gpu_prefill(b, prefill_impl=impl)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


@pytest.mark.parametrize("fp16", [False, True])
@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_mixed_step_write_then_decode_and_prefill(impl, fp16):
    """Workload 5: cache write of 2064 new tokens, then decode (16 sequences)
    and causal prefill (4 chunks of 512 over prefix-shared blocks); bf16, and
    the same step of an fp16 model."""
    b = W.workload(5, device=DEV, poison=True, fp16=fp16)
    kv = b.kv_dtype
    d = desc_of(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(d, b.k_new, b.v_new, kc, vc, b.slot_mapping)
    dec_out, dec_lse = gpu_decode(b, caches=(kc, vc))
    pf_out, pf_lse = gpu_prefill(b, caches=(kc, vc), prefill_impl=impl)
    # oracle: its own cache write of the same inputs, then attention
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    oc = (code, ok, ov)
    o_ref, l_ref = oracle_decode(b, ocaches=oc)
    assert_close(dec_out, o_ref, TOL[kv], "decode out")
    assert_close(dec_lse, l_ref, LSE_TOL[kv], "decode lse")
    # prefill: every query row of the four chunks x all heads
    o_ref, l_ref = oracle_prefill(b, ocaches=oc)
    assert_close(pf_out, o_ref, TOL[kv], "prefill out")
    assert_close(pf_lse, l_ref, LSE_TOL[kv], "prefill lse")


@pytest.mark.parametrize("fp16", [False, True])
@pytest.mark.parametrize("mode", ["fused", "streams", "serial"])
def test_mixed_step_as_the_bench_runs_it(mode, fp16):
    """Workload 5 through MixedStep, the step bench.py times: cache write,
    then decode and prefill in one persistent launch (fused), the decode on a
    second stream beside the balanced prefill (streams) or both in order on
    one stream (serial); every decode and prefill output against the oracle,
    the cache bit-exact, and the workspaces' counters back at zero."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.workload(5, device=DEV, poison=True, fp16=fp16)
    kv = b.kv_dtype
    d = desc_of(b)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    ws = B.mixed_workspace(d, S, maxL, DEV)
    dec_out = torch.full((S, 32, 128), float("nan"), device=DEV)
    dec_lse = torch.full((S, 32), float("nan"), device=DEV)
    pf_out = torch.full((b.q_prefill.shape[0], 32, 128), float("nan"), device=DEV)
    pf_lse = torch.full((b.q_prefill.shape[0], 32), float("nan"), device=DEV)
    qsl = b.query_start_loc
    pws = B.prefill_workspace(d, int(b.context_lens_prefill.shape[0]), int((qsl[1:] - qsl[:-1]).max()), DEV)
    ms = MixedStep(d, kc, vc, b.scale, decode_out=dec_out, decode_lse=dec_lse, workspace=ws,
                   max_context_len_decode=maxL, prefill_out=pf_out, prefill_lse=pf_lse,
                   max_q_len=int((qsl[1:] - qsl[:-1]).max()),
                   max_context_len_prefill=int(b.context_lens_prefill.max()), mode=mode,
                   prefill_workspace=pws)
    assert ms.mode == mode
    for _ in range(2):  # the second call reuses the workspace the first left behind
        dec_out.fill_(float("nan"))
        pf_out.fill_(float("nan"))
        kc.copy_(b.k_pool)
        vc.copy_(b.v_pool)
        ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode),
           (b.q_prefill, qsl, b.block_tables_prefill, b.context_lens_prefill))
        torch.cuda.synchronize()
        assert ws[:12].view(torch.int32).tolist() == [0, 0, 0], "error word and work counters"
        assert int(pws.view(torch.int32)[:64 + 4 * 8 * 8].abs().sum()) == 0, "prefill error word and counters"
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    ok, ov = oracle.cache_write(code, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(),
                                b.k_pool.cpu(), b.v_pool.cpu())
    assert np.array_equal(_bits(kc), ok) and np.array_equal(_bits(vc), ov)
    oc = (code, ok, ov)
    o_ref, l_ref = oracle_decode(b, ocaches=oc)
    assert_close(dec_out, o_ref, TOL[kv], "decode out")
    assert_close(dec_lse, l_ref, LSE_TOL[kv], "decode lse")
    o_ref, l_ref = oracle_prefill(b, ocaches=oc)
    assert_close(pf_out, o_ref, TOL[kv], "prefill out")
    assert_close(pf_lse, l_ref, LSE_TOL[kv], "prefill lse")


@pytest.mark.parametrize("fmt", [W.KV_FP8, W.KV_FP8_E5M2])
def test_mixed_step_with_8bit_cache(fmt):
    """Workload 5 with an 8-bit cache: the pool and the step's new tokens
    written by the library bit-exact against the oracle's encoding, then
    decode and the tcgen05 prefill (8-bit tiles widened to fp16) over it,
    every row against the oracle within the FP8 tolerance."""
    from paged_kv_attention_14_gb300.step import MixedStep
    b = W.workload(5, device=DEV, poison=True, fp8_cache=True, fp8_format=fmt)
    d = desc_of(b)
    kc, vc = gpu_caches(b)  # the whole pool, through the library's cache write
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    ws = B.decode_workspace(d, S, maxL, DEV)
    dec_out = torch.full((S, 32, 128), float("nan"), device=DEV)
    pf_out = torch.full((b.q_prefill.shape[0], 32, 128), float("nan"), device=DEV)
    pf_lse = torch.full((b.q_prefill.shape[0], 32), float("nan"), device=DEV)
    qsl = b.query_start_loc
    ms = MixedStep(d, kc, vc, b.scale, decode_out=dec_out, workspace=ws, max_context_len_decode=maxL,
                   prefill_out=pf_out, prefill_lse=pf_lse, max_q_len=512,
                   max_context_len_prefill=int(b.context_lens_prefill.max()), mode="streams")
    ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode),
       (b.q_prefill, qsl, b.block_tables_prefill, b.context_lens_prefill))
    torch.cuda.synchronize()
    code, okc, ovc = oracle_caches(b)
    okc, ovc = oracle.cache_write(code, 16, 8, 128, b.k_new.cpu(), b.v_new.cpu(), b.slot_mapping.cpu(), okc, ovc,
                                  b.k_scale, b.v_scale)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    oc = (code, okc, ovc)
    o_ref, _ = oracle_decode(b, ocaches=oc)
    assert_close(dec_out, o_ref, TOL[fmt], "decode out")
    o_ref, l_ref = oracle_prefill(b, ocaches=oc)
    assert_close(pf_out, o_ref, TOL[fmt], "prefill out")
    assert_close(pf_lse, l_ref, LSE_TOL[fmt], "prefill lse")


def test_graphed_step_replays_the_step_bit_for_bit():
    """step.GraphedStep (the bench's end-to-end path): the copies in, the
    single-launch step and the copies out captured as a CUDA graph; each
    replay gives exactly the outputs of a direct call on the same inputs."""
    from paged_kv_attention_14_gb300.step import GraphedStep, MixedStep
    b = W.workload(5, device=DEV, poison=True)
    d = desc_of(b)
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    ws = B.mixed_workspace(d, S, maxL, DEV)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    dec_out = torch.empty(S, 32, 128, device=DEV)
    pf_out = torch.empty(b.q_prefill.shape[0], 32, 128, device=DEV)
    qsl = b.query_start_loc
    ms = MixedStep(d, kc, vc, b.scale, decode_out=dec_out, workspace=ws, max_context_len_decode=maxL,
                   prefill_out=pf_out, max_q_len=512, max_context_len_prefill=2560, mode="fused")
    q_host = b.q_decode.cpu().pin_memory()
    q_dev = torch.empty_like(b.q_decode)
    out_host = torch.empty(dec_out.shape).pin_memory()
    pf_host = torch.empty(pf_out.shape).pin_memory()
    dec_args = (q_dev, b.block_tables_decode, b.context_lens_decode)
    pf_args = (b.q_prefill, qsl, b.block_tables_prefill, b.context_lens_prefill)

    def issue():
        q_dev.copy_(q_host, non_blocking=True)
        ms(b.k_new, b.v_new, b.slot_mapping, dec_args, pf_args)
        out_host.copy_(dec_out, non_blocking=True)
        pf_host.copy_(pf_out, non_blocking=True)

    g = GraphedStep(issue)
    ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode), pf_args)
    torch.cuda.synchronize()
    ref_dec, ref_pf = dec_out.cpu(), pf_out.cpu()
    for _ in range(3):
        out_host.zero_()
        pf_host.zero_()
        g()
        assert torch.equal(out_host, ref_dec) and torch.equal(pf_host, ref_pf)
    assert ws[:12].view(torch.int32).tolist() == [0, 0, 0]


def test_tcgen05_and_mma_sync_prefill_agree_on_mixed_step():
    b = W.workload(5, device=DEV, poison=True)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(desc_of(b), b.k_new, b.v_new, kc, vc, b.slot_mapping)  # the chunks' own K/V
    o1, l1 = gpu_prefill(b, caches=(kc, vc), prefill_impl=B.PA_PREFILL_MMA_SYNC)
    o2, l2 = gpu_prefill(b, caches=(kc, vc), prefill_impl=B.PA_PREFILL_TCGEN05)
    assert torch.isfinite(o1).all() and torch.isfinite(o2).all()
    assert (o1 - o2).abs().max().item() < 2e-3
    assert (l1 - l2).abs().max().item() < 2e-3


def test_tcgen05_prefill_with_q_and_out_at_16_byte_offsets():
    """q and out may start at any 16-byte boundary: the TMA maps of the Q
    tiles and of the output tiles then start off a 128-byte line.  The
    results equal those of aligned buffers bit for bit."""
    b = W.workload(5, device=DEV, poison=True)
    kc, vc = b.k_pool.clone(), b.v_pool.clone()
    B.pa_cache_write(desc_of(b), b.k_new, b.v_new, kc, vc, b.slot_mapping)
    o_ref, l_ref = gpu_prefill(b, caches=(kc, vc), prefill_impl=B.PA_PREFILL_TCGEN05)
    Tq, Hq, D = b.q_prefill.shape
    qbuf = torch.empty(b.q_prefill.numel() + 8, dtype=b.q_prefill.dtype, device=DEV)
    q_off = qbuf[8:].view(Tq, Hq, D)  # 16 bytes in
    q_off.copy_(b.q_prefill)
    obuf = torch.full((Tq * Hq * D + 4,), float("nan"), device=DEV)
    out_off = obuf[4:].view(Tq, Hq, D)  # 16 bytes in
    lbuf = torch.full((Tq * Hq + 1,), float("nan"), device=DEV)
    lse_off = lbuf[1:].view(Tq, Hq)  # 4 bytes in
    qsl = b.query_start_loc
    B.pa_prefill_chunk(desc_of(b, prefill_impl=B.PA_PREFILL_TCGEN05), out_off, q_off, qsl, kc, vc,
                       b.block_tables_prefill, b.context_lens_prefill, int((qsl[1:] - qsl[:-1]).max()),
                       int(b.context_lens_prefill.max()), b.scale, lse=lse_off)
    torch.cuda.synchronize()
    assert torch.equal(out_off, o_ref)
    assert torch.equal(lse_off, l_ref)
    assert torch.isnan(obuf[:4]).all() and torch.isnan(lbuf[:1]).all()  # nothing written before the views


def test_tcgen05_prefill_reports_bf16_values_beyond_fp16():
    """A bf16 V element of magnitude >= 2^16 does not fit the fp16 P.V product
    of PA_PREFILL_TCGEN05: the call reports PA_DEVERR_FP16_RANGE; the pair
    mode (P as a bf16 hi + lo pair, V as cached) computes it within tolerance
    and reports nothing.  Values just below the limit are exact in fp16."""
    b = W.random_prefill(330, [90, 20], [300, 20], 8, 2, 128, device=DEV, poison=True, shared_prefix_blocks=1)
    t0 = int(b.block_tables_prefill[0, 2])
    b.v_pool = b.v_pool.clone()
    b.v_pool[t0, 1, 3, 17] = 65280.0   # the largest bf16 below 2^16: fits fp16
    for impl, big, want in ((B.PA_PREFILL_TCGEN05, False, 0), (B.PA_PREFILL_TCGEN05_PAIR, True, 0),
                            (B.PA_PREFILL_TCGEN05, True, B.PA_DEVERR_FP16_RANGE)):
        if big:
            b.v_pool[t0, 1, 5, 9] = -70000.0
        ew = torch.zeros(1, dtype=torch.int32, device=DEV)
        d = B.make_desc(b.num_blocks, 2, 8, 128, prefill_impl=impl, error_word=ew)
        Tq = b.q_prefill.shape[0]
        out = torch.full((Tq, 8, 128), float("nan"), device=DEV)
        qsl = b.query_start_loc
        B.pa_prefill_chunk(d, out, b.q_prefill, qsl, b.k_pool, b.v_pool, b.block_tables_prefill,
                           b.context_lens_prefill, 90, 300, b.scale)
        torch.cuda.synchronize()
        assert int(ew[0]) == want, (impl, big)
        if want == 0:
            o_ref, _ = oracle_prefill(b)
            # the rounding of P (2^-11 relative in fp16) scales with |v|: the
            # bound is relative to the largest |v| here
            vmax = float(b.v_pool[torch.isfinite(b.v_pool)].float().abs().max())
            assert_close(out, o_ref, 1e-3 * vmax, "out")


def test_prefill_single_query_rows_match_decode_oracle():
    lens = [7, 16, 41, 300]
    d = W.random_decode(301, lens, 8, 2, 128, device=DEV, poison=True)
    p = W.random_prefill(301, [1, 1, 1, 1], lens, 8, 2, 128, device=DEV)
    p.q_prefill = d.q_decode.clone()
    p.k_pool, p.v_pool, p.num_blocks = d.k_pool, d.v_pool, d.num_blocks
    p.block_tables_prefill = d.block_tables_decode
    p.context_lens_prefill = d.context_lens_decode
    out, _ = gpu_prefill(p)
    o_ref, _ = oracle_decode(d)
    assert_close(out, o_ref, TOL[W.KV_BF16])
