"""GPU parity of the shared-prefix (cascade) path and of copy-on-write block
copies against the fp64 oracle.

Cascade: the groups' queries attend their shared prefix in one call
(pa_prefix_attention), each sequence attends its own suffix (pa_decode over
the suffix blocks), and pa_merge_partials combines the two; the result must
match the oracle's decode over the whole context.  Pool slots nobody may read
hold NaN.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import (LSE_TOL, TOL, assert_close, desc_of, gpu_caches, oracle_caches, oracle_decode, _CODES,
                        tcgen05_takes)

pytestmark = pytest.mark.gpu
DEV = "cuda"
IMPLS = [B.PA_PREFILL_MMA_SYNC, B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _gpu_prefix(b, caches, impl, splits=1, slots=None):
    """pa_prefix_attention into [S, Hq, slots, D] / [S, Hq, slots] (slots
    beyond the splits keep their NaN fill)."""
    c = b.meta["cascade"]
    S = b.q_decode.shape[0]
    slots = slots or splits
    out = torch.full((S, b.num_q_heads, slots, b.head_dim), float("nan"), device=DEV)
    lse = torch.full((S, b.num_q_heads, slots), float("nan"), device=DEV)
    qsl = c["query_start_loc"]
    max_q = int((qsl[1:] - qsl[:-1]).max())
    B.pa_prefix_attention(desc_of(b, prefill_impl=impl), out, lse, b.q_decode, qsl, caches[0], caches[1],
                          c["prefix_tables"], c["prefix_lens"], max_q, int(c["prefix_lens"].max()), b.scale,
                          num_splits=splits, out_slots=slots)
    torch.cuda.synchronize()
    return out, lse


def _merged(part_o, part_l):
    S, H, P, D = part_o.shape
    out = torch.empty(S, H, D, device=DEV)
    lse = torch.empty(S, H, device=DEV)
    B.pa_merge_partials(out, part_o.contiguous(), part_l.contiguous(), lse_out=lse)
    torch.cuda.synchronize()
    return out, lse


def _oracle_prefix(b, ocaches, pairs=None):
    c = b.meta["cascade"]
    kd, kc, vc = ocaches
    return oracle.prefix(kd, 16, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode.cpu(),
                         c["query_start_loc"].cpu(), kc, vc, c["prefix_tables"].cpu(), c["prefix_lens"].cpu(),
                         b.scale, b.k_scale, b.v_scale, pairs=pairs)


CASES = [
    # (kv, group sizes, prefix lens, suffix lens, Hq, Hkv, D)
    (W.KV_BF16, [3, 1, 2], [32, 16, 64], [1, 15, 16, 40, 7, 33], 8, 2, 128),
    (W.KV_F16, [5, 2], [256, 0], [3, 100, 17, 1, 64, 9, 250], 32, 8, 128),
    (W.KV_FP8, [4, 3], [160, 48], [1, 2, 3, 4, 5, 6, 700], 8, 2, 128),
    (W.KV_BF16, [2, 2], [48, 16], [5, 6, 7, 8], 4, 2, 64),
]


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("kv,groups,plens,slens,Hq,Hkv,D", CASES)
def test_prefix_attention_matches_oracle(kv, groups, plens, slens, Hq, Hkv, D, impl, splits):
    if not tcgen05_takes(impl, kv, D):
        pytest.skip("the tcgen05 prefill takes 16-bit caches, and 8-bit ones at head_dim 128 outside the pair mode")
    b = W.shared_prefix_decode(300 + sum(plens), groups, plens, slens, Hq, Hkv, D, kv_dtype=kv, device=DEV)
    out, lse = _merged(*_gpu_prefix(b, gpu_caches(b), impl, splits))
    o_ref, l_ref = _oracle_prefix(b, oracle_caches(b))
    empty = torch.tensor(np.repeat(b.meta["cascade"]["prefix_lens"].cpu().numpy(), groups) == 0)
    if empty.any():  # an empty prefix: out 0, lse -inf
        assert torch.all(out[empty.to(DEV)] == 0) and torch.all(torch.isinf(lse[empty.to(DEV)]))
    keep = ~empty
    assert_close(out[keep.to(DEV)], o_ref.reshape(-1, Hq, D)[keep.numpy()], TOL[kv], "out")
    assert_close(lse[keep.to(DEV)], l_ref.reshape(-1, Hq)[keep.numpy()], LSE_TOL[kv], "lse")


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("kv,groups,plens,slens,Hq,Hkv,D", CASES)
def test_cascade_prefix_suffix_merge_equals_full_decode(kv, groups, plens, slens, Hq, Hkv, D, impl, splits):
    if not tcgen05_takes(impl, kv, D):
        pytest.skip("the tcgen05 prefill takes 16-bit caches, and 8-bit ones at head_dim 128 outside the pair mode")
    b = W.shared_prefix_decode(400 + sum(plens), groups, plens, slens, Hq, Hkv, D, kv_dtype=kv, device=DEV)
    c = b.meta["cascade"]
    caches = gpu_caches(b)
    # the prefix splits go straight into the merge's part slots 0 .. splits - 1
    part_o, part_l = _gpu_prefix(b, caches, impl, splits, slots=splits + 1)
    # the own suffix: decode over each sequence's private blocks
    S = b.q_decode.shape[0]
    d = desc_of(b)
    ws = B.decode_workspace(d, S, int(c["suffix_lens"].max()), DEV)
    o_suf = torch.empty(S, Hq, D, device=DEV)
    l_suf = torch.empty(S, Hq, device=DEV)
    B.pa_decode(d, o_suf, b.q_decode, caches[0], caches[1], c["suffix_tables"], c["suffix_lens"],
                int(c["suffix_lens"].max()), b.scale, ws, lse=l_suf)
    part_o[:, :, splits] = o_suf
    part_l[:, :, splits] = l_suf
    out, lse = _merged(part_o, part_l)
    o_ref, l_ref = oracle_decode(b)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


@pytest.mark.parametrize("impl", IMPLS)
def test_wide_group_reads_a_long_prefix_once(impl):
    """64 sequences share a 4096-token prefix: 256 query rows per kv head, one
    tcgen05 tile, the keys in 19 splits; checked on sampled rows."""
    g = torch.Generator().manual_seed(8)
    slens = torch.randint(1, 300, (64,), generator=g).tolist()
    b = W.shared_prefix_decode(501, [64], [4096], slens, 32, 8, 128, device=DEV)
    out, lse = _merged(*_gpu_prefix(b, gpu_caches(b), impl, splits=19))
    rows = [0, 1, 31, 32, 63]
    pairs = [(r, h) for r in rows for h in range(32)]
    o_ref, l_ref = _oracle_prefix(b, oracle_caches(b), pairs=pairs)
    idx = torch.tensor([r * 32 + h for r, h in pairs], device=DEV)
    assert_close(out.reshape(-1, 128)[idx], o_ref, TOL[W.KV_BF16], "out")
    assert_close(lse.reshape(-1)[idx], l_ref, LSE_TOL[W.KV_BF16], "lse")


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8, W.KV_F16])
def test_copy_blocks_bit_exact(kv):
    b = W.random_decode(61, [40, 100, 7], 8, 4, 128, kv_dtype=kv, device=DEV, poison=True)
    kc, vc = gpu_caches(b)
    kc, vc = kc.clone(), vc.clone()
    gen = torch.Generator().manual_seed(2)
    perm = torch.randperm(b.num_blocks, generator=gen)
    src, dst = perm[:5].to(torch.int32), perm[5:10].to(torch.int32)
    before_k = kc.cpu().view(torch.uint8).numpy() if kc.dtype == torch.uint8 else kc.cpu().view(torch.int16).numpy()
    before_v = vc.cpu().view(torch.uint8).numpy() if vc.dtype == torch.uint8 else vc.cpu().view(torch.int16).numpy()
    B.pa_copy_blocks(desc_of(b), kc, vc, src.to(DEV), dst.to(DEV))
    torch.cuda.synchronize()
    code = _CODES[kv][1]
    rk, rv = oracle.copy_blocks(code, 16, b.num_kv_heads, b.head_dim, src, dst, before_k, before_v)
    got_k = kc.cpu().view(torch.uint8).numpy() if kc.dtype == torch.uint8 else kc.cpu().view(torch.int16).numpy()
    got_v = vc.cpu().view(torch.uint8).numpy() if vc.dtype == torch.uint8 else vc.cpu().view(torch.int16).numpy()
    assert np.array_equal(got_k.view(rk.dtype), rk) and np.array_equal(got_v.view(rv.dtype), rv)
