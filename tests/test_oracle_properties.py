"""Randomised properties of the oracle (hypothesis): identities that fix
the method's arithmetic independently of the oracle's own code.

- Attention over a key range equals the log-sum-exp merge of attention over
  any partition of it (the split-KV and cascade identity).
- A sliding window or a chunk at least as long as the context changes nothing.
- A 16-bit cache write is a scatter of bit patterns, whatever the slots.
"""
import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from paged_kv_attention_14_gb300 import workloads as W  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None)


@SETTINGS
@given(L=st.integers(1, 90), cuts=st.lists(st.integers(1, 89), max_size=5), seed=st.integers(0, 10_000),
       head=st.integers(0, 3))
def test_attention_over_a_range_is_the_merge_of_any_partition(L, cuts, seed, head):
    b = W.random_decode(seed, [L], 4, 2, 64, poison=True)
    table = b.block_tables_decode[0].numpy()
    q = b.q_decode[0, head]
    full_o, full_l = oracle.attend_range(oracle.KV_BF16, 16, 2, 64, q, b.k_pool, b.v_pool, table, head // 2, 0, L,
                                         b.scale)
    bounds = sorted({0, L, *[c for c in cuts if c < L]})
    parts = [oracle.attend_range(oracle.KV_BF16, 16, 2, 64, q, b.k_pool, b.v_pool, table, head // 2, lo, hi,
                                 b.scale) for lo, hi in zip(bounds[:-1], bounds[1:])]
    o, l = oracle.merge(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
    np.testing.assert_allclose(o, full_o, atol=1e-12, rtol=0)
    assert abs(l - full_l) < 1e-12


@SETTINGS
@given(lens=st.lists(st.integers(1, 70), min_size=1, max_size=4), extra=st.integers(0, 50),
       seed=st.integers(0, 10_000))
def test_window_or_chunk_covering_the_context_changes_nothing(lens, extra, seed):
    b = W.random_decode(seed, lens, 4, 2, 64, poison=True)
    args = (oracle.KV_BF16, 16, 2, 4, 64, b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode,
            b.context_lens_decode, b.scale)
    full, full_l = oracle.decode(*args)
    for kw in ({"window": max(lens) + extra}, {"chunk": max(lens) + extra}):
        o, l = oracle.decode(*args, **kw)
        assert np.array_equal(o, full) and np.array_equal(l, full_l)


@SETTINGS
@given(T=st.integers(0, 40), seed=st.integers(0, 10_000), fp16=st.booleans(), skip=st.integers(2, 9))
def test_16bit_cache_write_scatters_bit_patterns(T, seed, fp16, skip):
    g = torch.Generator().manual_seed(seed)
    NB, H, D = 5, 2, 64
    dt = torch.float16 if fp16 else torch.bfloat16
    k = torch.randn(T, H, D, generator=g).to(dt)
    v = torch.randn(T, H, D, generator=g).to(dt)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[::skip] = -1
    pool = torch.randn(NB, H, 16, D, generator=g).to(dt)
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    kc, vc = oracle.cache_write(code, 16, H, D, k, v, slots, pool, pool)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ref_k, ref_v = bits(pool).copy(), bits(pool).copy()
    keep = (slots >= 0).numpy()
    s = slots.numpy()[keep]
    ref_k[s // 16, :, s % 16, :] = bits(k)[keep]
    ref_v[s // 16, :, s % 16, :] = bits(v)[keep]
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)
