"""GPU parity of sliding-window and chunked-local attention (decode and
prefill, every kernel) against the fp64 oracle at the same settings.

Pages no query may see are made unreadable: their block-table entries point at
a spare block that holds NaN, so a kernel that read one would produce NaN.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import LSE_TOL, TOL, assert_close, gpu_caches, gpu_decode, gpu_prefill, oracle_caches, oracle_decode, \
    oracle_prefill, tcgen05_takes

pytestmark = pytest.mark.gpu
DEV = "cuda"

LOCAL = [(1, 0), (7, 0), (16, 0), (33, 0), (500, 0), (0, 16), (0, 64), (0, 100), (40, 64)]


def _first_key(pos, window, chunk):
    """Test setup only (which pages to make unreadable): the first key a query
    at `pos` may see under the two local-attention rules."""
    lo = 0
    if window:
        lo = max(lo, pos - window + 1)
    if chunk:
        lo = max(lo, (pos // chunk) * chunk)
    return lo


def _spare_block(tables, lens, num_blocks):
    used = set()
    for row, L in zip(tables.tolist(), lens.tolist()):
        used.update(row[: (L + 15) // 16])
    spare = [i for i in range(num_blocks) if i not in used]
    assert spare, "the generator's pool has spare (NaN-poisoned) blocks"
    return spare[0]


def _hide_pages_below(tables, lens, first_keys, spare):
    t = tables.clone()
    for s, lo in enumerate(first_keys):
        t[s, : lo // 16] = spare
    return t


@pytest.mark.parametrize("impl", [B.PA_DECODE_SIMT, B.PA_DECODE_MMA])
@pytest.mark.parametrize("window,chunk", LOCAL)
@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8, W.KV_F16])
def test_decode_local_attention(kv, window, chunk, impl):
    lens = [1, 9, 16, 17, 100, 513, 1025]
    b = W.random_decode(700 + window + chunk, lens, 8, 2, 128, kv_dtype=kv, device=DEV, poison=True)
    spare = _spare_block(b.block_tables_decode.cpu(), b.context_lens_decode.cpu(), b.num_blocks)
    firsts = [_first_key(L - 1, window, chunk) for L in lens]
    b.block_tables_decode = _hide_pages_below(b.block_tables_decode, b.context_lens_decode, firsts, spare)
    out, lse = gpu_decode(b, gpu_caches(b), decode_impl=impl, window=window, chunk=chunk)
    o_ref, l_ref = oracle_decode(b, oracle_caches(b), window=window, chunk=chunk)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


@pytest.mark.parametrize("impl", [B.PA_PREFILL_MMA_SYNC, B.PA_PREFILL_TCGEN05, B.PA_PREFILL_TCGEN05_PAIR])
@pytest.mark.parametrize("window,chunk", [(1, 0), (64, 0), (200, 0), (0, 48), (0, 128), (100, 256), (5000, 0)])
@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8, W.KV_F16])
def test_prefill_local_attention(kv, window, chunk, impl):
    if not tcgen05_takes(impl, kv, 128):
        pytest.skip("the tcgen05 prefill takes 16-bit caches, and 8-bit ones at head_dim 128 outside the pair mode")
    q_lens, ctx = [300, 37, 1, 129], [700, 37, 200, 900]
    b = W.random_prefill(800 + window + chunk, q_lens, ctx, 8, 2, 128, kv_dtype=kv, device=DEV, poison=True,
                         shared_prefix_blocks=2)
    spare = _spare_block(b.block_tables_prefill.cpu(), b.context_lens_prefill.cpu(), b.num_blocks)
    # pages before the first key of each chunk's earliest query are never read
    firsts = [_first_key(L - n, window, chunk) for n, L in zip(q_lens, ctx)]
    b.block_tables_prefill = _hide_pages_below(b.block_tables_prefill, b.context_lens_prefill, firsts, spare)
    out, lse = gpu_prefill(b, gpu_caches(b), prefill_impl=impl, window=window, chunk=chunk)
    o_ref, l_ref = oracle_prefill(b, oracle_caches(b), window=window, chunk=chunk)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


def test_local_attention_off_is_bitwise_the_full_path():
    """window = chunk = 0 runs the full-attention path unchanged; a window
    longer than every sequence gives the same numbers."""
    lens = [5, 300, 1000]
    b = W.random_decode(901, lens, 8, 2, 128, device=DEV, poison=True)
    caches = gpu_caches(b)
    full, _ = gpu_decode(b, caches)
    wide, _ = gpu_decode(b, caches, window=5000)
    assert torch.equal(full, wide)
