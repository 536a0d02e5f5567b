"""The tests' threaded oracle driver (``pa_helpers.oracle_in_parallel``)
returns exactly what one oracle call over all pairs returns, in the same
order: it only cuts the pair list into chunks that run on several threads."""
import numpy as np

import oracle
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import oracle_decode, oracle_prefill


def test_threaded_decode_equals_one_call():
    b = W.random_decode(41, [1, 33, 200, 17, 64], 8, 2, 64, device="cpu", poison=True)
    out, lse = oracle_decode(b)
    ref, ref_lse = oracle.decode(oracle.KV_BF16, 16, 2, 8, 64, b.q_decode, b.k_pool, b.v_pool,
                                 b.block_tables_decode, b.context_lens_decode, b.scale)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    pairs = [(4, 7), (0, 0), (2, 3), (2, 3)]
    o2, l2 = oracle_decode(b, pairs=pairs)
    idx = [4 * 8 + 7, 0, 2 * 8 + 3, 2 * 8 + 3]
    assert np.array_equal(o2, ref[idx]) and np.array_equal(l2, ref_lse[idx])


def test_threaded_prefill_equals_one_call():
    b = W.random_prefill(42, [5, 40, 1], [21, 70, 16], 4, 2, 64, device="cpu", poison=True,
                         shared_prefix_blocks=1)
    out, lse = oracle_prefill(b)
    ref, ref_lse = oracle.prefill(oracle.KV_BF16, 16, 2, 4, 64, b.q_prefill, b.query_start_loc, b.k_pool, b.v_pool,
                                  b.block_tables_prefill, b.context_lens_prefill, b.scale)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
