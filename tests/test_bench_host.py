"""Host-side accounting of bench.py against brute force: the algorithmic KV
bytes of a decode step and the algorithmic flops of the prefill chunks, with
and without local attention (the figures every bench number divides by)."""
import sys

import pytest
import torch

import bench
from paged_kv_attention_14_gb300 import workloads as W


def _visible(pos, window, chunk):
    """Brute force: the keys a query at `pos` may see, listed one by one."""
    return [t for t in range(pos + 1)
            if (not window or t > pos - window) and (not chunk or t // chunk == pos // chunk)]


@pytest.mark.parametrize("window,chunk", [(0, 0), (1, 0), (100, 0), (0, 64), (0, 1000), (50, 64)])
def test_decode_kv_bytes_count_each_visible_key_once(window, chunk):
    b = W.random_decode(5, [1, 17, 250, 1031], 8, 2, 64, poison=False)
    want = sum(len(_visible(L - 1, window, chunk)) for L in b.context_lens_decode.tolist()) * 2 * 64 * 2 * 2
    assert bench._decode_kv_bytes(b, window, chunk) == want
    if not window and not chunk:
        assert want == b.decode_kv_bytes()


@pytest.mark.parametrize("window,chunk", [(0, 0), (7, 0), (0, 32), (20, 48)])
def test_prefill_flops_count_each_visible_query_key_pair(window, chunk):
    b = W.random_prefill(6, [5, 40, 1], [5, 100, 33], 4, 2, 64, poison=False)
    qsl = b.query_start_loc.tolist()
    pairs = 0
    for s, L in enumerate(b.context_lens_prefill.tolist()):
        n = qsl[s + 1] - qsl[s]
        pairs += sum(len(_visible(p, window, chunk)) for p in range(L - n, L))
    assert bench._prefill_flops(b, window, chunk) == pairs * 4 * 64 * 4


def test_first_key_matches_the_library_rule():
    for pos in range(0, 300, 7):
        for window, chunk in [(0, 0), (1, 0), (16, 0), (0, 16), (10, 32)]:
            vis = _visible(pos, window, chunk)
            assert bench._first_key(pos, window, chunk) == vis[0]


def test_job_throughput_and_flags():
    assert bench._job_throughput(4, 100.0, 2.0) == 200.0
    sys_argv = sys.argv
    try:
        sys.argv = ["bench.py", "--fp16", "--workload", "4"]
        with pytest.raises(SystemExit):
            bench.main()
        sys.argv = ["bench.py", "--per-head-scales", "--workload", "2"]
        with pytest.raises(SystemExit):
            bench.main()
        sys.argv = ["bench.py", "--warmup", "2"]
        with pytest.raises(SystemExit):
            bench.main()
    finally:
        sys.argv = sys_argv
