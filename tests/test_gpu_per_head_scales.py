"""GPU parity of per-kv-head FP8 scales (``k_scales`` / ``v_scales`` of the
descriptor) against the fp64 oracle: cache writes bit-exact, decode (both
kernels) and prefill within the FP8 tolerance.  The kv heads carry values of
different magnitudes, each quantised with its own amax / format-max scale."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import (LSE_TOL, TOL, assert_close, desc_of, gpu_caches, gpu_decode,
                        gpu_prefill, oracle_caches, oracle_decode, oracle_prefill)

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = [W.KV_FP8, W.KV_FP8_E5M2]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


@pytest.mark.parametrize("kv", FMTS)
def test_cache_write_with_per_head_scales_is_bit_exact(kv):
    b = W.random_decode(31, [1, 16, 200, 777], 8, 4, 128, kv_dtype=kv, device=DEV, poison=False,
                        per_head_scales=True)
    kc, vc = gpu_caches(b)
    torch.cuda.synchronize()
    _, okc, ovc = oracle_caches(b)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    # the per-tensor arguments are not what the kernel used: per-head scales differ from them
    assert not torch.allclose(b.k_scales, torch.full_like(b.k_scales, b.k_scale))


@pytest.mark.parametrize("impl", [B.PA_DECODE_SIMT, B.PA_DECODE_MMA])
@pytest.mark.parametrize("D,Hq,Hkv,lens", [(128, 8, 4, [1, 15, 16, 17, 300, 2049]), (64, 4, 2, [7, 33, 250]),
                                           (128, 40, 8, [1, 100, 1025]), (128, 16, 2, [64, 65, 700])])
@pytest.mark.parametrize("kv", FMTS)
def test_decode_with_per_head_scales(kv, D, Hq, Hkv, lens, impl):
    if impl == B.PA_DECODE_SIMT and Hq // Hkv > 4:
        pytest.skip("the CUDA-core kernel takes group sizes up to 4")
    b = W.random_decode(40 + D + Hq, lens, Hq, Hkv, D, kv_dtype=kv, device=DEV, poison=True, per_head_scales=True)
    out, lse = gpu_decode(b, decode_impl=impl)
    o_ref, l_ref = oracle_decode(b)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


@pytest.mark.parametrize("kv", FMTS)
@pytest.mark.parametrize("impl", [B.PA_PREFILL_MMA_SYNC, B.PA_PREFILL_TCGEN05])
def test_prefill_with_per_head_scales(kv, impl):
    b = W.random_prefill(55, [5, 100, 1, 37], [5, 300, 33, 64], 8, 4, 128, kv_dtype=kv, device=DEV, poison=True,
                         shared_prefix_blocks=1, per_head_scales=True)
    out, lse = gpu_prefill(b, prefill_impl=impl)
    o_ref, l_ref = oracle_prefill(b)
    assert_close(out, o_ref, TOL[kv], "out")
    assert_close(lse, l_ref, LSE_TOL[kv], "lse")


def test_fp8_workload_with_per_head_scales():
    """Workload 4 with one scale per kv head, in full: bit-exact cache write of
    the whole pool and decode of all 128 sequences x 40 heads."""
    b = W.workload(4, device=DEV, poison=True, per_head_scales=True)
    caches = gpu_caches(b)
    out, lse = gpu_decode(b, caches=caches)
    code, okc, ovc = oracle_caches(b)
    assert np.array_equal(caches[0].cpu().numpy(), okc) and np.array_equal(caches[1].cpu().numpy(), ovc)
    o_ref, l_ref = oracle_decode(b, ocaches=(code, okc, ovc))
    assert_close(out, o_ref, TOL[W.KV_FP8], "out")
    assert_close(lse, l_ref, LSE_TOL[W.KV_FP8], "lse")
