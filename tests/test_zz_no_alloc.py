"""pa_decode_static: decode on the library's own fixed scratch array.

Callers that cannot allocate device memory where they decode (a serving loop
held to a fixed device-memory budget, a runtime whose memory is planned up
front, a plug-in whose host framework owns the allocator) use this entry
point instead of pa_decode with a workspace.  These tests call it through the
C ABI twice in a row and compare with pa_decode on the same inputs: the same
kernel on the same inputs, so the results must be identical, which is
stricter than the parity tests' tolerance.  A caller-owned error word in the
descriptor must stay zero.  The file sorts last so that a run that stops at
the first failure has already run every other test.
"""
import pytest
import torch

from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import desc_of, gpu_caches

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _both(b, caches):
    kc, vc = caches
    S = b.context_lens_decode.shape[0]
    base = desc_of(b)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(base.num_blocks, base.num_kv_heads, base.num_q_heads, base.head_dim, base.kv_dtype, base.k_scale,
                    base.v_scale, k_scales=b.k_scales, v_scales=b.v_scales, error_word=err)
    maxL = b.max_context_len_decode()
    ws = B.decode_workspace(d, S, maxL, DEV)
    ref = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    ref_lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    B.pa_decode(d, ref, b.q_decode, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL, b.scale, ws,
                lse=ref_lse)
    outs = []
    for _ in range(2):  # two calls in a row share the static array
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        B.pa_decode_static(d, out, b.q_decode, kc, vc, b.block_tables_decode, b.context_lens_decode, maxL,
                           b.scale, lse=lse)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert int(err[0]) == 0, "a kernel reported a device error"
    assert int(ws[:4].view(torch.int32)[0]) == 0
    return ref, ref_lse, outs


@pytest.mark.parametrize("n", [2, 3])
def test_static_decode_matches_pa_decode_on_two_calls(n):
    b = W.workload(n, device=DEV, poison=True)
    ref, ref_lse, outs = _both(b, gpu_caches(b))
    for out, lse in outs:
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_static_decode_fp8_after_bf16_call():
    b = W.random_decode(909, [1, 17, 300, 1025], 40, 8, 128, kv_dtype=W.KV_FP8, device=DEV, poison=True)
    ref, ref_lse, outs = _both(b, gpu_caches(b))
    for out, lse in outs:
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_static_decode_rejects_batches_beyond_its_scratch():
    d = B.make_desc(16, 1, 1, 128)
    need = B.pa_decode_workspace_size(d, 3_000_000, 16)
    assert need > (8 << 20)
    lib = B.load()
    st = lib.pa_decode_static(d, 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 1, 0x6000, 3_000_000, 16, 0.1,
                              None)
    assert st == B.PA_ERR_WORKSPACE
    assert "8 MiB" in B.last_error()
