"""Decode outputs in pinned host memory: the decode entry points take an
``out`` / ``lse`` that unified addressing maps from pinned host memory, and
the kernels store the result there.  It must equal the device-resident result
bit for bit, for both decode kernels and every decode entry point."""
import pytest
import torch

from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import desc_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _host_like(t):
    return torch.full(tuple(t.shape), float("nan"), dtype=t.dtype).pin_memory()


def _pair(b, impl):
    S = b.context_lens_decode.shape[0]
    out = torch.full((S, b.num_q_heads, b.head_dim), float("nan"), device=DEV)
    lse = torch.full((S, b.num_q_heads), float("nan"), device=DEV)
    return out, lse, _host_like(out), _host_like(lse), desc_of(b, decode_impl=impl), S, b.max_context_len_decode()


@pytest.mark.parametrize("impl", [B.PA_DECODE_MMA, B.PA_DECODE_SIMT])
@pytest.mark.parametrize("lens", [[512, 4096, 1, 0, 2049, 33], [16] * 40 + [3000]])
def test_pa_decode_writes_host_output_bit_for_bit(impl, lens):
    b = W.random_decode(1201 + len(lens), lens, 32, 8, 128, device=DEV, poison=True)
    out, lse, hout, hlse, d, S, maxL = _pair(b, impl)
    for o, l in ((out, lse), (hout, hlse)):
        B.pa_decode(d, o, b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode, b.context_lens_decode, maxL,
                    b.scale, B.decode_workspace(d, S, maxL, DEV), lse=l)
    torch.cuda.synchronize()
    assert torch.equal(hout, out.cpu()) and torch.equal(hlse, lse.cpu())


def test_pa_decode_append_and_static_write_host_output():
    b = W.workload(2, device=DEV, poison=False)
    out, lse, hout, hlse, d, S, maxL = _pair(b, B.PA_DECODE_MMA)
    for o, l in ((out, lse), (hout, hlse)):
        kc, vc = b.k_pool.clone(), b.v_pool.clone()
        B.pa_decode_append(d, o, b.q_decode, b.k_new, b.v_new, kc, vc, b.block_tables_decode, b.context_lens_decode,
                           maxL, b.scale, B.decode_workspace(d, S, maxL, DEV), lse=l)
    torch.cuda.synchronize()
    assert torch.equal(hout, out.cpu()) and torch.equal(hlse, lse.cpu())
    hout2, hlse2 = _host_like(out), _host_like(lse)
    B.pa_decode_static(d, hout2, b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode, b.context_lens_decode, maxL,
                       b.scale, lse=hlse2)
    torch.cuda.synchronize()
    assert torch.equal(hout2, out.cpu()) and torch.equal(hlse2, lse.cpu())


def test_unpinned_host_output_is_refused():
    b = W.random_decode(1210, [40, 17], 8, 2, 128, device=DEV, poison=False)
    d = desc_of(b)
    with pytest.raises(ValueError):
        B.pa_decode(d, torch.empty(2, 8, 128), b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode,
                    b.context_lens_decode, 40, b.scale, B.decode_workspace(d, 2, 40, DEV))
