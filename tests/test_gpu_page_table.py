"""Prefix-cache page bookkeeping on the GPU (pa_bind_blocks, pa_release_blocks)
against the oracle: page tables and owner counts bit-exact; the pages a
release returns to the pool compared as a set (their order in the free list
depends on the atomics and any order is valid), with the count exact."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import binding as B
from paged_kv_attention_14_gb300 import workloads as W
from pa_helpers import TOL, assert_close, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_14_gb300 import build
    B.load(build.build())


def _t(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=DEV)


def _scenario(seed, NB=4096, rows=256, MB=300, n_hits=200):
    rng = np.random.default_rng(seed)
    tables = np.full((rows, MB), -1, np.int32)
    refc = rng.integers(0, 4, NB).astype(np.int32)
    entries = [rng.permutation(NB)[:rng.integers(1, 60)].astype(np.int32) for _ in range(12)]
    seq_rows = rng.permutation(rows)[:n_hits].astype(np.int32)
    hits = []
    for _ in range(n_hits):
        e = entries[rng.integers(0, len(entries))]
        own = rng.permutation(NB)[:rng.integers(0, MB - 60)].astype(np.int32)
        hits.append(np.concatenate([e[:rng.integers(0, len(e) + 1)], own])[:MB])
    start = np.concatenate([[0], np.cumsum([len(h) for h in hits])]).astype(np.int32)
    return tables, refc, seq_rows, start, np.concatenate(hits).astype(np.int32), hits


def test_bind_blocks_bit_exact():
    tables, refc, rows, start, flat, hits = _scenario(31)
    d = B.make_desc(refc.shape[0], 8, 32, 128)
    bt, rc = _t(tables), _t(refc)
    B.pa_bind_blocks(d, bt, _t(rows), _t(start), _t(flat), rc)
    torch.cuda.synchronize()
    want_t, want_rc, err = oracle.bind_blocks(tables, rows, start, flat, refc)
    assert err == 0
    assert np.array_equal(bt.cpu().numpy(), want_t) and np.array_equal(rc.cpu().numpy(), want_rc)


def test_release_blocks_counts_exact_and_free_set_equal():
    tables, refc, rows, start, flat, hits = _scenario(32)
    bound_t, bound_rc, _ = oracle.bind_blocks(tables, rows, start, flat, refc)
    rng = np.random.default_rng(33)
    rel = rng.permutation(len(rows))[:120]
    rel_rows = rows[rel]
    counts = np.array([len(hits[i]) - int(rng.integers(0, 3)) if len(hits[i]) > 2 else len(hits[i])
                       for i in rel], np.int32)
    d = B.make_desc(refc.shape[0], 8, 32, 128)
    bt, rc = _t(bound_t), _t(bound_rc)
    free = torch.full((refc.shape[0],), -7, dtype=torch.int32, device=DEV)
    nfree = torch.tensor([5], dtype=torch.int32, device=DEV)  # five pages already in the pool's list
    B.pa_release_blocks(d, bt, _t(rel_rows), _t(counts), rc, free, nfree)
    torch.cuda.synchronize()
    want_t, want_rc, want_free, err = oracle.release_blocks(bound_t, rel_rows, counts, bound_rc)
    assert err == 0
    assert np.array_equal(bt.cpu().numpy(), want_t) and np.array_equal(rc.cpu().numpy(), want_rc)
    n = int(nfree[0])
    assert n == 5 + want_free.shape[0]
    got = free.cpu().numpy()
    assert np.all(got[:5] == -7) and np.all(got[n:] == -7)
    assert sorted(got[5:n].tolist()) == sorted(want_free.tolist())


def test_bookkeeping_errors_are_reported_and_skipped():
    NB = 16
    ew = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = B.make_desc(NB, 2, 4, 64, error_word=ew)
    refc = np.zeros(NB, np.int32)
    refc[1] = 1
    tables = np.array([[0, 1, 22, -1]], np.int32)
    bt, rc = _t(tables), _t(refc)
    free = torch.zeros(NB, dtype=torch.int32, device=DEV)
    nfree = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_release_blocks(d, bt, _t([0]), _t([3]), rc, free, nfree)
    torch.cuda.synchronize()
    want_t, want_rc, want_free, err = oracle.release_blocks(tables, np.array([0], np.int32),
                                                            np.array([3], np.int32), refc)
    assert err == 2
    assert int(ew[0]) == B.PA_DEVERR_REFCOUNT | B.PA_DEVERR_BAD_INDEX
    assert np.array_equal(bt.cpu().numpy(), want_t) and np.array_equal(rc.cpu().numpy(), want_rc)
    assert int(nfree[0]) == 1 and int(free[0]) == 1
    # a hit naming a page outside the pool, and a row outside the table
    ew.zero_()
    B.pa_bind_blocks(d, bt, _t([0, 5]), _t([0, 2, 3]), _t([3, NB + 1, 4]), rc)
    torch.cuda.synchronize()
    assert int(ew[0]) == B.PA_DEVERR_BAD_INDEX
    assert bt.cpu().numpy().tolist() == [[3, -1, 22, -1]]  # entry 1 was released above; the bad page is skipped


def test_decode_through_device_bound_prefix_pages():
    """A prefix-cache hit end to end: three new sequences are bound to the
    pages of a cached 4096-token prefix plus fresh pages of their own by
    pa_bind_blocks, and decode over the device-built tables matches the
    oracle decoding through the oracle's own bind of the same hits."""
    b = W.shared_prefix_decode(34, [3], [4096], [100, 17, 250], 32, 8, 128, device=DEV, poison=True)
    host_t = b.block_tables_decode.cpu().numpy()
    nb = (b.context_lens_decode.cpu().numpy() + 15) // 16
    S, MB = host_t.shape
    hits = [host_t[i, :nb[i]] for i in range(S)]
    start = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
    flat = np.concatenate(hits).astype(np.int32)
    refc = np.zeros(b.num_blocks, np.int32)
    d = B.make_desc(b.num_blocks, 8, 32, 128)
    bt = torch.full((S, MB), -1, dtype=torch.int32, device=DEV)
    rc = _t(refc)
    B.pa_bind_blocks(d, bt, _t(np.arange(S)), _t(start), _t(flat), rc)
    torch.cuda.synchronize()
    want_t, want_rc, _ = oracle.bind_blocks(np.full((S, MB), -1, np.int32), np.arange(S, dtype=np.int32), start,
                                            flat, refc)
    assert np.array_equal(bt.cpu().numpy(), want_t) and np.array_equal(rc.cpu().numpy(), want_rc)
    # the shared prefix pages have three owners, the own pages one
    assert int(rc[int(host_t[0, 0])]) == 3 and int(rc[int(host_t[0, nb[0] - 1])]) == 1
    kc, vc = b.k_pool, b.v_pool
    out = torch.empty(S, 32, 128, device=DEV)
    ws = B.decode_workspace(d, S, b.max_context_len_decode(), DEV)
    B.pa_decode(d, out, b.q_decode, kc, vc, bt, b.context_lens_decode, b.max_context_len_decode(), b.scale, ws)
    torch.cuda.synchronize()
    # the oracle side decodes through its own bind (want_t)
    b.block_tables_decode = torch.as_tensor(want_t)
    o_ref, _ = oracle_decode(b)
    assert_close(out, o_ref, TOL[W.KV_BF16], "out")
