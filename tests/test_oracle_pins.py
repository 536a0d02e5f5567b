"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a library routine (torch's CPU SDPA and
its float8_e4m3fn / float8_e5m2 codecs, numpy's float16), a closed form, an invariant, or the format
definition's fixed points -- chosen so that a plausible slip anywhere in the
oracle (wrong GQA index, wrong block offset, a dropped scale, an off-by-one in
the causal position, a sign in the merge, an exponent bias) fails one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_14_gb300 import workloads as W

BF16, FP8, E5M2, F16 = oracle.KV_BF16, oracle.KV_FP8_E4M3, oracle.KV_FP8_E5M2, oracle.KV_F16
#: 16-bit cache types: generator name -> oracle code
_KV16 = {W.KV_BF16: BF16, W.KV_F16: F16}
#: generator cache type -> (oracle code, torch 8-bit dtype)
_FP8_KINDS = {W.KV_FP8: (FP8, torch.float8_e4m3fn), W.KV_FP8_E5M2: (E5M2, torch.float8_e5m2)}


# ------------------------------------------------------------ helpers (independent)

def _bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _fp8_cache_to_f64(cache_u8: np.ndarray, scale: float, dtype=torch.float8_e4m3fn) -> np.ndarray:
    """Decode 8-bit cache bytes with torch's own float8 codec (library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(cache_u8)).view(dtype)
    return t.to(torch.float64).numpy() * float(scale)


def _f32(x) -> float:
    return float(np.float32(x))


def _dense_kv(pool_f64: np.ndarray, table_row, L, kh):
    """Gather logical tokens [0, L) of kv head kh with numpy fancy indexing."""
    t = np.arange(L)
    blk = np.asarray(table_row)[t // W.BLOCK_SIZE]
    return pool_f64[blk, kh, t % W.BLOCK_SIZE, :]


def _sdpa(q, k, v, scale, mask=None):
    """torch CPU scaled_dot_product_attention in float64 (library routine).
    The scale is an fp32 argument of the library, hence rounded to fp32 here."""
    scale = _f32(scale)
    q = torch.from_numpy(np.asarray(q, np.float64))[None, None]
    k = torch.from_numpy(np.asarray(k, np.float64))[None, None]
    v = torch.from_numpy(np.asarray(v, np.float64))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)[0, 0].numpy()


def _oracle_caches(b: W.PagedBatch):
    """Caches as the oracle reads them: bf16 pool as-is, or the E4M3 / E5M2
    encoding of the whole (small) pool made by the oracle's own cache write."""
    if b.kv_dtype in _KV16:
        return _KV16[b.kv_dtype], b.k_pool, b.v_pool
    code = _FP8_KINDS[b.kv_dtype][0]
    k, v, slots = b.pool_tokens_as_rows()
    z = np.zeros(tuple(b.k_pool.shape), np.uint8)
    kc, vc = oracle.cache_write(code, b.block_size, b.num_kv_heads, b.head_dim, k, v, slots, z, z,
                                b.k_scale, b.v_scale, k_scales=b.k_scales, v_scales=b.v_scales)
    return code, kc, vc


def _dense_pools(b: W.PagedBatch, kc, vc):
    """K and V pools in fp64: the bf16 / fp16 pool, or the 8-bit caches decoded by torch."""
    if b.kv_dtype in _KV16:
        return _bf16_to_f64(b.k_pool), _bf16_to_f64(b.v_pool)
    dt = _FP8_KINDS[b.kv_dtype][1]
    if b.k_scales is not None:  # per-kv-head scales
        ks = b.k_scales.double().numpy()[None, :, None, None]
        vs = b.v_scales.double().numpy()[None, :, None, None]
        return _fp8_cache_to_f64(kc, 1.0, dt) * ks, _fp8_cache_to_f64(vc, 1.0, dt) * vs
    return _fp8_cache_to_f64(kc, b.k_scale, dt), _fp8_cache_to_f64(vc, b.v_scale, dt)


def _oracle_decode(b: W.PagedBatch, pairs=None):
    kd, kc, vc = _oracle_caches(b)
    return oracle.decode(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode,
                         kc, vc, b.block_tables_decode, b.context_lens_decode, b.scale,
                         b.k_scale, b.v_scale, pairs=pairs, k_scales=b.k_scales, v_scales=b.v_scales)


# ------------------------------------------------------------------ E4M3 codec

def test_e4m3_fixed_points_of_the_format_definition():
    # OCP FP8 E4M3: bias 7, max finite 448, min normal 2^-6, min subnormal 2^-9,
    # no infinities, S.1111.111 is NaN
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x00) == 0.0 and math.copysign(1, oracle.e4m3_decode(0x80)) == -1
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    assert oracle.e4m3_decode(0x78) == 256.0  # exponent field 15, mantissa 0 is finite


def test_e4m3_decode_matches_torch_float8_for_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.all(both_nan | (ref == mine))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(mine[~both_nan]))
    finite_pos = mine[:0x7F]
    assert np.all(np.diff(finite_pos) > 0), "positive codes must be strictly increasing"


def test_e4m3_encode_matches_torch_rne_inside_the_finite_range():
    rng = np.random.default_rng(5)
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (pos[1:] + pos[:-1]) / 2  # exact ties: round half to even
    xs = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 60, 2000), rng.uniform(-448, 448, 2000),
                         mids, -mids, pos, -pos, [2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -12, 447.99, 463.9]])
    xs = xs.astype(np.float32)  # the encoder's input is an fp32 quotient
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(ref, mine), np.nonzero(ref != mine)


def test_e4m3_encode_saturates_and_keeps_nan_and_signed_zero():
    # the chosen reading: finite overflow saturates to +-448 (torch's codec,
    # which is non-saturating, returns NaN there instead)
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80  # rounds to zero, keeps the sign
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


# ------------------------------------------------------------------ E5M2 codec

def test_e5m2_fixed_points_of_the_format_definition():
    # OCP FP8 E5M2: bias 15, max finite 57344, min normal 2^-14, min subnormal
    # 2^-16, exponent field 31 is inf (mantissa 0) or NaN
    assert oracle.e5m2_decode(0x7B) == 57344.0
    assert oracle.e5m2_decode(0xFB) == -57344.0
    assert oracle.e5m2_decode(0x3C) == 1.0
    assert oracle.e5m2_decode(0x04) == 2.0 ** -14
    assert oracle.e5m2_decode(0x03) == 3 * 2.0 ** -16
    assert oracle.e5m2_decode(0x01) == 2.0 ** -16
    assert oracle.e5m2_decode(0x00) == 0.0 and math.copysign(1, oracle.e5m2_decode(0x80)) == -1
    assert oracle.e5m2_decode(0x7C) == math.inf and oracle.e5m2_decode(0xFC) == -math.inf
    assert all(math.isnan(oracle.e5m2_decode(c)) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))


def test_e5m2_decode_matches_torch_float8_for_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    mine = np.array([oracle.e5m2_decode(int(c)) for c in codes])
    same = (ref == mine) | (np.isnan(ref) & np.isnan(mine))
    assert same.all(), np.nonzero(~same)


def test_e5m2_encode_matches_torch_rne_inside_the_finite_range():
    rng = np.random.default_rng(6)
    pos = np.array([oracle.e5m2_decode(c) for c in range(0x7C)])
    mids = (pos[1:] + pos[:-1]) / 2  # exact ties: round half to even
    xs = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 4000, 2000), rng.uniform(-57344, 57344, 2000),
                         mids, -mids, pos, -pos, [2.0 ** -17, 3 * 2.0 ** -17, 2.0 ** -18, 57343.0, 61439.0]])
    xs = xs.astype(np.float32)  # the encoder's input is an fp32 quotient
    ref = torch.from_numpy(xs).to(torch.float8_e5m2).view(torch.uint8).numpy()
    mine = np.array([oracle.e5m2_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(ref, mine), np.nonzero(ref != mine)


def test_e5m2_encode_saturates_and_keeps_nan_and_signed_zero():
    # the chosen reading: finite overflow and +-inf saturate to +-57344 (torch's
    # non-saturating codec returns inf from 61440 on)
    assert oracle.e5m2_encode(61440.0) == 0x7B
    assert oracle.e5m2_encode(1e9) == 0x7B
    assert oracle.e5m2_encode(-1e30) == 0xFB
    assert oracle.e5m2_encode(float("inf")) == 0x7B
    assert oracle.e5m2_encode(float("-inf")) == 0xFB
    assert oracle.e5m2_encode(float("nan")) == 0x7F
    assert oracle.e5m2_encode(-0.0) == 0x80
    assert oracle.e5m2_encode(-2.0 ** -18) == 0x80  # rounds to zero, keeps the sign
    for c in list(range(0x7C)) + list(range(0x80, 0xFC)):
        assert oracle.e5m2_encode(oracle.e5m2_decode(c)) == c


def test_f16_decode_matches_numpy_float16_for_all_65536_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_decode(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # fixed points of the binary16 definition
    assert oracle.f16_decode(0x3C00) == 1.0 and oracle.f16_decode(0x7BFF) == 65504.0
    assert oracle.f16_decode(0x0001) == 2.0 ** -24 and oracle.f16_decode(0x0400) == 2.0 ** -14
    assert oracle.f16_decode(0xFC00) == -math.inf and math.copysign(1, oracle.f16_decode(0x8000)) < 0


# --------------------------------------------------------------- cache write

@pytest.mark.parametrize("fp16", [False, True])
def test_cache_write_16bit_is_a_scatter_of_bit_patterns(fp16):
    b = W.workload(5, poison=True, fp16=fp16)
    kc, vc = oracle.cache_write(F16 if fp16 else BF16, 16, 8, 128, b.k_new, b.v_new, b.slot_mapping,
                                b.k_pool, b.v_pool)
    ref_k = b.k_pool.view(torch.int16).numpy().view(np.uint16).copy()
    ref_v = b.v_pool.view(torch.int16).numpy().view(np.uint16).copy()
    s = b.slot_mapping.numpy()
    ref_k[s // 16, :, s % 16, :] = b.k_new.view(torch.int16).numpy().view(np.uint16)
    ref_v[s // 16, :, s % 16, :] = b.v_new.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


@pytest.mark.parametrize("kv", [W.KV_FP8, W.KV_FP8_E5M2])
def test_cache_write_skips_negative_slots_and_fp8_matches_torch_quantisation(kv):
    code, tdt = _FP8_KINDS[kv]
    g = torch.Generator().manual_seed(3)
    T, H, D, NB = 40, 2, 64, 8
    k = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    v = (3 * torch.randn(T, H, D, generator=g)).to(torch.bfloat16)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[::7] = -1
    ks = float(k.float().abs().max()) / W.FP8_MAX[kv]
    vs = float(v.float().abs().max()) / W.FP8_MAX[kv]
    z = np.full((NB, H, 16, D), 0xAB, np.uint8)
    kc, vc = oracle.cache_write(code, 16, H, D, k, v, slots, z, z, ks, vs)
    ref_k = z.copy()
    ref_v = z.copy()
    keep = slots >= 0
    s = slots[keep].numpy()
    qk = (k[keep].float() / torch.tensor(ks, dtype=torch.float32)).to(tdt).view(torch.uint8)
    qv = (v[keep].float() / torch.tensor(vs, dtype=torch.float32)).to(tdt).view(torch.uint8)
    ref_k[s // 16, :, s % 16, :] = qk.numpy()
    ref_v[s // 16, :, s % 16, :] = qv.numpy()
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


@pytest.mark.parametrize("kv", [W.KV_FP8, W.KV_FP8_E5M2])
def test_cache_write_per_head_scales_match_torch_quantisation_per_head(kv):
    code, tdt = _FP8_KINDS[kv]
    g = torch.Generator().manual_seed(4)
    T, H, D, NB = 33, 3, 64, 6
    f = torch.tensor([0.25, 1.0, 8.0])[None, :, None]
    k = (torch.randn(T, H, D, generator=g) * f).to(torch.bfloat16)
    v = (torch.randn(T, H, D, generator=g) / f).to(torch.bfloat16)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    ks = (k.float().abs().amax(dim=(0, 2)) / W.FP8_MAX[kv]).float()
    vs = (v.float().abs().amax(dim=(0, 2)) / W.FP8_MAX[kv]).float()
    z = np.zeros((NB, H, 16, D), np.uint8)
    # the per-tensor arguments are deliberately wrong: the per-head ones win
    kc, vc = oracle.cache_write(code, 16, H, D, k, v, slots, z, z, 123.0, 456.0, k_scales=ks, v_scales=vs)
    s = slots.numpy()
    qk = (k.float() / ks[None, :, None]).to(tdt).view(torch.uint8).numpy()
    qv = (v.float() / vs[None, :, None]).to(tdt).view(torch.uint8).numpy()
    ref_k, ref_v = z.copy(), z.copy()
    ref_k[s // 16, :, s % 16, :] = qk
    ref_v[s // 16, :, s % 16, :] = qv
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def test_per_head_scales_all_equal_to_the_tensor_scale_change_nothing():
    b = W.random_decode(17, [3, 40, 100], 8, 4, 64, kv_dtype=W.KV_FP8, poison=True)
    kd, kc, vc = _oracle_caches(b)
    args = (kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode, kc, vc,
            b.block_tables_decode, b.context_lens_decode, b.scale, b.k_scale, b.v_scale)
    o1, l1 = oracle.decode(*args)
    o2, l2 = oracle.decode(*args, k_scales=np.full(4, b.k_scale, np.float32), v_scales=np.full(4, b.v_scale, np.float32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------------------ decode attention

@pytest.mark.parametrize("kv,per_head", [(W.KV_BF16, False), (W.KV_F16, False), (W.KV_FP8, False),
                                         (W.KV_FP8_E5M2, False), (W.KV_FP8, True), (W.KV_FP8_E5M2, True)])
@pytest.mark.parametrize("D,Hq,Hkv", [(8, 2, 2), (64, 4, 2), (8, 10, 2), (64, 5, 1)])
def test_decode_matches_bruteforce_sdpa(kv, per_head, D, Hq, Hkv):
    lens = [1, 5, 16, 17, 40]
    b = W.random_decode(11 + D + Hq, lens, Hq, Hkv, D, kv_dtype=kv, poison=True, per_head_scales=per_head)
    out, lse = _oracle_decode(b)
    kd, kc, vc = _oracle_caches(b)
    kf, vf = _dense_pools(b, kc, vc)
    g = Hq // Hkv
    qf = _bf16_to_f64(b.q_decode)
    for s, L in enumerate(lens):
        for h in range(Hq):
            K = _dense_kv(kf, b.block_tables_decode[s].numpy(), L, h // g)
            V = _dense_kv(vf, b.block_tables_decode[s].numpy(), L, h // g)
            ref = _sdpa(qf[s, h][None], K, V, b.scale)[0]
            i = s * Hq + h
            np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)
            x = _f32(b.scale) * K @ qf[s, h]
            ref_lse = x.max() + math.log(np.exp(x - x.max()).sum())
            assert abs(lse[i] - ref_lse) < 1e-12


def test_decode_context_length_one_returns_v_exactly():
    b = W.workload(1, poison=True)
    out, lse = _oracle_decode(b)
    s = 0  # context length 1
    blk = int(b.block_tables_decode[0, 0])
    for h in range(4):
        v0 = b.v_pool[blk, h // 2, 0].to(torch.float64).numpy()
        assert np.array_equal(out[s * 4 + h], v0)


def test_decode_identical_keys_or_zero_query_give_mean_of_v():
    b = W.random_decode(21, [3, 16, 37], 4, 2, 64, poison=True)
    # identical keys: every cached key row of every block equals one vector
    kpool = b.k_pool.clone()
    kpool[:] = kpool[int(b.block_tables_decode[0, 0]), 0, 0].clone()
    b.k_pool = kpool
    out, _ = _oracle_decode(b)
    qzero = W.random_decode(21, [3, 16, 37], 4, 2, 64, poison=True)
    qzero.q_decode = torch.zeros_like(qzero.q_decode)
    out0, lse0 = _oracle_decode(qzero)
    vf = _bf16_to_f64(b.v_pool)
    for s, L in enumerate([3, 16, 37]):
        for h in range(4):
            mean_v = _dense_kv(vf, b.block_tables_decode[s].numpy(), L, h // 2).mean(0)
            np.testing.assert_allclose(out[s * 4 + h], mean_v, atol=1e-12, rtol=0)
            np.testing.assert_allclose(out0[s * 4 + h], mean_v, atol=1e-12, rtol=0)
            assert abs(lse0[s * 4 + h] - math.log(L)) < 1e-12


def test_decode_weights_sum_to_one_and_output_is_linear_in_v():
    b = W.random_decode(31, [9, 33], 4, 2, 64, poison=True)
    base = b.v_pool.clone()
    b.v_pool = torch.where(torch.isnan(base), base, torch.ones_like(base))
    ones, _ = _oracle_decode(b)
    np.testing.assert_allclose(ones, 1.0, atol=1e-13, rtol=0)
    b.v_pool = base
    o1, _ = _oracle_decode(b)
    b.v_pool = (2 * base.float()).to(torch.bfloat16)  # exact doubling in bf16
    o2, _ = _oracle_decode(b)
    np.testing.assert_allclose(o2, 2 * o1, atol=1e-12, rtol=0)


def test_decode_dominant_key_selects_its_value():
    b = W.random_decode(41, [20], 2, 1, 64, poison=True)
    q = b.q_decode[0, 0].float()
    blk = int(b.block_tables_decode[0, 13 // 16])
    kp = b.k_pool.clone()
    kp[blk, 0, 13 % 16] = (q * 40).to(torch.bfloat16)  # score gap far above 60
    b.k_pool = kp
    out, _ = _oracle_decode(b)
    v13 = b.v_pool[blk, 0, 13].to(torch.float64).numpy()
    np.testing.assert_allclose(out[0], v13, atol=1e-12, rtol=0)


def test_decode_invariant_under_permuting_physical_blocks():
    b = W.random_decode(51, [7, 16, 40, 33], 4, 2, 64, poison=True)
    out, lse = _oracle_decode(b)
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks)
    b2 = W.random_decode(51, [7, 16, 40, 33], 4, 2, 64, poison=True)
    b2.k_pool = b.k_pool[inv]  # new block j holds old block inv[j] ... so old block i moves to perm[i]
    b2.v_pool = b.v_pool[inv]
    t = b.block_tables_decode.clone().long()
    b2.block_tables_decode = torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32)
    out2, lse2 = _oracle_decode(b2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_decode_never_reads_poisoned_slots():
    for n in (1,):
        b = W.workload(n, poison=True)
        out, lse = _oracle_decode(b)
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    b = W.random_decode(61, [1, 15, 17, 31, 32], 10, 2, 8, kv_dtype=W.KV_FP8, poison=True)
    out, _ = _oracle_decode(b)
    assert np.all(np.isfinite(out))


def test_decode_pairs_subset_equals_full():
    b = W.random_decode(71, [12, 29], 4, 2, 64, poison=True)
    full, lf = _oracle_decode(b)
    pairs = [(1, 3), (0, 0), (1, 1)]
    sub, ls = _oracle_decode(b, pairs=pairs)
    for i, (s, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[s * 4 + h]) and ls[i] == lf[s * 4 + h]


# ------------------------------------------------------------------ merge

def test_merge_of_split_ranges_equals_unsplit():
    b = W.random_decode(81, [45], 2, 1, 64, poison=True)
    row = b.block_tables_decode[0]
    q = b.q_decode[0, 1]
    full, lf = oracle.attend_range(BF16, 16, 1, 64, q, b.k_pool, b.v_pool, row, 0, 0, 45, b.scale)
    for cuts in ([17], [1, 30], [16, 32, 44], [0, 45]):
        edges = [0] + cuts + [45]
        parts = [oracle.attend_range(BF16, 16, 1, 64, q, b.k_pool, b.v_pool, row, 0, a, c, b.scale)
                 for a, c in zip(edges[:-1], edges[1:])]
        mo, ml = oracle.merge(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
        np.testing.assert_allclose(mo, full, atol=1e-12, rtol=0)
        assert abs(ml - lf) < 1e-12


def test_merge_closed_forms():
    o = np.array([[1.0, 2.0], [3.0, -4.0]])
    mo, ml = oracle.merge(o, np.array([0.7, 0.7]))
    np.testing.assert_allclose(mo, [2.0, -1.0], atol=1e-15)
    assert abs(ml - (0.7 + math.log(2))) < 1e-15
    mo, ml = oracle.merge(o, np.array([-np.inf, 1.5]))
    np.testing.assert_array_equal(mo, o[1])
    assert ml == 1.5
    mo, ml = oracle.merge(o, np.array([-np.inf, -np.inf]))
    assert np.all(mo == 0) and ml == -np.inf
    # weights e^1 : e^0
    mo, _ = oracle.merge(o, np.array([1.0, 0.0]))
    w = math.e / (math.e + 1)
    np.testing.assert_allclose(mo, w * o[0] + (1 - w) * o[1], atol=1e-15)


# ----------------------------------------------------------------- prefill

def _oracle_prefill(b: W.PagedBatch, pairs=None):
    kd, kc, vc = _oracle_caches(b)
    return oracle.prefill(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_prefill,
                          b.query_start_loc, kc, vc, b.block_tables_prefill, b.context_lens_prefill,
                          b.scale, b.k_scale, b.v_scale, pairs=pairs, k_scales=b.k_scales, v_scales=b.v_scales)


@pytest.mark.parametrize("kv,per_head", [(W.KV_BF16, False), (W.KV_F16, False), (W.KV_FP8, False),
                                         (W.KV_FP8_E5M2, False), (W.KV_FP8, True), (W.KV_FP8_E5M2, True)])
def test_prefill_matches_bruteforce_sdpa_with_causal_mask(kv, per_head):
    q_lens, ctx = [5, 16, 1, 23], [5, 40, 33, 64]
    b = W.random_prefill(91, q_lens, ctx, 4, 2, 64, kv_dtype=kv, shared_prefix_blocks=1, per_head_scales=per_head)
    out, _ = _oracle_prefill(b)
    kd, kc, vc = _oracle_caches(b)
    kf, vf = _dense_pools(b, kc, vc)
    qf = _bf16_to_f64(b.q_prefill)
    qsl = b.query_start_loc.numpy()
    for s, (n, L) in enumerate(zip(q_lens, ctx)):
        for h in range(4):
            K = _dense_kv(kf, b.block_tables_prefill[s].numpy(), L, h // 2)
            V = _dense_kv(vf, b.block_tables_prefill[s].numpy(), L, h // 2)
            Q = qf[qsl[s]:qsl[s] + n, h]
            # bottom-right aligned causal mask: query i sits at key position L - n + i
            mask = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]
            ref = _sdpa(Q, K, V, b.scale, mask)
            got = out[(qsl[s] + np.arange(n)) * 4 + h]
            np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def test_prefill_single_query_equals_decode():
    lens = [7, 16, 41]
    d = W.random_decode(101, lens, 4, 2, 64, poison=True)
    p = W.random_prefill(101, [1, 1, 1], lens, 4, 2, 64)
    p.q_prefill = d.q_decode.clone()
    p.k_pool, p.v_pool = d.k_pool, d.v_pool
    p.block_tables_prefill = d.block_tables_decode
    p.context_lens_prefill = d.context_lens_decode
    po, pl = _oracle_prefill(p)
    do, dl = _oracle_decode(d)
    assert np.array_equal(po, do) and np.array_equal(pl, dl)


def test_prefill_in_two_chunks_equals_one_chunk():
    b = W.random_prefill(111, [30], [50], 4, 2, 64)
    one, _ = _oracle_prefill(b)
    # first chunk: 12 queries while only 32 tokens exist; then the last 18
    first = W.random_prefill(111, [30], [50], 4, 2, 64)
    first.q_prefill = b.q_prefill[:12].clone()
    first.query_start_loc = torch.tensor([0, 12], dtype=torch.int32)
    first.context_lens_prefill = torch.tensor([32], dtype=torch.int32)
    o1, _ = _oracle_prefill(first)
    second = W.random_prefill(111, [30], [50], 4, 2, 64)
    second.q_prefill = b.q_prefill[12:].clone()
    second.query_start_loc = torch.tensor([0, 18], dtype=torch.int32)
    o2, _ = _oracle_prefill(second)
    assert np.array_equal(np.concatenate([o1, o2]), one)


def test_prefill_shared_prefix_blocks_are_read_by_every_sequence():
    b = W.random_prefill(121, [4, 4, 4], [40, 40, 40], 2, 1, 8, shared_prefix_blocks=2)
    t = b.block_tables_prefill
    assert torch.equal(t[0, :2], t[1, :2]) and torch.equal(t[1, :2], t[2, :2])
    out, _ = _oracle_prefill(b)
    assert np.all(np.isfinite(out))
    # each sequence's queries see the shared keys: zeroing them changes every output
    b2 = W.random_prefill(121, [4, 4, 4], [40, 40, 40], 2, 1, 8, shared_prefix_blocks=2)
    vp = b2.v_pool.clone()
    vp[t[0, :2].long()] = 0
    b2.v_pool = vp
    out2, _ = _oracle_prefill(b2)
    for s in range(3):
        rows = slice(s * 4 * 2, (s + 1) * 4 * 2)
        assert not np.allclose(out[rows], out2[rows])


# ------------------------------------------------------ local attention

def _band_mask(n_q, L, first_pos, window=0, chunk=0):
    """Query rows at positions first_pos .. first_pos + n_q - 1 over keys 0 .. L-1:
    causal (torch.tril), within `window` keys ending at the query (torch.triu
    with diagonal -(window - 1)), and within the query's chunk of `chunk`
    positions (torch.block_diag of all-ones chunks).  Built from library
    routines, not from the oracle's formula."""
    full = torch.ones(L, L, dtype=torch.bool)
    m = torch.tril(full)
    if window:
        m &= torch.triu(full, diagonal=-(window - 1))
    if chunk:
        blocks = [torch.ones(min(chunk, L - i), min(chunk, L - i), dtype=torch.bool) for i in range(0, L, chunk)]
        m &= torch.block_diag(*blocks).bool()
    return m[first_pos:first_pos + n_q].numpy()


@pytest.mark.parametrize("window,chunk", [(1, 0), (5, 0), (16, 0), (23, 0), (0, 7), (0, 16), (9, 16), (40, 0)])
def test_local_attention_prefill_matches_sdpa_with_band_masks(window, chunk):
    q_lens, ctx = [5, 16, 1, 23], [5, 40, 33, 64]
    b = W.random_prefill(93, q_lens, ctx, 4, 2, 64, shared_prefix_blocks=1)
    out, lse = _oracle_prefill_local(b, window, chunk)
    kf, vf = _bf16_to_f64(b.k_pool), _bf16_to_f64(b.v_pool)
    qf = _bf16_to_f64(b.q_prefill)
    qsl = b.query_start_loc.numpy()
    for s, (n, L) in enumerate(zip(q_lens, ctx)):
        mask = _band_mask(n, L, L - n, window, chunk)
        for h in range(4):
            K = _dense_kv(kf, b.block_tables_prefill[s].numpy(), L, h // 2)
            V = _dense_kv(vf, b.block_tables_prefill[s].numpy(), L, h // 2)
            ref = _sdpa(qf[qsl[s]:qsl[s] + n, h], K, V, b.scale, mask)
            got = out[(qsl[s] + np.arange(n)) * 4 + h]
            np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("window,chunk", [(1, 0), (7, 0), (16, 0), (100, 0), (0, 16), (0, 5), (12, 32)])
def test_local_attention_decode_matches_sdpa_with_band_masks(window, chunk):
    lens = [1, 5, 16, 17, 40]
    b = W.random_decode(63, lens, 4, 2, 64, poison=True)
    kd, kc, vc = _oracle_caches(b)
    out, _ = oracle.decode(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode, kc, vc,
                           b.block_tables_decode, b.context_lens_decode, b.scale, window=window, chunk=chunk)
    kf, vf = _bf16_to_f64(b.k_pool), _bf16_to_f64(b.v_pool)
    qf = _bf16_to_f64(b.q_decode)
    for s, L in enumerate(lens):
        mask = _band_mask(1, L, L - 1, window, chunk)
        for h in range(4):
            K = _dense_kv(kf, b.block_tables_decode[s].numpy(), L, h // 2)
            V = _dense_kv(vf, b.block_tables_decode[s].numpy(), L, h // 2)
            ref = _sdpa(qf[s, h][None], K, V, b.scale, mask)[0]
            np.testing.assert_allclose(out[s * 4 + h], ref, atol=1e-12, rtol=0)


def test_local_attention_closed_forms():
    lens = [1, 9, 33]
    b = W.random_decode(64, lens, 4, 2, 64, poison=True)
    kd, kc, vc = _oracle_caches(b)
    args = (kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode, kc, vc, b.block_tables_decode,
            b.context_lens_decode, b.scale)
    full, full_lse = oracle.decode(*args)
    # a window at least as long as every sequence changes nothing
    wide, wide_lse = oracle.decode(*args, window=max(lens))
    assert np.array_equal(wide, full) and np.array_equal(wide_lse, full_lse)
    # a window (or chunk) of one key returns the V of the query's own position
    for kw in ({"window": 1}, {"chunk": 1}):
        one, one_lse = oracle.decode(*args, **kw)
        for s, L in enumerate(lens):
            blk = int(b.block_tables_decode[s, (L - 1) // 16])
            for h in range(4):
                v_last = b.v_pool[blk, h // 2, (L - 1) % 16].to(torch.float64).numpy()
                assert np.array_equal(one[s * 4 + h], v_last)


def _oracle_prefill_local(b: W.PagedBatch, window, chunk):
    kd, kc, vc = _oracle_caches(b)
    return oracle.prefill(kd, b.block_size, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_prefill,
                          b.query_start_loc, kc, vc, b.block_tables_prefill, b.context_lens_prefill,
                          b.scale, b.k_scale, b.v_scale, window=window, chunk=chunk)


# ---------------------------------------------------- shared prefix (cascade)

def _cascade_batch(kv=W.KV_BF16):
    return W.shared_prefix_decode(71, [3, 1, 2], [32, 16, 64], [1, 15, 16, 40, 7, 33], 4, 2, 64, kv_dtype=kv)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_F16])
def test_prefix_matches_bruteforce_sdpa_without_mask(kv):
    b = _cascade_batch(kv)
    c = b.meta["cascade"]
    code = _KV16[kv]
    out, lse = oracle.prefix(code, 16, 2, 4, 64, b.q_decode, c["query_start_loc"], b.k_pool, b.v_pool,
                             c["prefix_tables"], c["prefix_lens"], b.scale)
    kf, vf = _bf16_to_f64(b.k_pool), _bf16_to_f64(b.v_pool)
    qf = _bf16_to_f64(b.q_decode)
    qsl = c["query_start_loc"].numpy()
    for j in range(3):
        P = int(c["prefix_lens"][j])
        rows = np.arange(qsl[j], qsl[j + 1])
        for h in range(4):
            K = _dense_kv(kf, c["prefix_tables"][j].numpy(), P, h // 2)
            V = _dense_kv(vf, c["prefix_tables"][j].numpy(), P, h // 2)
            ref = _sdpa(qf[rows, h], K, V, b.scale)
            np.testing.assert_allclose(out[rows * 4 + h], ref, atol=1e-12, rtol=0)


def test_cascade_prefix_then_suffix_merged_equals_full_decode():
    """Closed form of the cascade: attention over [0, L) is the log-sum-exp
    merge of attention over the shared prefix and over the own suffix."""
    b = _cascade_batch()
    c = b.meta["cascade"]
    full, full_lse = oracle.decode(BF16, 16, 2, 4, 64, b.q_decode, b.k_pool, b.v_pool, b.block_tables_decode,
                                   b.context_lens_decode, b.scale)
    pre, pre_lse = oracle.prefix(BF16, 16, 2, 4, 64, b.q_decode, c["query_start_loc"], b.k_pool, b.v_pool,
                                 c["prefix_tables"], c["prefix_lens"], b.scale)
    suf, suf_lse = oracle.decode(BF16, 16, 2, 4, 64, b.q_decode, b.k_pool, b.v_pool, c["suffix_tables"],
                                 c["suffix_lens"], b.scale)
    for i in range(full.shape[0]):
        o, l = oracle.merge(np.stack([pre[i], suf[i]]), np.array([pre_lse[i], suf_lse[i]]))
        np.testing.assert_allclose(o, full[i], atol=1e-12, rtol=0)
        assert abs(l - full_lse[i]) < 1e-12


def test_prefix_of_zero_tokens_is_empty():
    b = _cascade_batch()
    c = b.meta["cascade"]
    out, lse = oracle.prefix(BF16, 16, 2, 4, 64, b.q_decode, c["query_start_loc"], b.k_pool, b.v_pool,
                             c["prefix_tables"], torch.zeros(3, dtype=torch.int32), b.scale)
    assert np.all(out == 0) and np.all(lse == -np.inf)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8])
def test_copy_blocks_is_a_whole_block_copy(kv):
    g = torch.Generator().manual_seed(9)
    NB, H, D = 12, 3, 64
    if kv == W.KV_BF16:
        k = torch.randn(NB, H, 16, D, generator=g).to(torch.bfloat16)
        v = torch.randn(NB, H, 16, D, generator=g).to(torch.bfloat16)
        kn, vn = k.view(torch.int16).numpy().view(np.uint16), v.view(torch.int16).numpy().view(np.uint16)
        code = BF16
    else:
        kn = torch.randint(0, 256, (NB, H, 16, D), generator=g, dtype=torch.uint8).numpy()
        vn = torch.randint(0, 256, (NB, H, 16, D), generator=g, dtype=torch.uint8).numpy()
        code = FP8
    src, dst = np.array([3, 0, 7], np.int32), np.array([9, 11, 4], np.int32)
    kc, vc = oracle.copy_blocks(code, 16, H, D, src, dst, kn, vn)
    ref_k, ref_v = kn.copy(), vn.copy()
    ref_k[dst], ref_v[dst] = kn[src], vn[src]
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


# ------------------------------------------------------------- golden fixtures

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_codes(name):
    with open(os.path.join(_GOLDEN, name)) as f:
        return {int(a, 16): float(b) for a, b in (line.split() for line in f)}


def test_oracle_matches_its_golden_fixtures():
    """tests/golden/ holds values written by make_golden.py from the oracle;
    any change of the oracle's arithmetic shows here."""
    for name, fn in (("e4m3_codes.txt", oracle.e4m3_decode), ("e5m2_codes.txt", oracle.e5m2_decode),
                     ("f16_specials.txt", oracle.f16_decode)):
        for c, v in _read_codes(name).items():
            got = fn(c)
            assert (math.isnan(v) and math.isnan(got)) or got == v, (name, c, got, v)
    b = W.workload(1, poison=True)
    out, lse = oracle.decode(BF16, 16, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode, b.k_pool, b.v_pool,
                             b.block_tables_decode, b.context_lens_decode, b.scale)
    with open(os.path.join(_GOLDEN, "workload1_decode.txt")) as f:
        rows = [line.split() for line in f if not line.startswith("#")]
    assert len(rows) == out.shape[0]
    # exp / log come from the host's libm: equal to the last few ulps across hosts
    for i, r in enumerate(rows):
        assert abs(float(r[2]) - lse[i]) <= 1e-13 * max(1.0, abs(lse[i]))
        np.testing.assert_allclose(out[i], np.array([float(x) for x in r[3:]]), rtol=1e-13, atol=1e-15)


# ------------------------------------------------ prefix-cache page bookkeeping

def _hit_case(seed=21, NB=64, S=6, MB=10):
    rng = np.random.default_rng(seed)
    tables = np.full((S, MB), -1, np.int32)
    refc = rng.integers(0, 3, NB).astype(np.int32)
    # two trie entries (page lists); sequences 1, 3, 4 hit them
    a = rng.permutation(NB)[:5].astype(np.int32)
    b = np.concatenate([a[:3], rng.permutation(NB)[:2].astype(np.int32)])
    rows = np.array([1, 3, 4], np.int32)
    hits = [a, b, a[:2]]
    start = np.concatenate([[0], np.cumsum([len(h) for h in hits])]).astype(np.int32)
    return tables, refc, rows, start, np.concatenate(hits), hits


def test_bind_blocks_against_numpy_slices_and_bincount():
    tables, refc, rows, start, flat, hits = _hit_case()
    bt, rc, err = oracle.bind_blocks(tables, rows, start, flat, refc)
    want_t = tables.copy()
    for r, h in zip(rows, hits):
        want_t[r, :len(h)] = h
    want_rc = refc + np.bincount(flat, minlength=refc.shape[0]).astype(np.int32)
    assert err == 0 and np.array_equal(bt, want_t) and np.array_equal(rc, want_rc)
    # pages shared by several hits gain one owner per hit
    assert rc[hits[0][0]] == refc[hits[0][0]] + 3


def test_release_blocks_closed_form_and_round_trip():
    tables, refc, rows, start, flat, hits = _hit_case()
    bt, rc, _ = oracle.bind_blocks(tables, rows, start, flat, refc)
    counts = np.array([len(h) for h in hits], np.int32)
    bt2, rc2, free, err = oracle.release_blocks(bt, rows, counts, rc)
    # releasing what was bound restores every count and empties the rows
    assert err == 0 and np.array_equal(rc2, refc) and np.all(bt2[rows] == -1)
    # pages that had no owner before the hit go back to the pool, each once
    assert sorted(free.tolist()) == sorted(p for p in set(flat.tolist()) if refc[p] == 0)


def test_release_returns_a_page_only_when_its_last_owner_leaves():
    NB = 8
    tables = np.array([[3, 5, -1], [3, 6, 7]], np.int32)
    refc = np.zeros(NB, np.int32)
    refc[[3, 5, 6, 7]] = [2, 1, 3, 1]
    bt, rc, free, err = oracle.release_blocks(tables, np.array([0], np.int32), np.array([2], np.int32), refc)
    assert err == 0 and rc.tolist() == [0, 0, 0, 1, 0, 0, 3, 1] and free.tolist() == [5]
    assert bt.tolist() == [[-1, -1, -1], [3, 6, 7]]
    bt, rc, free, err = oracle.release_blocks(bt, np.array([1], np.int32), np.array([3], np.int32), rc)
    assert err == 0 and rc.tolist() == [0, 0, 0, 0, 0, 0, 2, 0] and sorted(free.tolist()) == [3, 7]


def test_bookkeeping_errors_leave_pages_untouched():
    NB = 4
    refc = np.array([0, 1, 0, 0], np.int32)
    tables = np.array([[0, 1, 9]], np.int32)
    bt, rc, free, err = oracle.release_blocks(tables, np.array([0], np.int32), np.array([3], np.int32), refc)
    # page 0 has no owner, page 9 is outside the pool: both errors; page 1 freed
    assert err == 2 and rc.tolist() == [0, 0, 0, 0] and free.tolist() == [1]
    assert bt.tolist() == [[0, -1, 9]]
    bt, rc, err = oracle.bind_blocks(np.full((1, 3), -1, np.int32), np.array([0], np.int32),
                                     np.array([0, 2], np.int32), np.array([2, -1], np.int32), rc)
    assert err == 1 and bt.tolist() == [[2, -1, -1]] and rc.tolist() == [0, 0, 1, 0]
