"""Seeded synthetic inputs for the paged-attention workloads.

This module only draws random numbers and lays them out in the cache format;
it holds none of the attention arithmetic, so both the CUDA library's tests
and the fp64 oracle can consume what it makes.  Every workload is seeded with
``1000 + <workload number>``.

Workloads (block size 16 everywhere, q/k/v ~ N(0, 1)):

1. tiny paged decode: 4 sequences, context lengths {1, 7, 16, 33}, 4 q heads /
   2 kv heads, head_dim 64, pool of 64 physical blocks, scale 1/8.
2. Qwen3-8B-shaped decode: 32 sequences, lengths ~ U[512, 4096], 32 q / 8 kv
   heads, head_dim 128, bf16 KV, pool = ceil(1.25 x blocks needed).
3. long/skewed decode: 8 sequences with lengths
   clip(round(lognormal(ln 2048, 1.0)), 128, 32768) plus one of 131072,
   32 q / 8 kv heads, head_dim 128, bf16 KV.
4. FP8 KV decode: 128 sequences, lengths ~ U[1024, 8192], 40 q / 8 kv heads,
   head_dim 128, K/V stored E4M3 with per-tensor fp32 scales amax|src| / 448.
5. mixed continuous-batch step: 16 decode sequences (lengths ~ U[256, 4096])
   plus 4 prefill chunks of 512 new tokens on 2048-token prefixes whose first
   1024 tokens (64 blocks) are the same physical blocks in all four tables;
   new K/V for 16 + 4 x 512 tokens are written through a slot mapping first.

Physical block ids come from a seeded random permutation of the pool, so
tables are non-contiguous.  Table entries past a sequence's last block are -1.
With ``poison=True`` every pool slot that no sequence may read (unused
blocks, the tail of each sequence's last block, slots this step writes) holds
NaN, so any stray read shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

BLOCK_SIZE = 16
KV_BF16 = "bf16"
KV_FP8 = "fp8_e4m3"
KV_FP8_E5M2 = "fp8_e5m2"
KV_F16 = "fp16"
E4M3_MAX = 448.0
E5M2_MAX = 57344.0
#: the largest finite magnitude of each 8-bit cache format
FP8_MAX = {KV_FP8: E4M3_MAX, KV_FP8_E5M2: E5M2_MAX}


@dataclass
class PagedBatch:
    """One step's inputs.  All tensors live on ``device``; bf16 tensors hold the
    values (fp16 ones for an fp16 cache), 8-bit caches are produced from
    ``k_pool``/``v_pool`` by a cache write."""

    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str
    scale: float
    k_scale: float
    v_scale: float
    num_blocks: int
    # pool contents [num_blocks, num_kv_heads, block_size, head_dim] bf16:
    # the cache itself for bf16 KV, the values to be quantised for E4M3 KV
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    # decode part (one query per sequence)
    q_decode: Optional[torch.Tensor] = None          # [S_d, Hq, D] bf16
    block_tables_decode: Optional[torch.Tensor] = None   # int32 [S_d, MB]
    context_lens_decode: Optional[torch.Tensor] = None   # int32 [S_d]
    # prefill part (packed chunks)
    q_prefill: Optional[torch.Tensor] = None         # [Tq, Hq, D] bf16
    query_start_loc: Optional[torch.Tensor] = None   # int32 [S_p + 1]
    block_tables_prefill: Optional[torch.Tensor] = None
    context_lens_prefill: Optional[torch.Tensor] = None
    # K/V written this step and where
    k_new: Optional[torch.Tensor] = None             # [T, Hkv, D] bf16
    v_new: Optional[torch.Tensor] = None
    slot_mapping: Optional[torch.Tensor] = None      # int64 [T]
    # per-kv-head scales of an 8-bit cache (fp32 [Hkv]); None: per-tensor
    k_scales: Optional[torch.Tensor] = None
    v_scales: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def kv_elem_bytes(self) -> int:
        return 2 if self.kv_dtype in (KV_BF16, KV_F16) else 1

    def decode_kv_bytes(self) -> int:
        """Algorithmic KV bytes of the decode part: every valid K and V element
        of every (sequence, kv head) read once."""
        if self.context_lens_decode is None:
            return 0
        tokens = int(self.context_lens_decode.to(torch.int64).sum())
        return tokens * self.num_kv_heads * self.head_dim * 2 * self.kv_elem_bytes

    def max_context_len_decode(self) -> int:
        return int(self.context_lens_decode.max()) if self.context_lens_decode is not None else 0

    def pool_tokens_as_rows(self):
        """The whole pool as cache-write input: ([NB*B, Hkv, D] k, v, int64 slots)."""
        NB, H, B, D = self.k_pool.shape
        k = self.k_pool.permute(0, 2, 1, 3).reshape(NB * B, H, D).contiguous()
        v = self.v_pool.permute(0, 2, 1, 3).reshape(NB * B, H, D).contiguous()
        slots = torch.arange(NB * B, dtype=torch.int64, device=self.k_pool.device)
        return k, v, slots

    def to(self, device) -> "PagedBatch":
        out = PagedBatch(**{k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                            for k, v in self.__dict__.items()})
        return out


def _f32(x: float) -> float:
    """Scales are fp32 arguments of the C ABI: keep them fp32-representable."""
    return float(torch.tensor(x, dtype=torch.float32))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def act_dtype(kv_dtype: str) -> torch.dtype:
    """Element type of q and of new K/V rows: fp16 for an fp16 cache (the cache
    of an fp16 model), bf16 otherwise."""
    return torch.float16 if kv_dtype == KV_F16 else torch.bfloat16


def _randn(shape, g, device, dtype=torch.bfloat16) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def _pool_size(blocks_needed: int) -> int:
    return int(math.ceil(1.25 * blocks_needed))


def _tables(lens, perm, block_size, max_blocks=None):
    """Consecutive chunks of a permutation as block tables (int32, -1 padded)."""
    nblk = [(int(L) + block_size - 1) // block_size for L in lens]
    MB = max_blocks if max_blocks is not None else max(max(nblk), 1)
    t = torch.full((len(lens), MB), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(nblk):
        t[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
    return t, off


def _last_token_slots(tables, lens, block_size):
    slots = []
    for s, L in enumerate(lens):
        L = int(L)
        pos = L - 1
        slots.append(int(tables[s, pos // block_size]) * block_size + pos % block_size)
    return torch.tensor(slots, dtype=torch.int64)


def _readable_mask(num_blocks, block_size, tables_and_lens):
    """bool [NB, B]: slots some sequence reads (token position < its length)."""
    m = torch.zeros(num_blocks, block_size, dtype=torch.bool)
    for tables, lens in tables_and_lens:
        for s in range(tables.shape[0]):
            L = int(lens[s])
            nb = (L + block_size - 1) // block_size
            for j in range(nb):
                blk = int(tables[s, j])
                n_valid = min(block_size, L - j * block_size)
                m[blk, :n_valid] = True
    return m


def _fill_pool(b: PagedBatch, g, device, poison: bool, readable: torch.Tensor,
               written: Optional[torch.Tensor], per_head_scales: bool = False):
    shape = (b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
    b.k_pool = _randn(shape, g, device, act_dtype(b.kv_dtype))
    b.v_pool = _randn(shape, g, device, act_dtype(b.kv_dtype))
    if per_head_scales:
        # heads of different magnitudes (x 2^(h - Hkv/2)), each quantised with
        # its own scale amax(head) / the format's max
        f = torch.pow(2.0, torch.arange(b.num_kv_heads, dtype=torch.float32, device=device) - b.num_kv_heads // 2)
        b.k_pool = (b.k_pool.float() * f[None, :, None, None]).to(b.k_pool.dtype)
        b.v_pool = (b.v_pool.float() * f.flip(0)[None, :, None, None]).to(b.v_pool.dtype)
        mx = FP8_MAX[b.kv_dtype]
        b.k_scales = (b.k_pool.float().abs().amax(dim=(0, 2, 3)) / mx).to(torch.float32).contiguous()
        b.v_scales = (b.v_pool.float().abs().amax(dim=(0, 2, 3)) / mx).to(torch.float32).contiguous()
    if b.kv_dtype in FP8_MAX:
        # per-tensor scales from the source values (amax / the format's max)
        ka = float(b.k_pool.float().abs().max())
        va = float(b.v_pool.float().abs().max())
        if b.k_new is not None and b.meta.get("k_new_independent"):
            ka = max(ka, float(b.k_new.float().abs().max()))
            va = max(va, float(b.v_new.float().abs().max()))
        b.k_scale = _f32(ka / FP8_MAX[b.kv_dtype])
        b.v_scale = _f32(va / FP8_MAX[b.kv_dtype])
    if poison:
        bad = ~readable
        if written is not None:
            bad = bad.clone()
            wb = written // b.block_size
            wo = written % b.block_size
            bad[wb, wo] = True
        bad = bad.to(device)[:, None, :, None].expand(shape)
        nan = torch.tensor(float("nan"), dtype=b.k_pool.dtype, device=device)
        b.k_pool = torch.where(bad, nan, b.k_pool)
        b.v_pool = torch.where(bad, nan, b.v_pool)


def _decode_batch(name, seed, lens, Hq, Hkv, D, kv_dtype, scale, device, poison,
                  num_blocks=None, per_head_scales=False) -> PagedBatch:
    g_cpu = _gen(seed, "cpu")
    lens = torch.as_tensor(lens, dtype=torch.int32)
    needed = int(sum((int(L) + BLOCK_SIZE - 1) // BLOCK_SIZE for L in lens))
    NB = num_blocks if num_blocks is not None else _pool_size(needed)
    perm = torch.randperm(NB, generator=g_cpu)
    tables, _ = _tables(lens, perm, BLOCK_SIZE)
    S = len(lens)
    b = PagedBatch(name=name, block_size=BLOCK_SIZE, num_q_heads=Hq, num_kv_heads=Hkv,
                   head_dim=D, kv_dtype=kv_dtype, scale=_f32(scale), k_scale=1.0, v_scale=1.0,
                   num_blocks=NB, k_pool=None, v_pool=None)
    g = _gen(seed + 7, device)
    b.q_decode = _randn((S, Hq, D), g, device, act_dtype(kv_dtype))
    readable = _readable_mask(NB, BLOCK_SIZE, [(tables, lens)])
    _fill_pool(b, g, device, poison, readable, None, per_head_scales)
    b.block_tables_decode = tables.to(device)
    b.context_lens_decode = lens.to(device)
    # this step's new token of every sequence is its last one (position L - 1);
    # its K/V are the pool's values there, so writing them is idempotent
    slots = _last_token_slots(tables, lens, BLOCK_SIZE)
    NBv = b.k_pool
    blk, off = slots // BLOCK_SIZE, slots % BLOCK_SIZE
    b.k_new = NBv[blk.to(device), :, off.to(device), :].contiguous()
    b.v_new = b.v_pool[blk.to(device), :, off.to(device), :].contiguous()
    b.slot_mapping = slots.to(device)
    return b


#: the name each workload carries (and the bench reports)
WORKLOAD_NAMES = {
    1: "tiny paged decode: 4 seqs, lens {1,7,16,33}, 4q/2kv heads, D=64",
    2: "Qwen3-8B-shaped decode: 32 seqs, lens U[512,4096], 32q/8kv, D=128, bf16 KV",
    3: "long/skewed decode: 8 lognormal seqs in [128,32768] + 1 x 131072, 32q/8kv, D=128, bf16 KV",
    4: "FP8 KV decode: 128 seqs, lens U[1024,8192], 40q/8kv, D=128, E4M3 KV",
    5: "mixed continuous-batch step: 16 decode (U[256,4096]) + 4 x 512-token prefill chunks on 2048-token "
       "prefixes (1024 shared), 32q/8kv, D=128, bf16",
}


def workload(n: int, device="cpu", poison: bool = False, fp8_format: str = KV_FP8,
             fp16: bool = False, per_head_scales: bool = False, fp8_cache: bool = False) -> PagedBatch:
    """Build workload ``n`` (1..5) on ``device``.  ``fp8_format`` picks the
    8-bit cache format of workload 4 (E4M3, or E5M2 for the same shapes);
    ``fp16`` turns the bf16 workloads (1, 2, 3, 5) into fp16 ones: fp16 cache,
    q and new rows, from the same random draws; ``per_head_scales`` gives
    workload 4's kv heads different magnitudes and one scale each;
    ``fp8_cache`` gives workload 5 an 8-bit cache of format ``fp8_format``
    (the same draws, quantised with per-tensor amax / format-max scales)."""
    seed = 1000 + n
    kv16 = KV_F16 if fp16 else KV_BF16

    def name(i):
        return WORKLOAD_NAMES[i].replace("bf16", "fp16") if fp16 else WORKLOAD_NAMES[i]

    if n == 1:
        return _decode_batch(name(1) + (", fp16" if fp16 else ""),
                             seed, [1, 7, 16, 33], 4, 2, 64, kv16, 1.0 / 8.0, device, poison,
                             num_blocks=64)
    if n == 2:
        g = _gen(seed, "cpu")
        lens = torch.randint(512, 4096 + 1, (32,), generator=g)
        return _decode_batch(name(2),
                             seed, lens.tolist(), 32, 8, 128, kv16, 1.0 / math.sqrt(128),
                             device, poison)
    if n == 3:
        g = _gen(seed, "cpu")
        ln = torch.empty(8, dtype=torch.float64).log_normal_(math.log(2048.0), 1.0, generator=g)
        lens = [int(min(max(round(float(x)), 128), 32768)) for x in ln] + [131072]
        return _decode_batch(name(3),
                             seed, lens, 32, 8, 128, kv16, 1.0 / math.sqrt(128), device, poison)
    if n == 4:
        if fp16:
            raise ValueError("workload 4 is the 8-bit cache workload")
        g = _gen(seed, "cpu")
        lens = torch.randint(1024, 8192 + 1, (128,), generator=g)
        nm = WORKLOAD_NAMES[4] if fp8_format == KV_FP8 else WORKLOAD_NAMES[4].replace("E4M3", "E5M2")
        if per_head_scales:
            nm += ", per-head scales"
        return _decode_batch(nm,
                             seed, lens.tolist(), 40, 8, 128, fp8_format, 1.0 / math.sqrt(128),
                             device, poison, per_head_scales=per_head_scales)
    if n == 5:
        if fp8_cache:
            nm = WORKLOAD_NAMES[5].replace("bf16", "E4M3 KV" if fp8_format == KV_FP8 else "E5M2 KV")
            return _mixed_batch(seed, device, poison, fp8_format, nm)
        return _mixed_batch(seed, device, poison, kv16, name(5))
    raise ValueError(f"unknown workload {n}")


def _mixed_batch(seed, device, poison, kv_dtype=KV_BF16, name=WORKLOAD_NAMES[5]) -> PagedBatch:
    return mixed_batch(seed, device, poison, kv_dtype, name=name)


def mixed_batch(seed, device="cpu", poison: bool = False, kv_dtype=KV_BF16, name="mixed continuous-batch step",
                n_dec: int = 16, dec_range=(256, 4096), n_pf: int = 4, prefix: int = 2048, chunk: int = 512,
                shared: int = 1024) -> PagedBatch:
    """One continuous-batch step: n_dec decode sequences with context
    lengths U[dec_range], and n_pf prefill chunks of `chunk` new tokens on
    `prefix`-token prefixes whose first `shared` tokens sit in the same
    physical blocks for every chunk (a prefix-cache hit); 32 q / 8 kv heads,
    head_dim 128.  With the defaults this is workload 5."""
    Hq, Hkv, D, B = 32, 8, 128, BLOCK_SIZE
    g_cpu = _gen(seed, "cpu")
    dec_lens = torch.randint(dec_range[0], dec_range[1] + 1, (n_dec,), generator=g_cpu).to(torch.int32)
    pf_len = prefix + chunk
    shared_blocks = shared // B
    own_blocks = (pf_len - shared + B - 1) // B  # the last one partly filled unless pf_len is a block multiple
    dec_nblk = [(int(L) + B - 1) // B for L in dec_lens]
    needed = sum(dec_nblk) + shared_blocks + n_pf * own_blocks
    NB = _pool_size(needed)
    perm = torch.randperm(NB, generator=g_cpu)
    dec_tables, used = _tables(dec_lens, perm, B)
    shared_ids = perm[used:used + shared_blocks].to(torch.int32)
    used += shared_blocks
    pf_tables = torch.full((n_pf, shared_blocks + own_blocks), -1, dtype=torch.int32)
    for s in range(n_pf):
        pf_tables[s, :shared_blocks] = shared_ids
        pf_tables[s, shared_blocks:] = perm[used:used + own_blocks].to(torch.int32)
        used += own_blocks
    pf_lens = torch.full((n_pf,), pf_len, dtype=torch.int32)
    qsl = torch.arange(0, (n_pf + 1) * chunk, chunk, dtype=torch.int32)

    # slots written this step: each decode sequence's last token, then every
    # prefill chunk's 512 tokens (positions 2048..2559) -- all in own blocks
    dec_slots = _last_token_slots(dec_tables, dec_lens, B)
    pf_slots = []
    for s in range(n_pf):
        for pos in range(prefix, pf_len):
            pf_slots.append(int(pf_tables[s, pos // B]) * B + pos % B)
    slots = torch.cat([dec_slots, torch.tensor(pf_slots, dtype=torch.int64)])
    T = int(slots.shape[0])

    b = PagedBatch(name=name,
                   block_size=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, kv_dtype=kv_dtype,
                   scale=_f32(1.0 / math.sqrt(D)), k_scale=1.0, v_scale=1.0, num_blocks=NB,
                   k_pool=None, v_pool=None)
    g = _gen(seed + 7, device)
    act = act_dtype(kv_dtype)
    b.q_decode = _randn((n_dec, Hq, D), g, device, act)
    b.q_prefill = _randn((n_pf * chunk, Hq, D), g, device, act)
    b.k_new = _randn((T, Hkv, D), g, device, act)
    b.v_new = _randn((T, Hkv, D), g, device, act)
    b.meta["k_new_independent"] = True
    readable = _readable_mask(NB, B, [(dec_tables, dec_lens), (pf_tables, pf_lens)])
    _fill_pool(b, g, device, poison, readable, slots)
    b.block_tables_decode = dec_tables.to(device)
    b.context_lens_decode = dec_lens.to(device)
    b.block_tables_prefill = pf_tables.to(device)
    b.context_lens_prefill = pf_lens.to(device)
    b.query_start_loc = qsl.to(device)
    b.slot_mapping = slots.to(device)
    b.meta.update(shared_block_ids=shared_ids.tolist(), prefix=prefix, chunk=chunk)
    return b


def random_decode(seed: int, lens, Hq, Hkv, D, kv_dtype=KV_BF16, scale=None, device="cpu",
                  poison=True, num_blocks=None, per_head_scales=False) -> PagedBatch:
    """Small randomized decode case for property tests (same recipe as above)."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return _decode_batch(f"random decode seed {seed}", seed, lens, Hq, Hkv, D, kv_dtype, scale,
                         device, poison, num_blocks=num_blocks, per_head_scales=per_head_scales)


def random_prefill(seed: int, q_lens, ctx_lens, Hq, Hkv, D, kv_dtype=KV_BF16, scale=None,
                   device="cpu", poison=True, shared_prefix_blocks: int = 0,
                   per_head_scales: bool = False) -> PagedBatch:
    """Small randomized chunked-prefill case: sequence s has ctx_lens[s] cached
    tokens of which the last q_lens[s] are its chunk's queries.  Optionally the
    first ``shared_prefix_blocks`` blocks are the same physical blocks in every
    table (a prefix-cache hit)."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    B = BLOCK_SIZE
    g_cpu = _gen(seed, "cpu")
    S = len(ctx_lens)
    nblk = [(int(L) + B - 1) // B for L in ctx_lens]
    sh = shared_prefix_blocks
    needed = sum(n - sh for n in nblk) + sh
    NB = _pool_size(needed) + 2
    perm = torch.randperm(NB, generator=g_cpu)
    MB = max(nblk)
    tables = torch.full((S, MB), -1, dtype=torch.int32)
    used = sh
    for s in range(S):
        tables[s, :sh] = perm[:sh].to(torch.int32)
        n_own = nblk[s] - sh
        tables[s, sh:nblk[s]] = perm[used:used + n_own].to(torch.int32)
        used += n_own
    lens = torch.tensor(ctx_lens, dtype=torch.int32)
    qsl = torch.zeros(S + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    b = PagedBatch(name=f"random prefill seed {seed}", block_size=B, num_q_heads=Hq,
                   num_kv_heads=Hkv, head_dim=D, kv_dtype=kv_dtype, scale=_f32(scale), k_scale=1.0,
                   v_scale=1.0, num_blocks=NB, k_pool=None, v_pool=None)
    g = _gen(seed + 7, device)
    b.q_prefill = _randn((int(qsl[-1]), Hq, D), g, device, act_dtype(kv_dtype))
    readable = _readable_mask(NB, B, [(tables, lens)])
    _fill_pool(b, g, device, poison, readable, None, per_head_scales)
    b.block_tables_prefill = tables.to(device)
    b.context_lens_prefill = lens.to(device)
    b.query_start_loc = qsl.to(device)
    return b


def shared_prefix_decode(seed: int, group_sizes, prefix_lens, suffix_lens, Hq, Hkv, D, kv_dtype=KV_BF16,
                         scale=None, device="cpu", poison=True) -> PagedBatch:
    """Decode batch whose sequences come in groups sharing a prefix (a
    prefix-cache hit binds every sequence of group j to the same first
    prefix_lens[j] / 16 physical blocks; prefixes are whole blocks).  Sequence
    i of the batch (groups in order) has prefix_lens[j] + suffix_lens[i]
    tokens.  Besides the usual decode fields, ``meta["cascade"]`` holds the
    split a cascade needs: per group its query rows (query_start_loc over the
    batch's sequences), prefix block table and length; per sequence its
    suffix block table (its own blocks) and length."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    B = BLOCK_SIZE
    assert all(p % B == 0 for p in prefix_lens), "shared prefixes are whole blocks"
    S = sum(group_sizes)
    assert len(suffix_lens) == S
    g_cpu = _gen(seed, "cpu")
    pre_blocks = [p // B for p in prefix_lens]
    suf_blocks = [(int(x) + B - 1) // B for x in suffix_lens]
    needed = sum(pre_blocks) + sum(suf_blocks)
    NB = _pool_size(needed) + 2
    perm = torch.randperm(NB, generator=g_cpu).to(torch.int32)
    used = 0
    pre_ids = []
    for nbp in pre_blocks:
        pre_ids.append(perm[used:used + nbp])
        used += nbp
    MBp = max(max(pre_blocks), 1)
    MBs = max(max(suf_blocks), 1)
    prefix_tables = torch.full((len(group_sizes), MBp), -1, dtype=torch.int32)
    for j, ids in enumerate(pre_ids):
        prefix_tables[j, :len(ids)] = ids
    tables = torch.full((S, MBp + MBs), -1, dtype=torch.int32)
    suffix_tables = torch.full((S, MBs), -1, dtype=torch.int32)
    lens = torch.zeros(S, dtype=torch.int32)
    qsl = torch.zeros(len(group_sizes) + 1, dtype=torch.int32)
    i = 0
    for j, n in enumerate(group_sizes):
        for _ in range(n):
            own = perm[used:used + suf_blocks[i]]
            used += suf_blocks[i]
            tables[i, :pre_blocks[j]] = pre_ids[j]
            tables[i, pre_blocks[j]:pre_blocks[j] + suf_blocks[i]] = own
            suffix_tables[i, :suf_blocks[i]] = own
            lens[i] = prefix_lens[j] + int(suffix_lens[i])
            i += 1
        qsl[j + 1] = qsl[j] + n
    b = PagedBatch(name=f"shared-prefix decode seed {seed}", block_size=B, num_q_heads=Hq, num_kv_heads=Hkv,
                   head_dim=D, kv_dtype=kv_dtype, scale=_f32(scale), k_scale=1.0, v_scale=1.0, num_blocks=NB,
                   k_pool=None, v_pool=None)
    g = _gen(seed + 7, device)
    b.q_decode = _randn((S, Hq, D), g, device, act_dtype(kv_dtype))
    readable = _readable_mask(NB, B, [(tables, lens)])
    _fill_pool(b, g, device, poison, readable, None)
    b.block_tables_decode = tables.to(device)
    b.context_lens_decode = lens.to(device)
    b.meta["cascade"] = dict(query_start_loc=qsl.to(device), prefix_tables=prefix_tables.to(device),
                             prefix_lens=torch.tensor(prefix_lens, dtype=torch.int32, device=device),
                             suffix_tables=suffix_tables.to(device),
                             suffix_lens=torch.tensor([int(x) for x in suffix_lens], dtype=torch.int32,
                                                      device=device))
    return b
