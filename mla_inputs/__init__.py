"""Seeded synthetic inputs for the weight-absorbed MLA path.

This module only draws numbers. It holds none of the attention, matmul or
copy arithmetic of the method: the oracle (``oracle/``) and the CUDA binding
both take their inputs from here and from nowhere else.

Random source
-------------
The uniform generator is the 32-bit linear congruential generator of the
vllm.cpp MLA absorption test page (``test_ops_mla_absorb.cpp``, helper
``RandF32``): the state advances ``s <- s*1664525 + 1013904223 (mod 2^32)``
*before* each draw, and a draw is ``(s >> 8) / 2^24 * 2 - 1`` in [-1, 1).

Because an LCG step is affine, ``k`` steps compose into one affine map
``s -> A_k s + C_k (mod 2^32)``; ``lcg_states`` uses that to produce any
sub-range of a stream without walking it from the start, so a test can
regenerate the rows of one sampled sequence of a large cache cheaply.

Normal draws use Box-Muller over consecutive pairs of uniforms (draw ``2i``
and ``2i+1`` give normal ``i``; only the cosine branch is used).

bf16 inputs are fp32 draws rounded to nearest-even and kept as their raw
16-bit patterns (``uint16``); consumers widen them exactly.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

_A = 1664525
_C = 1013904223
_M32 = (1 << 32) - 1

# Per-tensor seeds; a configuration adds 1000 * its index.
SEED_Q_NOPE = 11
SEED_Q_PE = 22
SEED_C_KV = 33
SEED_K_PE = 44
SEED_W_UK = 55
SEED_W_UV = 66
SEED_TABLES = 77
SEED_LENGTHS = 88


def _jump(k: int) -> tuple[int, int]:
    """Affine coefficients (A_k, C_k) of k LCG steps, by square-and-multiply."""
    a_tot, c_tot = 1, 0          # identity map
    a_pow, c_pow = _A, _C        # one step
    while k:
        if k & 1:
            # apply (a_pow, c_pow) after (a_tot, c_tot)
            a_tot, c_tot = (a_pow * a_tot) & _M32, (a_pow * c_tot + c_pow) & _M32
        a_pow, c_pow = (a_pow * a_pow) & _M32, (a_pow * c_pow + c_pow) & _M32
        k >>= 1
    return a_tot, c_tot


_CHUNK = 1 << 22


def lcg_states(seed: int, start: int, count: int) -> np.ndarray:
    """States s_{start+1} .. s_{start+count} (uint32) of the stream seeded with ``seed``.

    s_0 = seed; draw i (0-based) uses s_{i+1}. uint32 array arithmetic wraps
    modulo 2^32, which is exactly the LCG's modulus.
    """
    out = np.empty(count, dtype=np.uint32)
    if count == 0:
        return out
    m = min(count, _CHUNK)
    # states of the first chunk by doubling: fill [0,1), then [1,2), [2,4) ...
    first = out[:m]
    a1, c1 = _jump(start + 1)
    first[0] = (a1 * (seed & _M32) + c1) & _M32
    filled = 1
    with np.errstate(over="ignore"):
        while filled < m:
            n = min(filled, m - filled)
            ak, ck = _jump(filled)
            np.multiply(first[:n], np.uint32(ak), out=first[filled:filled + n])
            first[filled:filled + n] += np.uint32(ck)
            filled += n
        pos = m
        while pos < count:
            n = min(m, count - pos)
            ak, ck = _jump(pos)
            np.multiply(first[:n], np.uint32(ak), out=out[pos:pos + n])
            out[pos:pos + n] += np.uint32(ck)
            pos += n
    return out


def _u24(seed: int, count: int, start: int) -> np.ndarray:
    """The 24-bit integer part (s >> 8) of each draw, as float32 (exact)."""
    return (lcg_states(seed, start, count) >> np.uint32(8)).astype(np.int32).astype(np.float32)


def uniform(seed: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` draws in [-1, 1) as float32 (exact: every value is k/2^23 - 1)."""
    v = _u24(seed, count, start)
    v *= np.float32(2.0 / (1 << 24))
    v -= np.float32(1.0)
    return v


def unit01(seed: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` draws in [0, 1) as float64 (the same stream mapped to [0,1))."""
    return _u24(seed, count, start).astype(np.float64) / float(1 << 24)


def normal(seed: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` N(0,1) draws (float32) by Box-Muller over uniform pairs."""
    u = _u24(seed, 2 * count, 2 * start).reshape(count, 2)
    u1 = np.float32(1 << 24) - u[:, 0]        # (1 - u1) * 2^24, in [1, 2^24]
    u1 *= np.float32(1.0 / (1 << 24))        # (0, 1]
    r = np.log(u1)
    r *= np.float32(-2.0)
    np.sqrt(r, out=r)
    t = u[:, 1] * np.float32(2.0 * math.pi / (1 << 24))
    np.cos(t, out=t)
    r *= t
    return r


def permutation(seed: int, n: int) -> np.ndarray:
    """A Fisher-Yates permutation of range(n) driven by the LCG (int64)."""
    p = np.arange(n, dtype=np.int64)
    u = unit01(seed, max(n - 1, 0))
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = int(u[k] * (i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def randint(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform on the closed range [lo, hi] (int64)."""
    u = unit01(seed, count)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = ((b[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 patterns to float32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def draw(kind: str, seed: int, count: int, scale: float = 1.0, start: int = 0) -> np.ndarray:
    """float32 draws of a named distribution: 'uniform' in [-1,1) or 'normal'."""
    if kind == "uniform":
        v = uniform(seed, count, start)
    elif kind == "normal":
        v = normal(seed, count, start)
    else:
        raise ValueError(kind)
    if scale != 1.0:
        v = (v.astype(np.float64) * scale).astype(np.float32)
    return v


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values in the run dtype's storage: float32 itself or bf16 bits."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(dtype)


def decode_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a stored array (float32, or bf16 bits)."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Workload geometry (the five workloads of the weight-absorbed MLA path)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Geometry:
    """Head geometry: n_head, d_nope (P), d_rope (R), d_v (V), kv_lora_rank (L)."""
    n_head: int
    d_nope: int
    d_rope: int
    d_v: int
    kv_rank: int

    @property
    def entry(self) -> int:
        return self.kv_rank + self.d_rope


V2_LITE = Geometry(16, 128, 64, 128, 512)
V3 = Geometry(128, 128, 64, 128, 512)
NOPE_64 = Geometry(64, 256, 0, 256, 512)


@dataclasses.dataclass
class DecodeWorkload:
    """A decode batch over a paged latent cache, one new token per sequence.

    ``cache`` holds the latent rows in storage dtype, shaped [num_blocks, page, E]
    and contiguous; ``block_table`` is int32 [B, max_blocks]; ``seq_lens`` int32 [B]
    counts the rows each sequence owns *after* this step's row is written.
    """
    name: str
    dtype: str
    geom: Geometry
    page: int
    seq_lens: np.ndarray
    block_table: np.ndarray
    num_blocks: int
    scale: float
    q_nope: np.ndarray          # [B, H, P]
    q_pe: np.ndarray            # [B, H, R]
    w_uk: np.ndarray            # [H, P, L]
    w_uv: np.ndarray            # [H, L, V]
    cache: Optional[np.ndarray]  # [num_blocks, page, E] (None: generate lazily)
    cache_kind: str
    cache_scale: float
    cache_seed: int
    new_kv_c: np.ndarray        # [B, L]   the row this step appends
    new_k_pe: np.ndarray        # [B, R]
    slots: np.ndarray           # int64 [B] slot of the appended row

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    def cache_rows(self, blocks: np.ndarray) -> np.ndarray:
        """Initial cache contents of the listed blocks, [len(blocks), page, E]."""
        if self.cache is not None:
            return self.cache[blocks]
        E, page = self.geom.entry, self.page
        out = np.empty((len(blocks), page, E), dtype=np.uint16 if self.dtype == "bf16" else np.float32)
        for i, blk in enumerate(np.asarray(blocks, dtype=np.int64)):
            v = draw(self.cache_kind, self.cache_seed, page * E, self.cache_scale,
                     start=int(blk) * page * E)
            out[i] = encode(v, self.dtype).reshape(page, E)
        return out

    def full_cache(self) -> np.ndarray:
        if self.cache is None:
            E, page = self.geom.entry, self.page
            v = draw(self.cache_kind, self.cache_seed, self.num_blocks * page * E, self.cache_scale)
            self.cache = encode(v, self.dtype).reshape(self.num_blocks, page, E)
        return self.cache


def _paged_tables(seed: int, seq_lens: np.ndarray, page: int, contiguous: bool,
                  num_blocks: Optional[int] = None) -> tuple[np.ndarray, int]:
    need = [(int(n) + page - 1) // page for n in seq_lens]
    max_blocks = max(max(need), 1)
    total = sum(need)
    nb = num_blocks if num_blocks is not None else max(total, 1)
    order = np.arange(nb, dtype=np.int64) if contiguous else permutation(seed, nb)
    table = np.zeros((len(seq_lens), max_blocks), dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = order[k:k + n]
        k += n
    return table, nb


def decode_workload(geom: Geometry, dtype: str, seq_lens, page: int = 64, *,
                    config_index: int = 0, contiguous_table: bool = False,
                    act_kind: str = "normal", act_scale: float = 0.1,
                    cache_kind: str = "normal", cache_scale: float = 0.1,
                    weight_kind: str = "normal", weight_scale: float = 1.0 / math.sqrt(512),
                    scale: Optional[float] = None, num_blocks: Optional[int] = None,
                    materialize_cache: bool = True, name: str = "decode") -> DecodeWorkload:
    """Build a seeded decode workload (see the module docstring for the recipe)."""
    off = 1000 * config_index
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, H, P, R, V, L = len(seq_lens), geom.n_head, geom.d_nope, geom.d_rope, geom.d_v, geom.kv_rank
    table, nb = _paged_tables(SEED_TABLES + off, seq_lens, page, contiguous_table, num_blocks)
    q_nope = encode(draw(act_kind, SEED_Q_NOPE + off, B * H * P, act_scale), dtype).reshape(B, H, P)
    q_pe = encode(draw(act_kind, SEED_Q_PE + off, B * H * R, act_scale), dtype).reshape(B, H, R)
    w_uk = encode(draw(weight_kind, SEED_W_UK + off, H * P * L, weight_scale), dtype).reshape(H, P, L)
    w_uv = encode(draw(weight_kind, SEED_W_UV + off, H * L * V, weight_scale), dtype).reshape(H, L, V)
    # The appended rows come from streams of their own (seed + 500) so that the
    # initial cache stream is independent of the batch.
    new_kv_c = encode(draw(cache_kind, SEED_C_KV + off + 500, B * L, cache_scale), dtype).reshape(B, L)
    new_k_pe = encode(draw(cache_kind, SEED_K_PE + off + 500, B * R, cache_scale), dtype).reshape(B, R)
    slots = np.empty(B, dtype=np.int64)
    for b in range(B):
        pos = int(seq_lens[b]) - 1          # the appended row is the last one
        slots[b] = -1 if pos < 0 else int(table[b, pos // page]) * page + pos % page
    w = DecodeWorkload(name=name, dtype=dtype, geom=geom, page=page, seq_lens=seq_lens,
                       block_table=table, num_blocks=nb,
                       scale=scale if scale is not None else 1.0 / math.sqrt(P + R),
                       q_nope=q_nope, q_pe=q_pe, w_uk=w_uk, w_uv=w_uv, cache=None,
                       cache_kind=cache_kind, cache_scale=cache_scale, cache_seed=SEED_C_KV + off,
                       new_kv_c=new_kv_c, new_k_pe=new_k_pe, slots=slots)
    if materialize_cache:
        w.full_cache()
    return w


def v2_lite_decode() -> DecodeWorkload:
    """V2-Lite fp32 decode: B=2, context 256, page 64, contiguous table, uniform data."""
    return decode_workload(V2_LITE, "f32", [256, 256], 64, config_index=0, contiguous_table=True,
                           act_kind="uniform", act_scale=1.0, cache_kind="uniform", cache_scale=1.0,
                           weight_kind="uniform", weight_scale=1.0 / math.sqrt(512),
                           scale=1.0 / math.sqrt(192), name="v2lite_f32_decode_b2_ctx256")


def v3_decode_small() -> DecodeWorkload:
    """V3 bf16 decode: B=4, context 4096 each, page 64, table a permutation of 256 blocks."""
    return decode_workload(V3, "bf16", [4096] * 4, 64, config_index=1,
                           scale=1.0 / math.sqrt(192), name="v3_bf16_decode_b4_ctx4096")


def v3_decode_large_lengths(batch: int = 64, lo: int = 1024, hi: int = 16384) -> np.ndarray:
    """Per-sequence context lengths of the large V3 decode, uniform on [lo, hi]."""
    return randint(SEED_LENGTHS + 3000, batch, lo, hi).astype(np.int32)


def v3_decode_large(materialize_cache: bool = True) -> DecodeWorkload:
    """V3 bf16 decode: B=64, lengths U[1024,16384], page 64, random block table."""
    return decode_workload(V3, "bf16", v3_decode_large_lengths(), 64, config_index=3,
                           scale=1.0 / math.sqrt(192), materialize_cache=materialize_cache,
                           name="v3_bf16_decode_b64_ctx1k-16k")


@dataclasses.dataclass
class WriteConcatWorkload:
    """Paged cache write into a unified-slot layer view, plus the q concat."""
    kv_c: np.ndarray        # bf16 bits [T, L]
    k_pe: np.ndarray        # bf16 bits [T, R]
    slots: np.ndarray       # int64 [T]
    num_blocks: int
    page: int
    n_layers: int
    layer: int
    q_nope_storage: np.ndarray  # bf16 bits [N, B, L] (the bmm output layout)
    q_pe: np.ndarray            # bf16 bits [B, N, R]

    @property
    def entry(self) -> int:
        return self.kv_c.shape[1] + self.k_pe.shape[1]


def write_concat_workload(ntok: int = 200, num_blocks: int = 32, page: int = 64,
                          L: int = 512, R: int = 64, n_layers: int = 3, layer: int = 1,
                          q_tokens: int = 64, q_heads: int = 128,
                          config_index: int = 2) -> WriteConcatWorkload:
    off = 1000 * config_index
    kv_c = to_bf16_bits(normal(SEED_C_KV + off, ntok * L)).reshape(ntok, L)
    k_pe = to_bf16_bits(normal(SEED_K_PE + off, ntok * R)).reshape(ntok, R)
    slots = permutation(SEED_TABLES + off, num_blocks * page)[:ntok].copy()
    q_nope = to_bf16_bits(normal(SEED_Q_NOPE + off, q_heads * q_tokens * L)).reshape(q_heads, q_tokens, L)
    q_pe = to_bf16_bits(normal(SEED_Q_PE + off, q_tokens * q_heads * R)).reshape(q_tokens, q_heads, R)
    return WriteConcatWorkload(kv_c, k_pe, slots, num_blocks, page, n_layers, layer, q_nope, q_pe)


@dataclasses.dataclass
class PrefillWorkload:
    """Causal prefill: every sequence's queries are the last q_len of kv_len rows."""
    dtype: str
    geom: Geometry
    page: int
    q_lens: np.ndarray       # int32 [B]
    kv_lens: np.ndarray      # int32 [B]
    block_table: np.ndarray  # int32 [B, max_blocks]
    num_blocks: int
    scale: float
    q_nope: np.ndarray       # [T, H, P]
    q_pe: np.ndarray         # [T, H, R]
    kv_c: np.ndarray         # [sum kv_len, L]  rows of every sequence, in order
    k_pe: np.ndarray         # [sum kv_len, R]
    w_uk: np.ndarray
    w_uv: np.ndarray

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_seqlens_kv(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.kv_lens)]).astype(np.int32)

    def slot_mapping(self) -> np.ndarray:
        """int64 slot of every kv row (in kv_c order)."""
        out = []
        for b, n in enumerate(self.kv_lens):
            t = np.arange(int(n), dtype=np.int64)
            out.append(self.block_table[b, t // self.page].astype(np.int64) * self.page + t % self.page)
        return np.concatenate(out) if out else np.zeros(0, np.int64)


def prefill_workload(geom: Geometry, dtype: str, q_lens, kv_lens, page: int = 64, *,
                     config_index: int = 4, act_kind: str = "normal", act_scale: float = 1.0,
                     weight_scale: float = 1.0 / math.sqrt(512),
                     scale: Optional[float] = None) -> PrefillWorkload:
    off = 1000 * config_index
    q_lens = np.asarray(q_lens, dtype=np.int32)
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    H, P, R, V, L = geom.n_head, geom.d_nope, geom.d_rope, geom.d_v, geom.kv_rank
    T, S = int(q_lens.sum()), int(kv_lens.sum())
    table, nb = _paged_tables(SEED_TABLES + off, kv_lens, page, False)
    return PrefillWorkload(
        dtype=dtype, geom=geom, page=page, q_lens=q_lens, kv_lens=kv_lens, block_table=table,
        num_blocks=nb, scale=scale if scale is not None else 1.0 / math.sqrt(P + R),
        q_nope=encode(draw(act_kind, SEED_Q_NOPE + off, T * H * P, act_scale), dtype).reshape(T, H, P),
        q_pe=encode(draw(act_kind, SEED_Q_PE + off, T * H * R, act_scale), dtype).reshape(T, H, R),
        kv_c=encode(draw(act_kind, SEED_C_KV + off, S * L, act_scale), dtype).reshape(S, L),
        k_pe=encode(draw(act_kind, SEED_K_PE + off, S * R, act_scale), dtype).reshape(S, R),
        w_uk=encode(draw("normal", SEED_W_UK + off, H * P * L, weight_scale), dtype).reshape(H, P, L),
        w_uv=encode(draw("normal", SEED_W_UV + off, H * L * V, weight_scale), dtype).reshape(H, L, V),
    )


def nope_prefill(n_seq: int = 4, seq_len: int = 2048) -> PrefillWorkload:
    """NoPE causal prefill: 64 heads, P=256, R=0, V=256, L=512, n_seq x seq_len."""
    return prefill_workload(NOPE_64, "bf16", [seq_len] * n_seq, [seq_len] * n_seq, 64,
                            config_index=4, scale=1.0 / math.sqrt(256))


# ---------------------------------------------------------------------------- ds_mla sparse decode

SEED_DS_MLA = 99


def ds_mla_entries(seed: int, n: int, unit_scales: bool = False) -> np.ndarray:
    """[n, 656] uint8 cache entries with the ds_mla byte structure, drawn directly (no
    conversion of values): 512 e4m3 codes with a random sign, an exponent field in
    [1, 9] and a random mantissa (about one in 64 a zero code), four little-endian
    float32 scales (1.0, or uniform in [1/128, 1/32)), and 64 little-endian bf16 rope
    values drawn N(0, 1) * 0.1."""
    m = n * 512
    code = (randint(seed, m, 0, 1) << 7) | (randint(seed + 1, m, 1, 9) << 3) | randint(seed + 2, m, 0, 7)
    code = np.where(randint(seed + 3, m, 0, 63) == 0, 0, code).astype(np.uint8).reshape(n, 512)
    if unit_scales:
        sc = np.ones((n, 4), np.float32)
    else:
        sc = (1.0 / 128 + unit01(seed + 4, n * 4) * (1.0 / 32 - 1.0 / 128)).astype(np.float32).reshape(n, 4)
    rope = to_bf16_bits(normal(seed + 5, n * 64) * np.float32(0.1)).reshape(n, 64)
    return np.concatenate([code, sc.astype("<f4").view(np.uint8).reshape(n, 16),
                           rope.astype("<u2").view(np.uint8).reshape(n, 128)], axis=1)


@dataclasses.dataclass
class SparseDecodeWorkload:
    """Sparse top-k decode over a ds_mla cache seen as one layer of a block-major
    multi-layer buffer: ``storage`` is the whole uint8 buffer [num_blocks, n_layers,
    page, 656] (other layers random bytes), the layer's view has byte strides
    (n_layers * page * 656, 656, 1) at byte offset layer * page * 656."""
    q_cat: np.ndarray        # bf16 bits [B, H, 576]
    storage: np.ndarray      # uint8, flat
    indices: np.ndarray      # int32 [B, topk], -1 = padding
    num_blocks: int
    page: int
    n_layers: int
    layer: int
    scale: float

    @property
    def offset(self) -> int:
        return self.layer * self.page * 656

    @property
    def strides(self) -> tuple[int, int, int]:
        return (self.n_layers * self.page * 656, 656, 1)


def sparse_decode_workload(batch: int = 2, heads: int = 128, topk: int = 128, num_blocks: int = 32,
                           page: int = 64, n_layers: int = 3, layer: int = 1, pattern: str = "blocks",
                           unit_scales: bool = True, config_index: int = 7) -> SparseDecodeWorkload:
    """``pattern`` "blocks": query b takes the first topk slots of its own num_blocks // batch
    consecutive blocks, padded with -1 (the pages' layout); "scattered": query b takes a
    random count in [0, topk] of distinct slots drawn from the whole cache in random order,
    with the -1 padding shuffled among them."""
    off = 1000 * config_index
    E = 656
    layer_bytes = ds_mla_entries(SEED_DS_MLA + off, num_blocks * page, unit_scales).reshape(num_blocks, page, E)
    other = randint(SEED_DS_MLA + off + 10, num_blocks * n_layers * page * E, 0, 255).astype(np.uint8)
    storage = other.reshape(num_blocks, n_layers, page, E)
    storage[:, layer] = layer_bytes
    idx = np.full((batch, topk), -1, np.int32)
    if pattern == "blocks":
        per = num_blocks // batch
        for b in range(batch):
            slots = np.arange(b * per * page, (b + 1) * per * page)[:topk]
            idx[b, :slots.size] = slots
    elif pattern == "scattered":
        n = num_blocks * page
        counts = np.minimum(randint(SEED_DS_MLA + off + 20, batch, 0, topk), n)
        starts = randint(SEED_DS_MLA + off + 21, batch, 0, n - 1)
        perm = permutation(SEED_DS_MLA + off + 22, n)
        for b in range(batch):
            slots = perm[(int(starts[b]) + np.arange(int(counts[b]))) % n]    # distinct, scattered
            row = np.concatenate([slots, np.full(topk - slots.size, -1)])
            idx[b] = row[permutation(SEED_DS_MLA + off + 30 + b, topk)]
    else:
        raise ValueError(pattern)
    q = to_bf16_bits(normal(SEED_Q_NOPE + off, batch * heads * 576) * np.float32(0.1)).reshape(batch, heads, 576)
    return SparseDecodeWorkload(q, storage.reshape(-1), idx, num_blocks, page, n_layers, layer, 576 ** -0.5)
