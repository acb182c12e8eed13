"""Double-precision CPU oracle for the weight-absorbed MLA path.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
library itself never calls it and must not. It shares no code with the CUDA
path: the only thing both sides take from elsewhere is the seeded input
generator module ``mla_inputs``.

Every function works in float64 on exact widenings of the stored inputs and
follows the passage it cites. Where a library primitive serves as a step
(``numpy.matmul``, ``numpy.exp``), it computes exactly what the definition
states; there is no blocking, fusion or reordering beyond that.

Sources (web pages; "P1/P2/P3" below):
  P1 - vllm.cpp ``tests/vt/test_ops_mla_absorb.cpp`` (BatchedMatmul and
       ConcatMlaNopeRope unit tests: the bmm oracle, the strided-view helpers,
       the q concat with a transposed nope operand, the broadcast k_pe head).
  P2 - memra-engine ``tests/mla_gpu_forward.rs`` (absorbed and naive MLA
       attention oracles, latent cache rows ``[c_kv | k_pe]``, the causal
       "queries a suffix of a populated cache" prefill, stepwise decode).
  P3 - vLLM ``tests/kernels/attention/test_mla_cross_layer_kernel_equivalence.py``
       (``concat_and_cache_mla`` into a unified-slot layer view, paged dense
       decode through a block table and ``cache_seqlens``).

Readings where the pages are silent (each is listed in the design notes):
  * softmax is the natural-exponential one with the row maximum subtracted;
    the LSE returned beside a decode is natural-log, ``m + ln(sum e^(s-m))``;
  * causal alignment is bottom-right: query i of a sequence with q_len queries
    and kv_len cached rows sits at position kv_len - q_len + i and sees rows
    0..pos (P2, "queries a suffix of a populated cache");
  * an empty key range gives o = 0 and lse = -inf;
  * a negative slot in a slot mapping marks padding and writes nothing;
  * an fp8 cache holds e4m3 codes; writing one divides the stored value by the
    cache scale in float32 (correctly rounded) and rounds to nearest e4m3, ties
    to even, saturating finite values at +-448 (P3 passes a scale to the cache
    write and descale_q / descale_k to the fp8 decode but prints neither the
    conversion nor the dequantisation); reading one multiplies the code's value
    by descale_k, and the query by descale_q;
  * a ds_mla entry's four float32 scales each cover 128 consecutive latent
    columns (scale g for columns 128g..128g+127), multiplied into the code's
    value; the scales and the bf16 rope values are little-endian (P3 builds the
    entry from tensors' bytes and says only "512B fp8 + 16B f32 scales + 128B
    bf16 rope"); a sparse query attends each listed slot once per listing and
    skips negative entries.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
from numpy.lib.stride_tricks import as_strided


# ---------------------------------------------------------------------------
# Strided views (P1, helpers ``Contig`` and ``View3``: shape and stride in
# ELEMENTS over an existing allocation, plus an element offset)
# ---------------------------------------------------------------------------

def strided_view(flat: np.ndarray, offset: int, shape: Sequence[int],
                 strides: Sequence[int]) -> np.ndarray:
    """Read-only view of ``flat[offset + sum_i idx_i * strides_i]`` with ``shape``."""
    flat = np.asarray(flat)
    assert flat.ndim == 1
    if len(shape) and min(shape) > 0:
        last = offset + sum((n - 1) * s for n, s in zip(shape, strides))
        assert 0 <= offset and last < flat.size, "view reaches outside its storage"
    item = flat.itemsize
    return as_strided(flat[offset:], shape=tuple(shape),
                      strides=tuple(s * item for s in strides), writeable=False)


# ---------------------------------------------------------------------------
# Step 1 and step 5: the absorption bmm's (P1, ``RefBmm``: out[g,m,n] =
# sum_k a[g,m,k] * b[g,k,n] over strided operands)
# ---------------------------------------------------------------------------

def bmm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """out[g,m,n] = sum_k a[g,m,k] b[g,k,n] in float64 (P1, the bmm oracle)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.ndim == 3 and b.ndim == 3 and a.shape[0] == b.shape[0] and a.shape[2] == b.shape[1]
    return np.matmul(a, b)


def absorb_q(q_nope_hbp: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[h,b,l] = sum_p q_nope[h,b,p] W_UK[h,p,l] (P1, the q-side W_UK fold)."""
    return bmm(q_nope_hbp, w_uk)


def v_up(o_lat_hbl: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """out[h,b,v] = sum_l o_lat[h,b,l] W_UV[h,l,v] (P1, the W_UV un-projection)."""
    return bmm(o_lat_hbl, w_uv)


# ---------------------------------------------------------------------------
# Step 2: q concat (P1, ConcatMlaNopeRope: a pure copy, exact; the rope operand
# may carry a single head that every head sees)
# ---------------------------------------------------------------------------

def concat_q(nope: np.ndarray, rope: np.ndarray) -> np.ndarray:
    """out[t,h,:] = [nope[t,h,:] | rope[t,h or 0,:]] as a bit copy of the storage."""
    T, H, L = nope.shape
    assert rope.ndim == 3 and rope.shape[0] == T and rope.shape[1] in (1, H)
    assert nope.dtype == rope.dtype
    R = rope.shape[2]
    out = np.empty((T, H, L + R), dtype=nope.dtype)
    out[:, :, :L] = nope
    out[:, :, L:] = np.broadcast_to(rope, (T, H, R))
    return out


# ---------------------------------------------------------------------------
# Step 3: paged latent cache write (P3, concat_and_cache_mla into a per-layer
# view with an inflated block stride and a storage offset; P2, the cache row
# is [c_kv | k_pe])
# ---------------------------------------------------------------------------

def cache_write(storage: np.ndarray, offset: int, num_blocks: Optional[int], page: int,
                strides: Sequence[int], kv_c: np.ndarray, k_pe: np.ndarray,
                slots: np.ndarray) -> np.ndarray:
    """Return a copy of the flat ``storage`` after writing row i to slot slots[i].

    The cache view is ``[num_blocks, page, L+R]`` at element ``offset`` with
    element strides ``strides``; slot s addresses block s // page, row s % page.
    Elements no slot addresses keep their bits. Negative slots write nothing.
    """
    out = np.array(storage, copy=True)
    T, L = kv_c.shape
    R = k_pe.shape[1]
    s0, s1, s2 = strides
    cols = np.arange(L + R, dtype=np.int64) * s2
    for i in range(T):
        s = int(slots[i])
        if s < 0:
            continue
        blk, row = s // page, s % page
        assert num_blocks is None or blk < num_blocks, "slot outside the cache"
        base = offset + blk * s0 + row * s1
        out[base + cols[:L]] = kv_c[i]
        out[base + cols[L:]] = k_pe[i]
    return out


# ---------------------------------------------------------------------------
# fp8 (e4m3) latent cache (P3: the dense fp8 decode tests store the 576-wide
# rows as float8 e4m3 and pass descale_q / descale_k; concat_and_cache_mla
# takes the cache dtype and a scale)
# ---------------------------------------------------------------------------

def e4m3_value(code) -> np.ndarray:
    """float64 value of e4m3 codes: 1 sign bit, 4 exponent bits with bias 7 and 3
    mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); there are no infinities
    and the two codes with every exponent and mantissa bit set are NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return sign * mag


# every non-negative finite e4m3 value, ascending: codes 0x00 .. 0x7E
_E4M3_POS = e4m3_value(np.arange(0x7F, dtype=np.uint8))


def e4m3_code(x) -> np.ndarray:
    """e4m3 code of float32 values: round to the nearest representable value, ties to
    the even code (the one with an even mantissa), finite values beyond 448 saturate to
    the largest finite code of their sign; signed zeros keep their sign; NaN -> 0x7F."""
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)   # first value >= |x|
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(take_lo & (a <= _E4M3_POS[0x7E]), lo, hi)
    code = np.where(a >= _E4M3_POS[0x7E], 0x7E, code)                  # saturate (and 448 itself)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def cache_write_fp8(storage: np.ndarray, offset: int, num_blocks: Optional[int], page: int,
                    strides: Sequence[int], kv_c: np.ndarray, k_pe: np.ndarray, slots: np.ndarray,
                    scale: float) -> np.ndarray:
    """The cache write into an e4m3 cache (flat uint8 ``storage``): row i becomes the
    codes of float32(x) / float32(scale) for x in [kv_c[i] | k_pe[i]] (the stored
    input values, float32-exact), written through ``cache_write``'s addressing."""
    s32 = np.float32(scale)
    kc = e4m3_code(np.asarray(kv_c, dtype=np.float32) / s32)
    kp = e4m3_code(np.asarray(k_pe, dtype=np.float32) / s32)
    return cache_write(storage, offset, num_blocks, page, strides, kc, kp, slots)


def paged_rows(storage: np.ndarray, offset: int, page: int, strides: Sequence[int],
               entry: int, block_row: np.ndarray, length: int) -> np.ndarray:
    """Rows 0..length-1 of one sequence: row t lives in block block_row[t // page],
    at row t % page of that block (P3, block_table + cache_seqlens)."""
    s0, s1, s2 = strides
    t = np.arange(length, dtype=np.int64)
    blk = np.asarray(block_row, dtype=np.int64)[t // page]
    base = offset + blk * s0 + (t % page) * s1
    idx = base[:, None] + np.arange(entry, dtype=np.int64)[None, :] * s2
    return np.asarray(storage)[idx]


# ---------------------------------------------------------------------------
# Step 4: attention over the latent cache
# ---------------------------------------------------------------------------

def softmax_rows(s: np.ndarray) -> np.ndarray:
    """p[..., t] = e^(s_t - max) / sum e^(s - max) along the last axis."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend_absorbed(q_lat: np.ndarray, q_pe: np.ndarray, c_kv: np.ndarray, k_pe: np.ndarray,
                    scale: float) -> tuple[np.ndarray, np.ndarray]:
    """One query's absorbed attention over rows 0..T-1 (P2, ``mla_attend_absorbed``).

    q_lat [H,L], q_pe [H,R], c_kv [T,L], k_pe [T,R]:
      s[h,t] = scale * (q_lat[h].c_kv[t] + q_pe[h].k_pe[t])
      o_lat[h] = sum_t softmax_t(s[h])[t] c_kv[t];  lse[h] = ln sum_t e^s[h,t]
    Returns (o_lat [H,L], lse [H]); T == 0 gives (0, -inf).
    """
    H, L = q_lat.shape
    T = c_kv.shape[0]
    if T == 0:
        return np.zeros((H, L)), np.full(H, -np.inf)
    s = scale * (q_lat @ c_kv.T + q_pe @ k_pe.T)          # [H, T]
    m = np.max(s, axis=1)
    e = np.exp(s - m[:, None])
    denom = np.sum(e, axis=1)
    o = (e @ c_kv) / denom[:, None]
    return o, m + np.log(denom)


def attend_naive(q_nope: np.ndarray, q_pe: np.ndarray, c_kv: np.ndarray, k_pe: np.ndarray,
                 w_uk: np.ndarray, w_uv: np.ndarray, scale: float) -> np.ndarray:
    """One query's attention in the non-absorbed form (P2, ``mla_attend_naive``).

    Decompress per head k_nope[t,h,p] = sum_l W_UK[h,p,l] c_kv[t,l] and
    v[t,h,j] = sum_l W_UV[h,l,j] c_kv[t,l]; the single k_pe head is shared by all
    heads (P1, ``_concat_k_nope_k_pe``). Then standard softmax attention:
      s[h,t] = scale * (q_nope[h].k_nope[t,h] + q_pe[h].k_pe[t]),
      o[h,j] = sum_t softmax_t(s[h])[t] v[t,h,j].
    q_nope [H,P], q_pe [H,R], c_kv [T,L], k_pe [T,R] -> o [H,V].
    """
    H = q_nope.shape[0]
    k_nope = np.einsum("hpl,tl->thp", w_uk, c_kv)
    v = np.einsum("hlj,tl->thj", w_uv, c_kv)
    s = scale * (np.einsum("hp,thp->ht", q_nope, k_nope) + q_pe @ k_pe.T)
    p = softmax_rows(s)
    return np.einsum("ht,thj->hj", p, v)


def combine(parts: Sequence[tuple[np.ndarray, np.ndarray]]) -> tuple[np.ndarray, np.ndarray]:
    """Merge split-KV partials (o_i [H,L], lse_i [H]) by their log-sum-exp weights:
    lse = ln sum_i e^lse_i and o = sum_i e^(lse_i - lse) o_i. A partial with
    lse_i = -inf (empty chunk) has weight 0; all empty gives (0, -inf)."""
    lses = np.stack([p[1] for p in parts])                # [k, H]
    os_ = np.stack([p[0] for p in parts])                 # [k, H, L]
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe[None, :]), 0.0)
    tot = np.sum(w, axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    o = np.where(finite[:, None],
                 np.einsum("kh,khl->hl", w, os_) / np.where(finite, tot, 1.0)[:, None], 0.0)
    return o, lse


def attend_split(q_lat, q_pe, c_kv, k_pe, scale, bounds: Sequence[int]):
    """Split-KV form: cut rows at ``bounds`` (0 = b_0 <= ... <= b_k = T), attend
    each chunk alone, and merge with :func:`combine`."""
    parts = [attend_absorbed(q_lat, q_pe, c_kv[a:b], k_pe[a:b], scale)
             for a, b in zip(bounds[:-1], bounds[1:])]
    return combine(parts)


def _split_rows(rows: np.ndarray, L: int) -> tuple[np.ndarray, np.ndarray]:
    return rows[:, :L], rows[:, L:]


def decode(q_cat: np.ndarray, storage: np.ndarray, offset: int, page: int,
           strides: Sequence[int], L: int, R: int, block_table: np.ndarray,
           seq_lens: np.ndarray, scale: float,
           batch_ids: Optional[Sequence[int]] = None) -> tuple[np.ndarray, np.ndarray]:
    """Paged decode (P3 dense decode; P2 stepwise decode with t_q = 1).

    q_cat [B,H,L+R] float64; the cache is the flat ``storage`` (float64 values)
    seen as [nb, page, L+R] at ``offset`` with ``strides``. Sequence b attends
    all of its seq_lens[b] rows. Returns o_lat [B,H,L] and lse [B,H] for the
    sequences in ``batch_ids`` (default: all).
    """
    ids = range(q_cat.shape[0]) if batch_ids is None else batch_ids
    os_, ls_ = [], []
    for b in ids:
        rows = paged_rows(storage, offset, page, strides, L + R, block_table[b], int(seq_lens[b]))
        c_kv, kp = _split_rows(rows, L)
        o, lse = attend_absorbed(q_cat[b, :, :L], q_cat[b, :, L:], c_kv, kp, scale)
        os_.append(o)
        ls_.append(lse)
    return np.stack(os_), np.stack(ls_)


def decode_fp8(q_cat: np.ndarray, storage: np.ndarray, offset: int, page: int,
               strides: Sequence[int], L: int, R: int, block_table: np.ndarray,
               seq_lens: np.ndarray, scale: float, descale_q: float, descale_k: float,
               batch_ids: Optional[Sequence[int]] = None) -> tuple[np.ndarray, np.ndarray]:
    """Dense decode over an e4m3 cache (P3, ``flash_mla_with_kvcache_fp8`` with
    descale_q / descale_k): every cache value is its code's value times descale_k,
    the query is q_cat times descale_q, and then it is ``decode``."""
    values = e4m3_value(storage) * float(descale_k)
    return decode(np.asarray(q_cat) * float(descale_q), values, offset, page, strides, L, R,
                  block_table, seq_lens, scale, batch_ids)


# ---------------------------------------------------------------------------
# fp8 ds_mla sparse decode (P3, ``flash_mla_with_kvcache`` with
# ``is_fp8_kvcache`` and ``indices``: a 656-byte entry per token, 512 bytes of
# e4m3 latent codes, four float32 scales, 64 bf16 rope values; top-k int32
# slot indices per query, -1 for padding)
# ---------------------------------------------------------------------------

DS_MLA_ENTRY = 656          # bytes of one cache entry
DS_MLA_L = 512              # latent columns, stored as e4m3 codes in bytes 0..511
DS_MLA_GROUP = 128          # latent columns per float32 scale (four scales, bytes 512..527)
DS_MLA_R = 64               # rope columns, bf16 in bytes 528..655


def ds_mla_values(entries: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The values of [N, 656] ds_mla entries (uint8): c_kv [N, 512] and k_pe [N, 64],
    float64. c_kv[n, i] = value(code[n, i]) * scale[n, i // 128], the scales read as
    little-endian float32 from bytes 512..527; k_pe the little-endian bf16 values of
    bytes 528..655."""
    e = np.ascontiguousarray(entries, dtype=np.uint8).reshape(-1, DS_MLA_ENTRY)
    n_groups = DS_MLA_L // DS_MLA_GROUP
    scales = e[:, DS_MLA_L:DS_MLA_L + 4 * n_groups].copy().view("<f4").astype(np.float64)
    rope_bits = e[:, DS_MLA_L + 4 * n_groups:].copy().view("<u2").astype(np.uint32)
    k_pe = (rope_bits << 16).astype("<u4").view("<f4").astype(np.float64)
    c_kv = e4m3_value(e[:, :DS_MLA_L]) * np.repeat(scales, DS_MLA_GROUP, axis=1)
    return c_kv, k_pe


def decode_sparse_ds_mla(q_cat: np.ndarray, storage: np.ndarray, offset: int, num_blocks: int,
                         page: int, strides: Sequence[int], indices: np.ndarray, scale: float,
                         batch_ids: Optional[Sequence[int]] = None) -> tuple[np.ndarray, np.ndarray]:
    """Sparse decode over an fp8 ds_mla cache.

    The cache is the flat byte ``storage`` seen as [num_blocks, page, 656] at byte
    ``offset`` with byte ``strides``. Query b (q_cat [B, H, 576], float64) attends
    the rows at slots indices[b, j] >= 0, slot = block * page + row, in any order,
    each listed slot once per listing; negative entries are padding. The row's key
    is [c_kv | k_pe] and its value c_kv (``ds_mla_values``); then it is
    ``attend_absorbed``. A slot past the cache raises. Returns o_lat [n, H, 512]
    and lse [n, H] for ``batch_ids`` (default: all); no valid slot gives (0, -inf).
    """
    s0, s1, s2 = strides
    ids = range(q_cat.shape[0]) if batch_ids is None else batch_ids
    storage = np.asarray(storage)
    os_, ls_ = [], []
    for b in ids:
        sl = np.asarray(indices[b], dtype=np.int64)
        sl = sl[sl >= 0]
        if np.any(sl >= num_blocks * page):
            raise ValueError(f"slot {int(sl.max())} past a cache of {num_blocks * page} rows")
        base = offset + (sl // page) * s0 + (sl % page) * s1
        ent = storage[base[:, None] + np.arange(DS_MLA_ENTRY, dtype=np.int64)[None, :] * s2]
        c_kv, kp = ds_mla_values(ent)
        o, lse = attend_absorbed(q_cat[b, :, :DS_MLA_L], q_cat[b, :, DS_MLA_L:], c_kv, kp, scale)
        os_.append(o)
        ls_.append(lse)
    return np.stack(os_), np.stack(ls_)


def prefill(q_cat: np.ndarray, cu_seqlens_q: np.ndarray, kv_lens: np.ndarray,
            storage: np.ndarray, offset: int, page: int, strides: Sequence[int],
            L: int, R: int, block_table: np.ndarray, scale: float,
            rows_wanted: Optional[Sequence[int]] = None) -> tuple[np.ndarray, np.ndarray]:
    """Causal prefill over the paged cache (P2 gate 1: pure prefill t_q == t_kv
    and the chunked shape where the queries are a suffix of the cached rows).

    q_cat [T,H,L+R]; query i of sequence b (global row cu[b] + i) sits at
    position kv_lens[b] - q_len_b + i and attends rows 0..pos. Returns
    o_lat [n,H,L] and lse [n,H] for the global query rows ``rows_wanted``
    (default: every row).
    """
    T = q_cat.shape[0]
    wanted = range(T) if rows_wanted is None else rows_wanted
    seq_of = np.searchsorted(np.asarray(cu_seqlens_q), np.arange(T), side="right") - 1
    cache_rows: dict[int, np.ndarray] = {}
    os_, ls_ = [], []
    for r in wanted:
        b = int(seq_of[r])
        q_len = int(cu_seqlens_q[b + 1] - cu_seqlens_q[b])
        pos = int(kv_lens[b]) - q_len + (r - int(cu_seqlens_q[b]))
        if b not in cache_rows:
            cache_rows[b] = paged_rows(storage, offset, page, strides, L + R,
                                       block_table[b], int(kv_lens[b]))
        rows = cache_rows[b][: max(pos + 1, 0)]
        c_kv, kp = _split_rows(rows, L)
        o, lse = attend_absorbed(q_cat[r, :, :L], q_cat[r, :, L:], c_kv, kp, scale)
        os_.append(o)
        ls_.append(lse)
    return np.stack(os_), np.stack(ls_)


# ---------------------------------------------------------------------------
# The whole path for one decode step (absorb -> concat -> cache write ->
# decode -> v_up), P2 ``gpu_core_parity`` and the stepwise decode gate.
# ---------------------------------------------------------------------------

def decode_step(q_nope: np.ndarray, q_pe: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray,
                new_kv_c: np.ndarray, new_k_pe: np.ndarray, slots: np.ndarray,
                storage: np.ndarray, offset: int, page: int, strides: Sequence[int],
                block_table: np.ndarray, seq_lens: np.ndarray, scale: float,
                batch_ids: Optional[Sequence[int]] = None):
    """One decode step of B sequences, every value float64.

    q_nope [B,H,P], q_pe [B,H,R], new rows [B,L] / [B,R] written at ``slots``
    into the flat cache ``storage`` before attention. Returns
    (out [n,H,V], o_lat [n,H,L], lse [n,H], storage_after) for ``batch_ids``.
    """
    B, H, P = q_nope.shape
    L = w_uk.shape[2]
    R = q_pe.shape[2]
    ids = list(range(B)) if batch_ids is None else list(batch_ids)
    q_lat = absorb_q(np.transpose(q_nope[ids], (1, 0, 2)), w_uk)        # [H,n,L]
    q_cat = concat_q(np.transpose(q_lat, (1, 0, 2)), q_pe[ids])         # [n,H,L+R]
    after = cache_write(storage, offset, None, page, strides, new_kv_c, new_k_pe, slots)
    o_lat, lse = decode(q_cat, after, offset, page, strides, L, R,
                        block_table[ids], seq_lens[ids], scale)
    out = v_up(np.transpose(o_lat, (1, 0, 2)), w_uv)                    # [H,n,V]
    return np.transpose(out, (1, 0, 2)), o_lat, lse, after


def brute_force_attention(q_nope, q_pe, c_kv, k_pe, w_uk, w_uv, scale):
    """Tiny-shape attention by explicit loops and ``math.exp`` (non-absorbed form),
    for pinning the vectorised forms above on a handful of values."""
    H, P = len(q_nope), len(q_nope[0])
    R = len(q_pe[0])
    T, L = len(c_kv), len(c_kv[0])
    V = len(w_uv[0][0])
    out = [[0.0] * V for _ in range(H)]
    for h in range(H):
        scores = []
        for t in range(T):
            acc = 0.0
            for p in range(P):
                k = 0.0
                for l in range(L):
                    k += w_uk[h][p][l] * c_kv[t][l]
                acc += q_nope[h][p] * k
            for r in range(R):
                acc += q_pe[h][r] * k_pe[t][r]
            scores.append(scale * acc)
        top = max(scores)
        ws = [math.exp(x - top) for x in scores]
        tot = sum(ws)
        for j in range(V):
            val = 0.0
            for t in range(T):
                v = 0.0
                for l in range(L):
                    v += w_uv[h][l][j] * c_kv[t][l]
                val += ws[t] / tot * v
            out[h][j] = val
    return out
