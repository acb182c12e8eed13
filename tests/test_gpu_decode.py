"""Step 4 (decode) on the GPU: paged split-KV decode with LSE combine against the
float64 oracle, on the V2-Lite fp32 and V3 bf16 workloads, the shrunk memra
geometries, degenerate lengths, several split counts, a unified-slot cache view
(bit-identical to the contiguous cache) and the full-size variable-length batch
on sampled sequences."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def _device_cache(cache_bits, dtype, layout, n_layers=3, layer=1, fill_seed=999):
    """The cache on the device, contiguous or as one layer of a unified block-major slot."""
    import torch
    nb, page, E = cache_bits.shape
    if layout == "contiguous":
        return to_dev(cache_bits, dtype), None
    other = mi.encode(mi.draw("normal", fill_seed, nb * n_layers * page * E, 0.1), dtype)
    big = to_dev(other, dtype).view(nb, n_layers, page, E)
    big[:, layer].copy_(to_dev(cache_bits, dtype))
    view = big[:, layer]
    assert not view.is_contiguous() and view.stride(0) == n_layers * page * E
    return view, big


def run_decode(mla, q_bits, cache_bits, table, lens, dtype, L, R, scale, num_splits=0,
               layout="contiguous"):
    import torch
    B, H, E = q_bits.shape
    cache, keep = _device_cache(cache_bits, dtype, layout)
    q = to_dev(q_bits, dtype)
    o = poisoned((B, H, L), dtype)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode(o, q, cache, torch.from_numpy(np.ascontiguousarray(table, np.int32)).cuda(),
                   torch.from_numpy(np.asarray(lens, np.int32)).cuda(), L, R, scale, lse_out=lse,
                   num_splits=num_splits)
    mla.mla_device_error()
    del keep
    return o, lse.cpu().numpy().astype(np.float64)


def oracle_decode(q_bits, cache_bits, table, lens, dtype, L, R, scale, ids=None):
    nb, page, E = cache_bits.shape
    storage = mi.decode_f64(cache_bits.reshape(-1), dtype)
    return orc.decode(mi.decode_f64(q_bits, dtype), storage, 0, page, (page * E, E, 1), L, R,
                      np.asarray(table), np.asarray(lens), scale, batch_ids=ids)


# LSE bounds. fp32: 1e-3. bf16 on the tensor-core path: each score's weight is
# P = bf16(bf16(E_0) * bf16(E_1)), three roundings of unit roundoff 2^-8, and the LSE is the
# log of the sum of exactly those P (consistent with the P the output uses), so a row with
# one key can be off by ln(1 + 3 * 2^-8) < 1.2e-2; rows with many keys average far below.
LSE_TOL = {"f32": 1e-3, "bf16": 1.2e-2}


def check_lse(got, want, dtype="f32"):
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin)
    if fin.any():
        assert np.max(np.abs(got[fin] - want[fin])) < LSE_TOL[dtype]


@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_decode_v2_lite_fp32(mla, num_splits):
    w = mi.v2_lite_decode()
    g = w.geom
    q = mi.encode(mi.draw("uniform", 11, w.batch * g.n_head * g.entry), "f32").reshape(w.batch, g.n_head, g.entry)
    o, lse = run_decode(mla, q, w.full_cache(), w.block_table, w.seq_lens, "f32", g.kv_rank, g.d_rope,
                        w.scale, num_splits)
    want, want_lse = oracle_decode(q, w.full_cache(), w.block_table, w.seq_lens, "f32", g.kv_rank,
                                   g.d_rope, w.scale)
    check_close(to_f64(o), want, "f32", f"v2-lite decode splits={num_splits}")
    check_lse(lse, want_lse)


@pytest.mark.parametrize("sharp", [1.0, 30.0])
def test_decode_v3_bf16_and_view_bit_identity(mla, sharp):
    w = mi.v3_decode_small()
    g = w.geom
    q = mi.encode(mi.draw("normal", 1011, w.batch * g.n_head * g.entry, 0.1 * sharp), "bf16").reshape(
        w.batch, g.n_head, g.entry)
    args = (q, w.full_cache(), w.block_table, w.seq_lens, "bf16", g.kv_rank, g.d_rope, w.scale)
    o, lse = run_decode(mla, *args)
    want, want_lse = oracle_decode(*args)
    info = check_close(to_f64(o), want, "bf16", f"v3 decode x{sharp}")
    check_lse(lse, want_lse)
    o_view, lse_view = run_decode(mla, *args, layout="unified")
    assert np.array_equal(to_host_bits(o_view), to_host_bits(o))      # strided view: same bits
    assert np.array_equal(lse_view, lse)
    o2, _ = run_decode(mla, *args)
    assert np.array_equal(to_host_bits(o2), to_host_bits(o))          # run to run: same bits
    del info


@pytest.mark.parametrize("dims", [(4, 24, 8, 32, 64), (3, 12, 4, 20, 48), (4, 32, 0, 32, 64)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_small_geometries_ragged_lengths(mla, dims, dtype):
    H, P, R, V, L = dims
    E = L + R
    lens = [0, 1, 2, 63, 64, 65, 200, 1000, 5]
    page = 16
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 3
    perm = mi.permutation(70, nb)
    table = np.full((len(lens), max(need) + 2), -7, np.int32)      # unused entries are garbage
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("uniform", 71, nb * page * E), dtype).reshape(nb, page, E)
    q = mi.encode(mi.draw("uniform", 72, len(lens) * H * E, 2.0), dtype).reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(P + R)
    for splits in (0, 1, 5, 64):
        o, lse = run_decode(mla, q, cache, table, lens, dtype, L, R, scale, splits)
        want, want_lse = oracle_decode(q, cache, table, lens, dtype, L, R, scale)
        check_close(to_f64(o), want, dtype, f"dims {dims} splits {splits}")
        check_lse(lse, want_lse, dtype)
        got = to_f64(o)
        assert np.all(got[0] == 0) and np.all(lse[0] == -np.inf)      # empty sequence
        row0 = mi.decode_f64(cache[table[1, 0], 0, :L], dtype)
        assert np.array_equal(got[1], np.broadcast_to(row0, (H, L)))  # one row: that row, exactly


@pytest.mark.parametrize("splits", [1, 2, 0])
def test_decode_v3_consecutive_empty_sequences(mla, splits):
    # V3 shapes (the tensor-core path) with runs of zero-length sequences between real ones, so
    # one work unit walks several empty segments back to back: each must still produce o = 0 and
    # lse = -inf, and the sequences after them must be right.
    H, E, L, R = mi.V3.n_head, mi.V3.entry, mi.V3.kv_rank, mi.V3.d_rope
    lens = [0, 0, 70, 0, 0, 0, 129, 0, 64, 0, 0, 1, 0]
    page = 64
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 2
    perm = mi.permutation(81, nb)
    table = np.full((len(lens), max(need) + 1), -3, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("normal", 82, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    q = mi.encode(mi.draw("normal", 83, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(192)
    o, lse = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, splits)
    want, want_lse = oracle_decode(q, cache, table, lens, "bf16", L, R, scale)
    check_close(to_f64(o), want, "bf16", f"consecutive empty sequences, splits {splits}")
    check_lse(lse, want_lse, "bf16")
    got = to_f64(o)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0) and np.all(lse[b] == -np.inf)


def test_decode_v3_segment_boundaries_repeated(mla):
    # A work unit that finishes one sequence and goes on to the next hands the tensor memory
    # from one segment to the next while the previous segment's epilogue may still read its row
    # sums; whether that goes wrong depends on timing, so the same split batch is decoded many
    # times (fresh, differently filled workspaces) and every result is checked.
    import torch
    H, E, L, R = mi.V3.n_head, mi.V3.entry, mi.V3.kv_rank, mi.V3.d_rope
    lens = [0, 0, 70, 0, 0, 0, 129, 0, 64, 0, 0, 1, 0]
    page = 64
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 2
    perm = mi.permutation(81, nb)
    table = np.full((len(lens), max(need) + 1), -3, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache_bits = mi.encode(mi.draw("normal", 82, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    q_bits = mi.encode(mi.draw("normal", 83, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(192)
    want, want_lse = oracle_decode(q_bits, cache_bits, table, lens, "bf16", L, R, scale)
    B = len(lens)
    q, cache = to_dev(q_bits, "bf16"), to_dev(cache_bits, "bf16")
    table_d = torch.from_numpy(table).cuda()
    lens_d = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    for rep in range(24):
        splits = (2, 3, 5)[rep % 3]
        ws = torch.full((mla.mla_decode_workspace_size(B, H, L, splits),), (0x00, 0x41, 0xFF)[rep % 3],
                        dtype=torch.uint8, device="cuda")
        o = poisoned((B, H, L), "bf16")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode(o, q, cache, table_d, lens_d, L, R, scale, lse_out=lse, num_splits=splits, workspace=ws)
        mla.mla_device_error()
        check_close(to_f64(o), want, "bf16", f"repeat {rep}, splits {splits}")
        check_lse(lse.cpu().numpy().astype(np.float64), want_lse, "bf16")


@pytest.mark.parametrize("sharp", [1.0, 30.0])
def test_decode_large_variable_lengths_all_sequences(mla, sharp):
    # The bench configuration: B=64 sequences of 1K..16K rows, auto split count. Every sequence is
    # checked against the oracle, so the ones the schedule cuts across two or more work units are
    # covered along with the shortest and the longest; q x 30 makes the softmax far from uniform,
    # so the per-tile rescaling and the merge of split sequences are exercised, not averaged away.
    w = mi.v3_decode_large(materialize_cache=True)
    g = w.geom
    q = mi.encode(mi.draw("normal", 3011, w.batch * g.n_head * g.entry, 0.1 * sharp), "bf16").reshape(
        w.batch, g.n_head, g.entry)
    o, lse = run_decode(mla, q, w.full_cache(), w.block_table, w.seq_lens, "bf16", g.kv_rank,
                        g.d_rope, w.scale)
    got = to_f64(o)
    assert np.all(np.isfinite(got))
    want, want_lse = oracle_decode(q, w.full_cache(), w.block_table, w.seq_lens, "bf16", g.kv_rank,
                                   g.d_rope, w.scale)
    check_close(got, want, "bf16", f"large decode, q x {sharp}, all sequences")
    for b in (int(np.argmin(w.seq_lens)), int(np.argmax(w.seq_lens))):
        check_close(got[b], want[b], "bf16", f"large decode, q x {sharp}, sequence {b} alone")
    check_lse(lse, want_lse, "bf16")


def _ragged_batch(B, H, E, max_len, page, seed, dtype):
    lens = (mi.randint(seed, B, 0, max_len + 1) * (mi.unit01(seed + 1, B) < 0.85)).astype(np.int64)
    need = [(int(n) + page - 1) // page for n in lens]
    nb = sum(need) + 1
    perm = mi.permutation(seed + 2, nb)
    table = np.zeros((B, max(max(need), 1)), np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("normal", seed + 3, nb * page * E, 0.5), dtype).reshape(nb, page, E)
    q = mi.encode(mi.draw("normal", seed + 4, B * H * E, 0.5), dtype).reshape(B, H, E)
    return [int(x) for x in lens], table, cache, q


@pytest.mark.parametrize("splits", [0, 1100])
def test_decode_schedule_beyond_shared_memory(mla, splits):
    # 2100 sequences (the schedule keeps at most 2048 in shared memory) and, with 1100 splits,
    # more work units than its shared unit array holds: both fall back to the workspace arrays.
    H, L, R, page = 16, 512, 64, 16
    E = L + R
    lens, table, cache, q = _ragged_batch(2100, H, E, 80, page, 301, "bf16")
    scale = 1.0 / math.sqrt(192)
    o, lse = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, splits)
    got = to_f64(o)
    assert np.all(np.isfinite(got))
    ids = [0, 1, 2, 1000, 2047, 2048, 2049, 2099] + [b for b in range(len(lens)) if lens[b] == 0][:2]
    want, want_lse = oracle_decode(q, cache, table, lens, "bf16", L, R, scale, ids=ids)
    check_close(got[ids], want, "bf16", f"2100 sequences, splits {splits}")
    check_lse(lse[ids], want_lse, "bf16")


def test_decode_v3_more_units_than_tiles(mla):
    # The tensor-core path with 1100 work units for a batch of fewer tiles: most units get empty
    # ranges, the unit boundaries live in the workspace, and the result must not change.
    H, E, L, R = mi.V3.n_head, mi.V3.entry, mi.V3.kv_rank, mi.V3.d_rope
    lens, table, cache, q = _ragged_batch(8, H, E, 1500, 64, 311, "bf16")
    scale = 1.0 / math.sqrt(192)
    o1, lse1 = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, 1100)
    o0, lse0 = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, 0)
    want, want_lse = oracle_decode(q, cache, table, lens, "bf16", L, R, scale)
    check_close(to_f64(o1), want, "bf16", "v3 decode, 1100 units")
    check_lse(lse1, want_lse, "bf16")
    check_close(to_f64(o0), want, "bf16", "v3 decode, default units")


@pytest.mark.parametrize("R", [0, 64])
def test_decode_64_heads_tensor_core(mla, R):
    # 64 heads (the memra NoPE geometry with R = 0, or a 64-head slice of V3 with rope) take the
    # tensor-core decode with half of its 128-row tile masked: ragged lengths across page and tile
    # boundaries, an empty sequence, several split counts, against the oracle.
    H, L, page = 64, 512, 64
    E = L + R
    lens = [1, 37, 64, 65, 200, 0, 1000, 129]
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 3
    perm = mi.permutation(160 + R, nb)
    table = np.full((len(lens), max(need) + 1), -5, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("normal", 161 + R, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    q = mi.encode(mi.draw("normal", 162 + R, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(256 if R == 0 else 192)
    want, want_lse = oracle_decode(q, cache, table, lens, "bf16", L, R, scale)
    for splits in (0, 1, 3):
        o, lse = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, splits)
        check_close(to_f64(o), want, "bf16", f"64-head decode R={R}, splits {splits}")
        check_lse(lse, want_lse, "bf16")


@pytest.mark.parametrize("page", [8, 16, 32, 128])
def test_decode_v3_tensor_core_page_sizes(mla, page):
    # The tensor-core path takes pages of 8, 16 and 32 rows (several TMA boxes per 64-key tile,
    # one per page) and pages of 128 rows (tiles starting inside a page), besides 64: ragged
    # lengths across page and tile boundaries, a random block table, two split counts.
    H, E, L, R = mi.V3.n_head, mi.V3.entry, mi.V3.kv_rank, mi.V3.d_rope
    lens = [1, 37, 200, 64, 129, 8, 450]
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 3
    perm = mi.permutation(180 + page, nb)
    table = np.full((len(lens), max(need) + 1), -5, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("normal", 181, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    q = mi.encode(mi.draw("normal", 182, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(192)
    want, want_lse = oracle_decode(q, cache, table, lens, "bf16", L, R, scale)
    for splits in (0, 3):
        o, lse = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale, splits)
        check_close(to_f64(o), want, "bf16", f"page {page}, splits {splits}")
        check_lse(lse, want_lse, "bf16")
