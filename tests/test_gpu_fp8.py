"""The fp8 (e4m3) latent cache on the GPU: the cache write into an e4m3 cache and the
decode over it, against the float64 oracle (``cache_write_fp8``, ``decode_fp8``).

The cache write is checked bit for bit over a whole 3-layer unified-slot buffer
(sentinel bytes everywhere it must not write), including saturating values and
both source dtypes. The decode follows the vLLM page's dense fp8 decode test:
128 heads, 576-wide e4m3 rows, page 64, descale_q and descale_k, read through a
unified-slot layer view bit-identically to a contiguous cache, and within the
path's tolerances of the oracle (bf16 max-abs 2e-2 and relative L2 1e-2; fp32
max-abs 1e-4)."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def _u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


@pytest.mark.parametrize("src", ["bf16", "f32"])
@pytest.mark.parametrize("scale", [1.0, 0.5, 0.37])
def test_fp8_cache_write_unified_view_bit_exact(mla, src, scale):
    import torch
    w = mi.write_concat_workload()
    T, L, R, page, nb, layers, layer = w.kv_c.shape[0], 512, 64, w.page, w.num_blocks, w.n_layers, w.layer
    E = L + R
    # values of several magnitudes, a few far beyond the e4m3 range (they saturate)
    mag = np.where(mi.unit01(7101, T * E) < 0.05, 3000.0, 3.0)
    kv = mi.encode(mi.draw("normal", 7102, T * L) * mag[: T * L], src).reshape(T, L)
    kp = mi.encode(mi.draw("normal", 7103, T * R) * mag[T * L:T * E], src).reshape(T, R)
    slots = w.slots.copy()
    slots[::17] = -1                                            # padding rows write nothing
    storage = mi.permutation(7104, nb * layers * page * E).astype(np.uint8)   # sentinel bytes
    big = _u8(storage)
    view = big.as_strided((nb, page, E), (layers * page * E, E, 1), layer * page * E)
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    mla.mla_cache_write_fp8(view, to_dev(kv, src), to_dev(kp, src), torch.from_numpy(slots).cuda(), sc)
    mla.mla_device_error()
    want = orc.cache_write_fp8(storage, layer * page * E, nb, page, (layers * page * E, E, 1),
                               mi.decode_f64(kv, src), mi.decode_f64(kp, src), slots, scale)
    assert np.array_equal(big.cpu().numpy(), want)


def _fp8_batch(H, L, R, lens, page, seed, descale_k):
    """e4m3 codes of N(0,1)*0.1 / descale_k cache rows (so the dequantised values are ~N(0,1)*0.1)."""
    E = L + R
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 2
    perm = mi.permutation(seed, nb)
    table = np.full((len(lens), max(max(need), 1) + 1), -1, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    vals = mi.draw("normal", seed + 1, nb * page * E, 0.1) / np.float32(descale_k)
    codes = orc.e4m3_code(vals.astype(np.float32)).reshape(nb, page, E)
    return codes, table


@pytest.mark.parametrize("dtype,geom", [("bf16", "v3"), ("f32", "v2lite")])
def test_fp8_decode_matches_oracle_and_view(mla, dtype, geom):
    import torch
    g = mi.V3 if geom == "v3" else mi.V2_LITE
    H, L, R = g.n_head, g.kv_rank, g.d_rope
    E = L + R
    lens = [1, 63, 64, 65, 700, 2000, 0, 129]
    page = 64
    dq, dk = 0.5, 2.0
    codes, table = _fp8_batch(H, L, R, lens, page, 7201 + H, dk)
    q_bits = mi.encode(mi.draw("normal", 7210 + H, len(lens) * H * E, 0.2), dtype).reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(E)
    want, want_lse = orc.decode_fp8(mi.decode_f64(q_bits, dtype), codes.reshape(-1), 0, page, (page * E, E, 1),
                                    L, R, table, np.array(lens), scale, dq, dk)
    q = to_dev(q_bits, dtype)
    tab = torch.from_numpy(table).cuda()
    lens_d = torch.from_numpy(np.array(lens, np.int32)).cuda()
    dqt = torch.tensor([dq], dtype=torch.float32, device="cuda")
    dkt = torch.tensor([dk], dtype=torch.float32, device="cuda")

    def run(cache, splits=0):
        o = poisoned((len(lens), H, L), dtype)
        lse = torch.full((len(lens), H), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_fp8(o, q, cache, tab, lens_d, L, R, scale, descale_q=dqt, descale_k=dkt, lse_out=lse,
                           num_splits=splits)
        mla.mla_device_error()
        return o, lse.cpu().numpy().astype(np.float64)

    o, lse = run(_u8(codes))
    check_close(to_f64(o), want, dtype, f"fp8 decode {geom}")
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - want_lse[fin])) < (1e-3 if dtype == "f32" else 1e-2)
    assert np.all(to_f64(o)[6] == 0) and np.all(lse[6] == -np.inf)      # the empty sequence
    # the page's check: one layer of a block-major unified slot reads bit-identically
    nb = codes.shape[0]
    unified = mi.permutation(7220, nb * 3 * page * E).astype(np.uint8)
    unified = np.where((unified & 0x7F) == 0x7F, 0, unified).astype(np.uint8).reshape(nb, 3, page, E)
    unified[:, 1] = codes
    u = _u8(unified)
    view = u[:, 1]
    assert not view.is_contiguous()
    o_view, lse_view = run(view)
    assert np.array_equal(to_host_bits(o_view), to_host_bits(o))
    assert np.array_equal(lse_view, lse)
    # other split counts: same tolerance
    o3, _ = run(_u8(codes), splits=5)
    check_close(to_f64(o3), want, dtype, f"fp8 decode {geom}, 5 splits")


def test_fp8_write_then_decode_round_trip(mla):
    # the step as a server runs it: new rows written into the e4m3 cache by the fp8 cache write,
    # then decoded with descale_k = the write's scale; against the oracle doing the same two steps
    import torch
    H, L, R, page = 128, 512, 64, 64
    E = L + R
    lens = [130, 64, 1]
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 1
    table = np.zeros((len(lens), max(need)), np.int32)
    perm = mi.permutation(7301, nb)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    slots = np.concatenate([[table[b, t // page] * page + t % page for t in range(lens[b])]
                            for b in range(len(lens))]).astype(np.int64)
    rows = int(sum(lens))
    kv = mi.encode(mi.draw("normal", 7302, rows * L, 0.3), "bf16").reshape(rows, L)
    kp = mi.encode(mi.draw("normal", 7303, rows * R, 0.3), "bf16").reshape(rows, R)
    cache = torch.zeros((nb, page, E), dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.25], dtype=torch.float32, device="cuda")
    mla.mla_cache_write_fp8(cache, to_dev(kv, "bf16"), to_dev(kp, "bf16"), torch.from_numpy(slots).cuda(), sc)
    q_bits = mi.encode(mi.draw("normal", 7304, len(lens) * H * E, 0.3), "bf16").reshape(len(lens), H, E)
    o = poisoned((len(lens), H, L), "bf16")
    mla.mla_decode_fp8(o, to_dev(q_bits, "bf16"), cache, torch.from_numpy(table).cuda(),
                       torch.from_numpy(np.array(lens, np.int32)).cuda(), L, R, 1.0 / math.sqrt(192),
                       descale_k=sc)
    mla.mla_device_error()
    st = orc.cache_write_fp8(np.zeros(nb * page * E, np.uint8), 0, nb, page, (page * E, E, 1),
                             mi.decode_f64(kv, "bf16"), mi.decode_f64(kp, "bf16"), slots, 0.25)
    assert np.array_equal(cache.cpu().numpy().reshape(-1), st)
    want, _ = orc.decode_fp8(mi.decode_f64(q_bits, "bf16"), st, 0, page, (page * E, E, 1), L, R, table,
                             np.array(lens), 1.0 / math.sqrt(192), 1.0, 0.25)
    check_close(to_f64(o), want, "bf16", "fp8 write then decode")


@pytest.mark.parametrize("H,R,page,dq,dk", [(128, 64, 16, -0.5, 2.0), (64, 0, 128, 1.0, 0.25),
                                           (64, 64, 64, 2.0, -1.0), (128, 0, 64, 1.0, 1.0),
                                           (128, 64, 48, 1.0, 0.5)],
                         ids=["h128_page16_neg_dq", "h64_nope_page128", "h64_rope_neg_dk", "h128_nope",
                              "h128_page48_rows_gathered"])
def test_fp8_decode_bf16_queries_geometries_and_descale_signs(mla, H, R, page, dq, dk):
    # the bf16-query decode over e4m3 rows at other head counts, rope widths and page sizes, with
    # descales of either sign (the score scale is then negative: the row maximum must follow)
    import torch
    L = 512
    E = L + R
    lens = [0, 1, 64, 65, 333, 1500, 63]
    codes, table = _fp8_batch(H, L, R, lens, page, 7401 + H + R + page, abs(dk))
    q_bits = mi.encode(mi.draw("normal", 7410 + H + R, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    scale = 1.0 / math.sqrt(E)
    want, want_lse = orc.decode_fp8(mi.decode_f64(q_bits, "bf16"), codes.reshape(-1), 0, page, (page * E, E, 1),
                                    L, R, table, np.array(lens), scale, dq, dk)
    o = poisoned((len(lens), H, L), "bf16")
    lse = torch.full((len(lens), H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_fp8(o, to_dev(q_bits, "bf16"), _u8(codes), torch.from_numpy(table).cuda(),
                       torch.from_numpy(np.array(lens, np.int32)).cuda(), L, R, scale,
                       descale_q=torch.tensor([dq], dtype=torch.float32, device="cuda"),
                       descale_k=torch.tensor([dk], dtype=torch.float32, device="cuda"), lse_out=lse)
    mla.mla_device_error()
    check_close(to_f64(o), want, "bf16", f"fp8 decode H={H} R={R} page={page}")
    got_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    assert np.max(np.abs(got_lse[fin] - want_lse[fin])) < 1e-2
    assert np.all(to_f64(o)[0] == 0)


def test_fp8_decode_single_row_reads_every_code_exactly(mla):
    # one cached row holding every finite code: with one key the softmax weight is 1, so o_lat is
    # that row's values, which bf16 holds exactly (subnormals and signs included; -0 reads as 0
    # after the weighted sum)
    import torch
    H, L, R, page = 128, 512, 64, 64
    E = L + R
    codes = np.arange(256, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0                         # no NaN codes in a score
    row = np.concatenate([codes, codes[::-1], np.full(R, 0x38, np.uint8)])   # rope: 1.0
    cache = np.zeros((2, page, E), np.uint8)
    cache[1, 0] = row
    table = np.array([[1]], np.int32)
    q_bits = mi.encode(mi.draw("normal", 7501, H * E, 0.1), "bf16").reshape(1, H, E)
    o = poisoned((1, H, L), "bf16")
    mla.mla_decode_fp8(o, to_dev(q_bits, "bf16"), _u8(cache), torch.from_numpy(table).cuda(),
                       torch.tensor([1], dtype=torch.int32, device="cuda"), L, R, 0.1)
    mla.mla_device_error()
    want = orc.e4m3_value(row[:L])
    got = to_f64(o)[0]
    assert np.array_equal(got, np.broadcast_to(want, (H, L)))


def test_sparse_decode_single_slot_reads_every_code_exactly(mla):
    # the ds_mla entry of one slot with every finite code and power-of-two scales: o_lat is the
    # products, exactly
    import torch
    H = 64
    codes = np.arange(256, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    lat = np.concatenate([codes, codes[::-1]])
    scales = np.array([1.0, 0.5, 2.0, 0.25], "<f4")
    rope = mi.to_bf16_bits(mi.normal(7502, 64) * np.float32(0.1))
    entry = np.concatenate([lat, scales.view(np.uint8), rope.astype("<u2").view(np.uint8)])
    cache = np.zeros((3, 16, 656), np.uint8)
    cache[2, 5] = entry
    q_bits = mi.encode(mi.draw("normal", 7503, H * 576, 0.1), "bf16").reshape(1, H, 576)
    o = poisoned((1, H, 512), "bf16")
    mla.mla_decode_sparse_fp8(o, to_dev(q_bits, "bf16"), _u8(cache),
                              torch.tensor([[-1, 2 * 16 + 5, -1]], dtype=torch.int32, device="cuda"), 0.1)
    mla.mla_device_error()
    want = orc.ds_mla_values(entry[None, :])[0][0]
    assert np.array_equal(to_f64(o)[0], np.broadcast_to(want, (H, 512)))


def test_fp8_decode_nan_code_poisons_only_its_sequence(mla):
    # a NaN code in one sequence's cache makes that sequence's output NaN (the oracle's reading
    # of a NaN code) and leaves the other sequences exact to the tolerance
    import torch
    H, L, R, page = 128, 512, 64, 64
    E = L + R
    lens = [200, 150]
    codes, table = _fp8_batch(H, L, R, lens, page, 7601, 1.0)
    blk = int(table[1, 1])
    codes[blk, 7, 300] = 0x7F                                   # NaN, in sequence 1's rows
    q_bits = mi.encode(mi.draw("normal", 7602, 2 * H * E, 0.3), "bf16").reshape(2, H, E)
    o = poisoned((2, H, L), "bf16")
    mla.mla_decode_fp8(o, to_dev(q_bits, "bf16"), _u8(codes), torch.from_numpy(table).cuda(),
                       torch.from_numpy(np.array(lens, np.int32)).cuda(), L, R, 1.0 / math.sqrt(E))
    mla.mla_device_error()
    with np.errstate(invalid="ignore"):
        want, _ = orc.decode_fp8(mi.decode_f64(q_bits, "bf16"), codes.reshape(-1), 0, page, (page * E, E, 1), L, R,
                                 table, np.array(lens), 1.0 / math.sqrt(E), 1.0, 1.0)
    got = to_f64(o)
    assert np.all(np.isnan(want[1])) and np.all(np.isnan(got[1]))
    check_close(got[0], want[0], "bf16", "fp8 decode next to a NaN sequence")


@pytest.mark.parametrize("H,R", [(128, 64), (64, 0)])
@pytest.mark.parametrize("tiny", [False, True], ids=["huge_elements", "tiny_rows"])
def test_fp8_decode_query_rows_of_any_magnitude(mla, H, R, tiny):
    # The e4m3 path's queries must keep every row's scores as its bf16 values give them, whatever
    # the row's magnitude. huge_elements: some rows hold one element of 2^18, 2^20 or -2^21 (beyond
    # f16's range, so a conversion of the queries to f16 would fail them) in a column whose cache
    # codes are all zero, so the scores stay ordinary; one row is zero. tiny_rows: every query
    # times 2^-24 (below f16's smallest subnormal) with the softmax scale times 2^24, so the
    # scores are the ordinary ones again.
    import torch
    L, page = 512, 64
    E = L + R
    lens = [300, 1000, 65]
    B = len(lens)
    codes, table = _fp8_batch(H, L, R, lens, page, 7701 + H, 1.0)
    q = mi.draw("normal", 7702 + H, B * H * E, 0.3).reshape(B, H, E).astype(np.float64)
    scale = 1.0 / math.sqrt(E)
    if tiny:
        q *= 2.0 ** -24
        scale *= 2.0 ** 24
    else:
        cols = [100, 300] + ([520, 560] if R else [])        # both CTAs' halves, rope included
        codes[:, :, cols] = 0
        pick = mi.permutation(7703 + H, B * H).reshape(B, H)
        for b in range(B):
            for h in range(H):
                k = pick[b, h] % 8
                if k < 3:
                    q[b, h, cols[pick[b, h] % len(cols)]] = (2.0 ** 18, 2.0 ** 20, -(2.0 ** 21))[k]
        q[1, 5] = 0.0
    q_bits = mi.to_bf16_bits(q.astype(np.float32))
    want, want_lse = orc.decode_fp8(mi.decode_f64(q_bits, "bf16"), codes.reshape(-1), 0, page, (page * E, E, 1),
                                    L, R, table, np.array(lens), scale, 1.0, 1.0)
    o = poisoned((B, H, L), "bf16")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_fp8(o, to_dev(q_bits, "bf16"), _u8(codes), torch.from_numpy(table).cuda(),
                       torch.from_numpy(np.array(lens, np.int32)).cuda(), L, R, scale, lse_out=lse)
    mla.mla_device_error()
    check_close(to_f64(o), want, "bf16", f"fp8 decode, query magnitudes (tiny={tiny}), H={H} R={R}")
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_lse))
    assert np.max(np.abs(got_lse - want_lse)) < 1e-2
