"""Step 4 (prefill) on the GPU: causal attention of many queries per sequence over
the paged cache, bottom-right aligned (pure prefill and queries that are a
suffix of a populated cache), against the float64 oracle."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _tables(kv_lens, page, seed):
    need = [(n + page - 1) // page for n in kv_lens]
    nb = sum(need) + 1
    perm = mi.permutation(seed, nb)
    table = np.zeros((len(kv_lens), max(max(need), 1)), np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    return table, nb


def run_prefill(mla, q_bits, cache_bits, table, q_lens, kv_lens, dtype, L, R, scale):
    import torch
    T, H, E = q_bits.shape
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    o = poisoned((T, H, L), dtype)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_prefill(o, to_dev(q_bits, dtype), to_dev(cache_bits, dtype),
                    torch.from_numpy(table).cuda(), torch.from_numpy(cu).cuda(),
                    torch.from_numpy(np.asarray(kv_lens, np.int32)).cuda(), int(max(q_lens)), L, R, scale,
                    lse_out=lse)
    mla.mla_device_error()
    return o, lse.cpu().numpy().astype(np.float64), cu


@pytest.mark.parametrize("dims", [(4, 24, 8, 32, 64), (3, 12, 4, 20, 48), (4, 32, 0, 32, 64)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_small_geometries(mla, dims, dtype):
    H, P, R, V, L = dims
    E = L + R
    q_lens = [6, 3, 17, 1, 70]
    kv_lens = [6, 11, 17, 1, 200]             # pure prefill and suffix-of-cache shapes
    page = 16
    table, nb = _tables(kv_lens, page, 80)
    cache = mi.encode(mi.draw("uniform", 81, nb * page * E), dtype).reshape(nb, page, E)
    q = mi.encode(mi.draw("uniform", 82, sum(q_lens) * H * E, 2.0), dtype).reshape(sum(q_lens), H, E)
    scale = 1.0 / math.sqrt(P + R)
    o, lse, cu = run_prefill(mla, q, cache, table, q_lens, kv_lens, dtype, L, R, scale)
    storage = mi.decode_f64(cache.reshape(-1), dtype)
    want, want_lse = orc.prefill(mi.decode_f64(q, dtype), cu, np.array(kv_lens), storage, 0, page,
                                 (page * E, E, 1), L, R, table, scale)
    check_close(to_f64(o), want, dtype, f"prefill dims {dims}")
    assert np.max(np.abs(lse - want_lse)) < 1e-3


def test_prefill_fp32_production_nope_geometry(mla):
    # The f32 core at the NoPE production geometry (64 heads, rank 512, no rope, 256-d nope and
    # v heads: scale 1/sqrt(256)) with the (t_q, t_kv) shapes of the memra prefill gate, pure
    # prefill and a suffix of a populated cache, held to max-abs 1e-4 and to 1e-4 * max(|o|, 1).
    H, L, R, page = 64, 512, 0, 64
    E = L + R
    q_lens = [4, 3, 17]
    kv_lens = [4, 9, 17]
    table, nb = _tables(kv_lens, page, 88)
    cache = mi.encode(mi.draw("uniform", 89, nb * page * E), "f32").reshape(nb, page, E)
    q = mi.encode(mi.draw("uniform", 90, sum(q_lens) * H * E), "f32").reshape(sum(q_lens), H, E)
    scale = 1.0 / math.sqrt(256)
    o, lse, cu = run_prefill(mla, q, cache, table, q_lens, kv_lens, "f32", L, R, scale)
    storage = mi.decode_f64(cache.reshape(-1), "f32")
    want, want_lse = orc.prefill(mi.decode_f64(q, "f32"), cu, np.array(kv_lens), storage, 0, page,
                                 (page * E, E, 1), L, R, table, scale)
    info = check_close(to_f64(o), want, "f32", "fp32 prefill, production NoPE geometry")
    assert info["scaled"] <= 1e-4, info
    assert np.max(np.abs(lse - want_lse)) < 1e-4


def test_prefill_nope_full_size_sampled(mla):
    # 4 x 2048 causal, 64 heads, L=512, R=0; q_lat-like queries ~N(0,1)*0.7, latent rows ~N(0,1).
    H, L, R, page = 64, 512, 0, 64
    q_lens = kv_lens = [2048] * 4
    table, nb = _tables(kv_lens, page, 4077)
    cache = mi.encode(mi.draw("normal", 4033, nb * page * L), "bf16").reshape(nb, page, L)
    T = sum(q_lens)
    q = mi.encode(mi.draw("normal", 4011, T * H * L, 0.7), "bf16").reshape(T, H, L)
    scale = 1.0 / math.sqrt(256)
    o, lse, cu = run_prefill(mla, q, cache, table, q_lens, kv_lens, "bf16", L, R, scale)
    got = to_f64(o)
    assert np.all(np.isfinite(got))
    rows = [0, 1, 63, 64, 1000, 2047, 2048, 4095, 6000, 8191]
    storage = mi.decode_f64(cache.reshape(-1), "bf16")
    want, want_lse = orc.prefill(mi.decode_f64(q, "bf16"), cu, np.array(kv_lens), storage, 0, page,
                                 (page * L, L, 1), L, R, table, scale, rows_wanted=rows)
    check_close(got[rows], want, "bf16", "nope prefill (sampled rows)")
    assert np.max(np.abs(lse[rows] - want_lse)) < 1e-2


@pytest.mark.parametrize("H,R", [(128, 64), (64, 0)])
def test_prefill_tensor_core_rows_without_keys(mla, H, R):
    # The tensor-core shapes with sequences whose query rows see no cache row at all (kv_len 0,
    # or more queries than cached rows), back to back, next to ordinary ones and an empty query
    # range: such rows give o = 0 and lse = -inf, and the rows after them must be right.
    L, page = 512, 64
    E = L + R
    q_lens = [5, 3, 70, 1, 10, 0, 130]
    kv_lens = [0, 0, 70, 1, 4, 10, 300]
    table, nb = _tables(kv_lens, page, 91)
    cache = mi.encode(mi.draw("normal", 92, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    T = sum(q_lens)
    q = mi.encode(mi.draw("normal", 93, T * H * E, 0.5), "bf16").reshape(T, H, E)
    scale = 1.0 / math.sqrt(192)
    o, lse, cu = run_prefill(mla, q, cache, table, q_lens, kv_lens, "bf16", L, R, scale)
    storage = mi.decode_f64(cache.reshape(-1), "bf16")
    want, want_lse = orc.prefill(mi.decode_f64(q, "bf16"), cu, np.array(kv_lens), storage, 0, page,
                                 (page * E, E, 1), L, R, table, scale)
    got = to_f64(o)
    check_close(got, want, "bf16", f"prefill rows without keys H={H} R={R}")
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - want_lse[fin])) < 1.2e-2   # ln(1 + 3 * 2^-8): see the decode tests
    assert np.all(got[~fin.all(axis=1)] == 0)


@pytest.mark.parametrize("page", [16, 128])
@pytest.mark.parametrize("H,R", [(128, 64), (64, 0)])
def test_prefill_tensor_core_page_sizes(mla, page, H, R):
    # Pages of 16 rows (four TMA boxes per 64-key tile) and of 128 rows (tiles starting inside
    # a page) on the tensor-core prefill, with pure-prefill and suffix-of-cache sequences.
    L = 512
    E = L + R
    q_lens = [70, 33, 1, 129]
    kv_lens = [70, 130, 17, 300]
    table, nb = _tables(kv_lens, page, 190 + page)
    cache = mi.encode(mi.draw("normal", 191, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    T = sum(q_lens)
    q = mi.encode(mi.draw("normal", 192, T * H * E, 0.5), "bf16").reshape(T, H, E)
    scale = 1.0 / math.sqrt(192)
    o, lse, cu = run_prefill(mla, q, cache, table, q_lens, kv_lens, "bf16", L, R, scale)
    storage = mi.decode_f64(cache.reshape(-1), "bf16")
    want, want_lse = orc.prefill(mi.decode_f64(q, "bf16"), cu, np.array(kv_lens), storage, 0, page,
                                 (page * E, E, 1), L, R, table, scale)
    check_close(to_f64(o), want, "bf16", f"prefill page {page} H={H} R={R}")
    assert np.max(np.abs(lse - want_lse)) < 1.2e-2   # ln(1 + 3 * 2^-8): see the decode tests
