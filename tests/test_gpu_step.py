"""The whole path on the GPU: absorb -> concat -> cache write -> decode -> v_up for
one decode step (and absorb -> concat -> cache write -> prefill -> v_up for a
prefill), through the C ABI, against the oracle's float64 composition of the
same steps."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def gpu_decode_step(mla, w, layout="contiguous", num_splits=0):
    """Run one decode step of workload ``w`` through the library; returns (out, o_lat, cache)."""
    import torch
    g, dt = w.geom, w.dtype
    B, H, P, R, V, L = w.batch, g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank
    E = L + R
    q_nope = to_dev(w.q_nope, dt)                               # [B,H,P]
    q_pe = to_dev(w.q_pe, dt)                                   # [B,H,R]
    w_uk, w_uv = to_dev(w.w_uk, dt), to_dev(w.w_uv, dt)
    q_lat_store = poisoned((H, B, L), dt)                       # bmm output [H,B,L]
    mla.mla_absorb_q(q_lat_store, q_nope.transpose(0, 1), w_uk)
    q_cat = poisoned((B, H, E), dt)
    mla.mla_concat_q(q_cat, q_lat_store.transpose(0, 1), q_pe)
    if layout == "contiguous":
        cache = to_dev(w.full_cache(), dt)
    else:
        nb, page = w.num_blocks, w.page
        big = torch.zeros((nb, 3, page, E), dtype=cache_dtype(dt), device="cuda")
        big[:, 1].copy_(to_dev(w.full_cache(), dt))
        cache = big[:, 1]
    mla.mla_cache_write(cache, to_dev(w.new_kv_c, dt), to_dev(w.new_k_pe, dt),
                        torch.from_numpy(w.slots).cuda())
    o_lat = poisoned((B, H, L), dt)
    mla.mla_decode(o_lat, q_cat, cache, torch.from_numpy(w.block_table).cuda(),
                   torch.from_numpy(w.seq_lens).cuda(), L, R, w.scale, num_splits=num_splits)
    out_store = poisoned((B, H, V), dt)
    mla.mla_v_up(out_store.transpose(0, 1), o_lat.transpose(0, 1), w_uv)
    mla.mla_device_error()
    return out_store, o_lat, cache


def cache_dtype(dt):
    import torch
    return torch.float32 if dt == "f32" else torch.bfloat16


def oracle_decode_step(w, ids=None):
    g, dt = w.geom, w.dtype
    E, page = g.entry, w.page
    storage = mi.decode_f64(w.full_cache().reshape(-1), dt)
    return orc.decode_step(mi.decode_f64(w.q_nope, dt), mi.decode_f64(w.q_pe, dt),
                           mi.decode_f64(w.w_uk, dt), mi.decode_f64(w.w_uv, dt),
                           mi.decode_f64(w.new_kv_c, dt), mi.decode_f64(w.new_k_pe, dt), w.slots,
                           storage, 0, page, (page * E, E, 1), w.block_table, w.seq_lens, w.scale,
                           batch_ids=ids)


@pytest.mark.parametrize("which", ["v2lite_f32", "v3_bf16"])
def test_decode_step_end_to_end(mla, which):
    w = mi.v2_lite_decode() if which == "v2lite_f32" else mi.v3_decode_small()
    out, o_lat, cache = gpu_decode_step(mla, w)
    want_out, want_olat, _, after = oracle_decode_step(w)
    check_close(to_f64(o_lat), want_olat, w.dtype, f"{which} o_lat")
    check_close(to_f64(out), want_out, w.dtype, f"{which} out")
    # the appended rows are in the cache bit for bit
    got_cache = to_host_bits(cache).reshape(-1)
    assert np.array_equal(mi.decode_f64(got_cache, w.dtype), after)


def test_decode_step_unified_view_matches_contiguous(mla):
    w = mi.v3_decode_small()
    out_a, olat_a, _ = gpu_decode_step(mla, w)
    out_b, olat_b, _ = gpu_decode_step(mla, w, layout="unified")
    assert np.array_equal(to_host_bits(olat_a), to_host_bits(olat_b))
    assert np.array_equal(to_host_bits(out_a), to_host_bits(out_b))


def test_prefill_pipeline_nope_sampled(mla):
    """The NoPE prefill workload end to end on sampled rows: absorb -> concat (R=0) ->
    cache write of every row -> causal prefill -> v_up."""
    import torch
    w = mi.nope_prefill()
    g = w.geom
    H, P, R, V, L = g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank
    T = int(w.q_lens.sum())
    E = L + R
    dt = "bf16"
    q_nope = to_dev(w.q_nope, dt)
    q_lat = poisoned((H, T, L), dt)
    mla.mla_absorb_q(q_lat, q_nope.transpose(0, 1), to_dev(w.w_uk, dt))
    q_cat = poisoned((T, H, E), dt)
    mla.mla_concat_q(q_cat, q_lat.transpose(0, 1), to_dev(w.q_pe, dt))
    cache = torch.zeros((w.num_blocks, w.page, E), dtype=torch.bfloat16, device="cuda")
    mla.mla_cache_write(cache, to_dev(w.kv_c, dt), to_dev(w.k_pe, dt),
                        torch.from_numpy(w.slot_mapping()).cuda())
    o_lat = poisoned((T, H, L), dt)
    cu = torch.from_numpy(w.cu_seqlens_q).cuda()
    mla.mla_prefill(o_lat, q_cat, cache, torch.from_numpy(w.block_table).cuda(), cu,
                    torch.from_numpy(w.kv_lens).cuda(), int(w.q_lens.max()), L, R, w.scale)
    out = poisoned((T, H, V), dt)
    mla.mla_v_up(out.transpose(0, 1), o_lat.transpose(0, 1), to_dev(w.w_uv, dt))
    mla.mla_device_error()
    rows = [0, 5, 2047, 2048, 5000, 8191]
    # oracle: absorb the sampled rows, write every row into a float64 cache, prefill, v_up
    q_lat64 = orc.absorb_q(np.transpose(mi.decode_f64(w.q_nope[rows], dt), (1, 0, 2)),
                           mi.decode_f64(w.w_uk, dt))                       # [H,n,L]
    storage = orc.cache_write(np.zeros(w.num_blocks * w.page * E), 0, w.num_blocks, w.page,
                              (w.page * E, E, 1), mi.decode_f64(w.kv_c, dt), mi.decode_f64(w.k_pe, dt),
                              w.slot_mapping())
    q_full = np.zeros((T, H, E))
    q_full[rows, :, :L] = np.transpose(q_lat64, (1, 0, 2))
    want_olat, _ = orc.prefill(q_full, w.cu_seqlens_q, w.kv_lens, storage, 0, w.page, (w.page * E, E, 1),
                               L, R, w.block_table, w.scale, rows_wanted=rows)
    want_out = np.transpose(orc.v_up(np.transpose(want_olat, (1, 0, 2)), mi.decode_f64(w.w_uv, dt)),
                            (1, 0, 2))
    check_close(to_f64(o_lat)[rows], want_olat, dt, "prefill pipeline o_lat")
    check_close(to_f64(out)[rows], want_out, dt, "prefill pipeline out")


def gpu_decode_v_up_step(mla, w, num_splits=0):
    """Absorb, concat, cache write, then decode and v_up as the one call mla_decode_v_up;
    returns (out, lse)."""
    import torch
    g, dt = w.geom, w.dtype
    B, H, R, V, L = w.batch, g.n_head, g.d_rope, g.d_v, g.kv_rank
    E = L + R
    q_lat_store = poisoned((H, B, L), dt)
    mla.mla_absorb_q(q_lat_store, to_dev(w.q_nope, dt).transpose(0, 1), to_dev(w.w_uk, dt))
    q_cat = poisoned((B, H, E), dt)
    mla.mla_concat_q(q_cat, q_lat_store.transpose(0, 1), to_dev(w.q_pe, dt))
    cache = to_dev(w.full_cache(), dt)
    mla.mla_cache_write(cache, to_dev(w.new_kv_c, dt), to_dev(w.new_k_pe, dt), torch.from_numpy(w.slots).cuda())
    out = poisoned((B, H, V), dt)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_v_up(out, q_cat, cache, torch.from_numpy(w.block_table).cuda(),
                        torch.from_numpy(w.seq_lens).cuda(), L, R, w.scale, to_dev(w.w_uv, dt), lse_out=lse,
                        num_splits=num_splits)
    mla.mla_device_error()
    return out, lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("splits", [0, 5])
@pytest.mark.parametrize("which", ["v2lite_f32", "v3_bf16"])
def test_decode_v_up_one_call_matches_oracle(mla, which, splits):
    # bf16 at V = 128 runs the combine and the un-projection as one kernel; fp32 runs them as
    # the separate kernels behind the same call
    w = mi.v2_lite_decode() if which == "v2lite_f32" else mi.v3_decode_small()
    out, lse = gpu_decode_v_up_step(mla, w, splits)
    want_out, _, want_lse, _ = oracle_decode_step(w)
    check_close(to_f64(out), want_out, w.dtype, f"{which} out, {splits} splits")
    assert np.max(np.abs(lse - want_lse)) < (1e-3 if w.dtype == "f32" else 1.2e-2)


def test_decode_v_up_equals_decode_then_v_up(mla):
    # the fused kernel rounds o_lat to bf16 before the MMA as the two calls do; only the
    # tensor core's summation order differs, so the outputs agree to about one bf16 step
    w = mi.v3_decode_small()
    out_sep, _, _ = gpu_decode_step(mla, w)
    out_one, _ = gpu_decode_v_up_step(mla, w)
    a, b = to_f64(out_sep), to_f64(out_one)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6)


def test_decode_v_up_nope_geometry_two_v_tiles_ragged_batch(mla):
    # 64 heads, R = 0, V = 256 (two 128-wide v tiles), 70 sequences (two chunks of 64), ragged
    # and empty lengths, split across units
    lens = np.array([(37 * i * i + 11 * i) % 900 for i in range(70)], np.int32)
    lens[5] = 0
    lens[66] = 0
    w = mi.decode_workload(mi.NOPE_64, "bf16", lens, 64, config_index=21, name="nope_vup")
    out, lse = gpu_decode_v_up_step(mla, w, num_splits=40)
    ids = [0, 5, 17, 33, 63, 64, 66, 69]
    want_out, _, want_lse, _ = oracle_decode_step(w, ids)
    check_close(to_f64(out)[ids], want_out, "bf16", "NoPE geometry out")
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse[ids]), fin)
    assert np.max(np.abs(lse[ids][fin] - want_lse[fin])) < 1.2e-2
    assert np.all(to_f64(out)[5] == 0) and np.all(to_f64(out)[66] == 0)
