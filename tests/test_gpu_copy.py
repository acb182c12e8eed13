"""Steps 2 and 3 on the GPU: q concat and paged cache write, bit-exact against the
oracle's gathers, with NaN-poisoned outputs and sentinel-filled neighbours."""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import BF16_POISON, poisoned, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def _bits(x, dtype):
    return mi.to_bf16_bits(x) if dtype == "bf16" else x.astype(np.float32)


def _run_concat(mla, nope_t, rope_t, dtype):
    import torch
    T, H, L = nope_t.shape
    R = rope_t.shape[2]
    out = poisoned((T, H, L + R), dtype)
    mla.mla_concat_q(out, nope_t, rope_t)
    torch.cuda.synchronize()
    return to_host_bits(out)


def test_concat_unified_config_transposed_nope(mla):
    # q_nope storage [N=128, B=64, 512] (the bmm output), viewed as its [64,128,512] transpose.
    w = mi.write_concat_workload()
    N, B, L = w.q_nope_storage.shape
    store = to_dev(w.q_nope_storage, "bf16")
    nope = store.as_strided((B, N, L), (L, B * L, 1))
    assert not nope.is_contiguous()
    rope = to_dev(w.q_pe, "bf16")
    got = _run_concat(mla, nope, rope, "bf16")
    nope_h = orc.strided_view(w.q_nope_storage.reshape(-1), 0, (B, N, L), (L, B * L, 1))
    want = orc.concat_q(np.ascontiguousarray(nope_h), w.q_pe)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", ["contiguous_v3", "broadcast_rope", "nope_only", "odd_widths"])
def test_concat_cases(mla, dtype, case):
    T, H, L, R, Hr = {"contiguous_v3": (16, 128, 512, 64, 128), "broadcast_rope": (11, 16, 128, 64, 1),
                      "nope_only": (5, 8, 512, 0, 8), "odd_widths": (7, 5, 13, 3, 5)}[case]
    nope = _bits(mi.normal(55, T * H * L), dtype).reshape(T, H, L)
    rope = _bits(mi.normal(66, T * Hr * R), dtype).reshape(T, Hr, R)
    if dtype == "bf16" and nope.size > 4:
        nope.reshape(-1)[1] = 0x8000          # -0
        nope.reshape(-1)[3] = 0x7FC1          # a NaN payload
    got = _run_concat(mla, to_dev(nope, dtype), to_dev(rope, dtype), dtype)
    want = orc.concat_q(nope, rope)
    if dtype == "f32":
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(got, want)


def _unified(nb, n_layers, page, E, fill=0x1234):
    import torch
    return torch.full((nb, n_layers * page * E), fill, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def test_cache_write_unified_slot_view_no_bleed(mla):
    import torch
    w = mi.write_concat_workload()
    nb, page, E, n_layers, layer = w.num_blocks, w.page, w.entry, w.n_layers, w.layer
    L = w.kv_c.shape[1]
    kv_c, k_pe = to_dev(w.kv_c, "bf16"), to_dev(w.k_pe, "bf16")
    slots = torch.from_numpy(w.slots).cuda()
    big = _unified(nb, n_layers, page, E)
    flat = big.view(-1)
    view = flat.as_strided((nb, page, E), (n_layers * page * E, E, 1), layer * page * E)
    assert view.stride(0) == 110592 and view.storage_offset() == 36864
    mla.mla_cache_write(view, kv_c, k_pe, slots)
    # the contiguous per-layer reference through the same kernel
    ref = torch.zeros((nb, page, E), dtype=torch.bfloat16, device="cuda")
    mla.mla_cache_write(ref, kv_c, k_pe, slots)
    mla.mla_device_error()
    got = to_host_bits(flat)
    want = orc.cache_write(np.full(nb * n_layers * page * E, 0x1234, np.uint16), layer * page * E, nb,
                           page, (n_layers * page * E, E, 1), w.kv_c, w.k_pe, w.slots)
    assert np.array_equal(got, want)                                  # rows and neighbours, bit for bit
    written = np.zeros(nb * page, bool)
    written[w.slots] = True
    v = got.reshape(nb, n_layers, page, E)[:, layer].reshape(nb * page, E)
    assert np.array_equal(v[written], to_host_bits(ref).reshape(nb * page, E)[written])
    del L


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_write_padding_odd_widths_and_out_of_range(mla, dtype):
    import torch
    nb, page, L, R = 6, 16, 13, 3                          # odd widths: element path
    E, T = L + R, 40
    kv = _bits(mi.normal(1, T * L), dtype).reshape(T, L)
    kp = _bits(mi.normal(2, T * R), dtype).reshape(T, R)
    slots = mi.permutation(3, nb * page)[:T].copy()
    slots[4] = -1                                           # padding
    cache = to_dev(_bits(np.full(nb * page * E, 0.5, np.float32), dtype), dtype).view(nb, page, E)
    mla.mla_cache_write(cache, to_dev(kv, dtype), to_dev(kp, dtype), torch.from_numpy(slots).cuda())
    mla.mla_device_error()
    want = orc.cache_write(_bits(np.full(nb * page * E, 0.5, np.float32), dtype), 0, nb, page,
                           (page * E, E, 1), kv, kp, slots)
    got = to_host_bits(cache).reshape(-1)
    assert np.array_equal(got.view(np.uint16) if dtype == "bf16" else got.view(np.uint32),
                          want.view(np.uint16) if dtype == "bf16" else want.view(np.uint32))
    # a slot past the cache writes nothing and is reported
    bad = torch.tensor([nb * page + 3, 0], dtype=torch.int64, device="cuda")
    before = to_host_bits(cache).copy()
    mla.mla_cache_write(cache, to_dev(kv[:2], dtype), to_dev(kp[:2], dtype), bad)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_device_error()
    assert e.value.status == mla.MLA_ERR_DEVICE_DATA
    after = to_host_bits(cache)
    row0 = after.reshape(nb * page, E)[0]                   # slot 0 took token 1's row
    assert np.array_equal(row0[:L], kv[1]) and np.array_equal(row0[L:], kp[1])
    mask = np.ones(nb * page, bool)
    mask[0] = False
    assert np.array_equal(after.reshape(nb * page, E)[mask], before.reshape(nb * page, E)[mask])
    mla.mla_device_error()                                  # the error word was cleared


def test_poison_constant_is_the_pages():
    assert BF16_POISON == 0x7FC0


FUSED_CASES = [  # heads, batch, K (nope width), L, R, rope heads
    (128, 64, 128, 512, 64, 128),   # V3 decode batch 64 (tensor-core bmm)
    (16, 5, 128, 512, 64, 1),       # V2-Lite, one rope head broadcast
    (3, 7, 12, 20, 3, 3),           # odd widths (SIMT bmm, element concat)
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", FUSED_CASES, ids=["v3_b64", "v2lite_bcast", "odd"])
def test_absorb_into_q_cat_then_concat_in_place(mla, dtype, case):
    # The absorb writes q_lat straight into q_cat's first L columns through a [H,B,L] view;
    # the concat then gets those columns as its nope operand and moves only the rope.
    import math
    import torch
    from helpers import check_close, to_f64
    H, B, K, L, R, Hr = case
    qn = mi.encode(mi.draw("uniform", 71, B * H * K), dtype).reshape(B, H, K)
    w = mi.encode(mi.draw("uniform", 72, H * K * L, 1.0 / math.sqrt(K)), dtype).reshape(H, K, L)
    rope = _bits(mi.normal(73, B * Hr * R), dtype).reshape(B, Hr, R)
    q_cat = poisoned((B, H, L + R), dtype)
    lat = q_cat[:, :, :L]
    mla.mla_absorb_q(lat.transpose(0, 1), to_dev(qn, dtype).transpose(0, 1), to_dev(w, dtype))
    mla.mla_concat_q(q_cat, lat, to_dev(rope, dtype))
    torch.cuda.synchronize()
    got_bits = to_host_bits(q_cat)
    qn64 = np.transpose(mi.decode_f64(qn, dtype), (1, 0, 2))                # [H,B,K]
    want_lat = np.transpose(orc.bmm(qn64, mi.decode_f64(w, dtype)), (1, 0, 2))  # [B,H,L]
    check_close(to_f64(q_cat)[:, :, :L], want_lat, dtype, "absorbed latent columns")
    # the rope columns are the oracle's concat of them, bit for bit
    want_rope = orc.concat_q(got_bits[:, :, :L], rope)[:, :, L:]
    assert np.array_equal(got_bits[:, :, L:].view(np.uint16 if dtype == "bf16" else np.uint32),
                          want_rope.view(np.uint16 if dtype == "bf16" else np.uint32))
    # the latent columns are what the same absorb writes into a buffer of its own
    sep = poisoned((H, B, L), dtype)
    mla.mla_absorb_q(sep, to_dev(qn, dtype).transpose(0, 1), to_dev(w, dtype))
    torch.cuda.synchronize()
    assert np.array_equal(np.transpose(to_host_bits(sep), (1, 0, 2)), got_bits[:, :, :L])


@pytest.mark.parametrize("in_place", [False, True], ids=["separate_nope", "absorbed_in_place"])
def test_concat_and_cache_write_in_one_launch(mla, in_place):
    # Steps 2 and 3 together: the q_cat rows and the cache rows are the oracle's gathers,
    # bit for bit, and the neighbouring layers of the unified cache keep their sentinel.
    import torch
    w = mi.write_concat_workload()
    nb, page, E, n_layers, layer = w.num_blocks, w.page, w.entry, w.n_layers, w.layer
    N, B, L = w.q_nope_storage.shape
    R = w.q_pe.shape[2]
    store = to_dev(w.q_nope_storage, "bf16")
    nope = store.as_strided((B, N, L), (L, B * L, 1))
    out = poisoned((B, N, L + R), "bf16")
    if in_place:
        out[:, :, :L].copy_(nope)
        nope = out[:, :, :L]
    big = _unified(nb, n_layers, page, E)
    flat = big.view(-1)
    view = flat.as_strided((nb, page, E), (n_layers * page * E, E, 1), layer * page * E)
    mla.mla_concat_q_cache_write(out, nope, to_dev(w.q_pe, "bf16"), view, to_dev(w.kv_c, "bf16"),
                                 to_dev(w.k_pe, "bf16"), torch.from_numpy(w.slots).cuda())
    mla.mla_device_error()
    nope_h = orc.strided_view(w.q_nope_storage.reshape(-1), 0, (B, N, L), (L, B * L, 1))
    assert np.array_equal(to_host_bits(out), orc.concat_q(np.ascontiguousarray(nope_h), w.q_pe))
    want = orc.cache_write(np.full(nb * n_layers * page * E, 0x1234, np.uint16), layer * page * E, nb,
                           page, (n_layers * page * E, E, 1), w.kv_c, w.k_pe, w.slots)
    assert np.array_equal(to_host_bits(flat), want)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", ["odd_widths", "no_tokens", "no_rows"])
def test_concat_and_cache_write_in_one_launch_edges(mla, dtype, case):
    # Odd widths take the element path (two launches inside the call); an empty half leaves
    # only the other one to run.
    import torch
    T, H, L, R, Hr = (7, 5, 13, 3, 5) if case != "no_rows" else (0, 5, 16, 8, 5)
    nb, page, Lc, Rc = 6, 16, (13 if case == "odd_widths" else 512), (3 if case == "odd_widths" else 64)
    ntok = 0 if case == "no_tokens" else 40
    nope = _bits(mi.normal(81, T * H * L), dtype).reshape(T, H, L)
    rope = _bits(mi.normal(82, T * Hr * R), dtype).reshape(T, Hr, R)
    kv = _bits(mi.normal(83, ntok * Lc), dtype).reshape(ntok, Lc)
    kp = _bits(mi.normal(84, ntok * Rc), dtype).reshape(ntok, Rc)
    slots = mi.permutation(85, nb * page)[:ntok].copy()
    if ntok:
        slots[4] = -1
    E = Lc + Rc
    fill = _bits(np.full(nb * page * E, 0.5, np.float32), dtype)
    cache = to_dev(fill, dtype).view(nb, page, E)
    out = poisoned((T, H, L + R), dtype)
    mla.mla_concat_q_cache_write(out, to_dev(nope, dtype), to_dev(rope, dtype), cache, to_dev(kv, dtype),
                                 to_dev(kp, dtype), torch.from_numpy(slots).cuda())
    mla.mla_device_error()
    u = np.uint16 if dtype == "bf16" else np.uint32
    assert np.array_equal(to_host_bits(out).view(u), orc.concat_q(nope, rope).view(u))
    want = orc.cache_write(fill, 0, nb, page, (page * E, E, 1), kv, kp, slots)
    assert np.array_equal(to_host_bits(cache).reshape(-1).view(u), want.view(u))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", FUSED_CASES + [(64, 6, 256, 512, 0, 64)], ids=["v3_b64", "v2lite_bcast", "odd", "nope_h64"])
@pytest.mark.parametrize("bad_slot", [False, True], ids=["slots_ok", "slot_past_cache"])
def test_absorb_concat_cache_write_in_one_call(mla, dtype, case, bad_slot):
    # Steps 1 to 3 in one call (the copies alongside the absorb): the latent columns of q_cat
    # are the oracle's product and bit-identical to mla_absorb_q into a buffer of its own, the
    # rope columns and the whole unified cache buffer (its other layers' sentinels included)
    # are the oracle's, bit for bit; a slot past the cache is reported and skipped.
    import math
    import torch
    from helpers import check_close, to_f64
    H, B, K, L, R, Hr = case
    qn = mi.encode(mi.draw("uniform", 91, B * H * K), dtype).reshape(B, H, K)
    w = mi.encode(mi.draw("uniform", 92, H * K * L, 1.0 / math.sqrt(K)), dtype).reshape(H, K, L)
    rope = _bits(mi.normal(93, B * Hr * R), dtype).reshape(B, Hr, R)
    nb, page, n_layers, layer = 6, 16, 3, 1
    E = L + R
    ntok = 21
    kv = _bits(mi.normal(94, ntok * L), dtype).reshape(ntok, L)
    kp = _bits(mi.normal(95, ntok * R), dtype).reshape(ntok, R)
    slots = mi.permutation(96, nb * page)[:ntok].copy()
    slots[3] = -1                                              # padding: writes nothing
    if bad_slot:
        slots[7] = nb * page + 2
    fill = _bits(mi.normal(97, nb * n_layers * page * E), dtype)
    big = to_dev(fill, dtype)
    view = big.as_strided((nb, page, E), (n_layers * page * E, E, 1), layer * page * E)
    q_cat = poisoned((B, H, E), dtype)
    mla.mla_absorb_concat_cache_write(q_cat, to_dev(qn, dtype).transpose(0, 1), to_dev(w, dtype), to_dev(rope, dtype),
                                      view, to_dev(kv, dtype), to_dev(kp, dtype), torch.from_numpy(slots).cuda())
    if bad_slot:
        with pytest.raises(mla.MlaError) as e:
            mla.mla_device_error()
        assert e.value.status == mla.MLA_ERR_DEVICE_DATA
        slots[7] = -1                                          # what the oracle writes: the rest
    else:
        mla.mla_device_error()
    got = to_host_bits(q_cat)
    qn64 = np.transpose(mi.decode_f64(qn, dtype), (1, 0, 2))                    # [H,B,K]
    want_lat = np.transpose(orc.bmm(qn64, mi.decode_f64(w, dtype)), (1, 0, 2))  # [B,H,L]
    check_close(to_f64(q_cat)[:, :, :L], want_lat, dtype, "absorbed latent columns")
    sep = poisoned((H, B, L), dtype)
    mla.mla_absorb_q(sep, to_dev(qn, dtype).transpose(0, 1), to_dev(w, dtype))
    torch.cuda.synchronize()
    assert np.array_equal(np.transpose(to_host_bits(sep), (1, 0, 2)), got[:, :, :L])
    u = np.uint16 if dtype == "bf16" else np.uint32
    want_rope = orc.concat_q(got[:, :, :L], rope)[:, :, L:]
    assert np.array_equal(got[:, :, L:].view(u), want_rope.view(u))
    want_cache = orc.cache_write(fill, layer * page * E, nb, page, (n_layers * page * E, E, 1), kv, kp, slots)
    assert np.array_equal(to_host_bits(big).reshape(-1).view(u), want_cache.view(u))
