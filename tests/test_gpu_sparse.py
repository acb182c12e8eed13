"""Sparse top-k decode over an fp8 ds_mla cache on the GPU, against the float64 oracle
(``decode_sparse_ds_mla``).

The first case is the vLLM page's FlashMLA fp8 sparse decode configuration: 2 queries of
128 heads, 576-wide queries, 656-byte entries (unit scales), page 64, 32 blocks seen as
the middle layer of a 3-layer block-major buffer, top-k 128 with each query on its own
blocks. The layer view must read bit-identically to a contiguous copy, with finite,
nonzero output; both must be within the path's tolerances of the oracle (bf16 max-abs
2e-2 and relative L2 1e-2; fp32 max-abs 1e-4). The other cases scatter the slots over
the whole cache with ragged valid counts (none, some, all), non-unit scales, padding
interleaved, several split counts, a slot past the cache and a zero top-k."""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def _u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _views(w):
    """The unified buffer on the device and its layer view [num_blocks, page, 656]."""
    big = _u8(w.storage)
    E = 656
    view = big.as_strided((w.num_blocks, w.page, E), w.strides, w.offset)
    return big, view


def _run(mla, w, q, view, dtype, idx=None, splits=0):
    import torch
    B, H = q.shape[0], q.shape[1]
    o = poisoned((B, H, 512), dtype)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ind = torch.from_numpy(np.ascontiguousarray(w.indices if idx is None else idx, dtype=np.int32)).cuda()
    mla.mla_decode_sparse_fp8(o, q, view, ind, w.scale, lse_out=lse, num_splits=splits)
    mla.mla_device_error()
    return o, lse.cpu().numpy().astype(np.float64)


def _check_lse(lse, want, dtype):
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.max(np.abs(lse[fin] - want[fin])) < (1e-3 if dtype == "f32" else 1e-2)


def test_sparse_decode_pages_configuration(mla):
    w = mi.sparse_decode_workload()                       # batch 2, 128 heads, top-k 128, unit scales
    q = to_dev(w.q_cat, "bf16")
    _, view = _views(w)
    assert not view.is_contiguous() and view.stride(0) == 3 * 64 * 656
    o_view, lse_view = _run(mla, w, q, view, "bf16")
    contiguous = view.contiguous()
    o_ref, lse_ref = _run(mla, w, q, contiguous, "bf16")
    assert np.array_equal(to_host_bits(o_view), to_host_bits(o_ref))            # the page's check
    assert np.array_equal(lse_view, lse_ref)
    got = to_f64(o_ref)
    assert np.isfinite(got).all() and np.abs(got).max() > 0
    want, want_lse = orc.decode_sparse_ds_mla(mi.decode_f64(w.q_cat, "bf16"), w.storage, w.offset, w.num_blocks,
                                              w.page, w.strides, w.indices, w.scale)
    check_close(got, want, "bf16", "sparse decode, the pages' configuration")
    _check_lse(lse_ref, want_lse, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_sparse_decode_scattered_slots_ragged_counts(mla, dtype, splits):
    w = mi.sparse_decode_workload(batch=7, heads=128, topk=320, num_blocks=24, page=64, pattern="scattered",
                                  unit_scales=False, config_index=8)
    idx = w.indices.copy()
    idx[2] = -1                                            # a query with no valid slot
    idx[4, : idx.shape[1] // 2] = np.arange(idx.shape[1] // 2)   # half full, in slot order
    q_bits = w.q_cat if dtype == "bf16" else mi.bf16_bits_to_f32(w.q_cat)
    q = to_dev(q_bits, dtype)
    _, view = _views(w)
    o, lse = _run(mla, w, q, view, dtype, idx, splits)
    want, want_lse = orc.decode_sparse_ds_mla(mi.decode_f64(w.q_cat, "bf16"), w.storage, w.offset, w.num_blocks,
                                              w.page, w.strides, idx, w.scale)
    check_close(to_f64(o), want, dtype, f"sparse decode, {splits} splits")
    _check_lse(lse, want_lse, dtype)
    assert np.all(to_f64(o)[2] == 0) and np.all(lse[2] == -np.inf)


def test_sparse_decode_64_heads_and_sharp_scores(mla):
    # fewer heads, and queries scaled so the softmax is sharp (the rescaling path matters)
    w = mi.sparse_decode_workload(batch=3, heads=64, topk=256, num_blocks=16, page=64, pattern="scattered",
                                  unit_scales=False, config_index=9)
    q_bits = mi.to_bf16_bits(mi.bf16_bits_to_f32(w.q_cat) * np.float32(40.0))
    q = to_dev(q_bits, "bf16")
    _, view = _views(w)
    o, lse = _run(mla, w, q, view, "bf16")
    want, want_lse = orc.decode_sparse_ds_mla(mi.decode_f64(q_bits, "bf16"), w.storage, w.offset, w.num_blocks,
                                              w.page, w.strides, w.indices, w.scale)
    check_close(to_f64(o), want, "bf16", "sparse decode, sharp")
    _check_lse(lse, want_lse, "bf16")


def test_sparse_decode_slot_past_the_cache_is_skipped_and_reported(mla):
    w = mi.sparse_decode_workload(batch=2, heads=16, topk=64, num_blocks=8, page=16, config_index=10)
    idx = w.indices.copy()
    idx[1, 3] = w.num_blocks * w.page + 5
    q = to_dev(w.q_cat, "bf16")
    _, view = _views(w)
    import torch
    o = poisoned((2, 16, 512), "bf16")
    mla.mla_decode_sparse_fp8(o, q, view, torch.from_numpy(idx).cuda(), w.scale)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_device_error()
    assert e.value.status == mla.MLA_ERR_DEVICE_DATA
    skipped = idx.copy()
    skipped[1, 3] = -1
    want, _ = orc.decode_sparse_ds_mla(mi.decode_f64(w.q_cat, "bf16"), w.storage, w.offset, w.num_blocks,
                                       w.page, w.strides, skipped, w.scale)
    check_close(to_f64(o), want, "bf16", "sparse decode without the bad slot")
    mla.mla_device_error()                                  # the error word was cleared


def test_sparse_decode_zero_topk_and_argument_errors(mla):
    import torch
    w = mi.sparse_decode_workload(batch=2, heads=16, topk=8, num_blocks=4, page=16, config_index=11)
    q = to_dev(w.q_cat, "bf16")
    _, view = _views(w)
    o, lse = _run(mla, w, q, view, "bf16", idx=np.zeros((2, 0), np.int32))
    assert np.all(to_f64(o) == 0) and np.all(lse == -np.inf)
    ind = torch.from_numpy(w.indices).cuda()
    bad_q = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_sparse_fp8(torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda"), bad_q, view,
                                  ind, w.scale)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    with pytest.raises(mla.MlaError) as e:                  # an entry that is not 656 bytes
        mla.mla_decode_sparse_fp8(torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda"), q,
                                  view[:, :, :576], ind, w.scale)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_sparse_decode_large_batch_sampled(mla):
    # 64 queries x 128 heads, top-k 2048 over a 1024-block cache: every query's output against
    # the oracle on a sample of queries
    w = mi.sparse_decode_workload(batch=64, heads=128, topk=2048, num_blocks=1024, page=64, n_layers=1, layer=0,
                                  pattern="scattered", unit_scales=False, config_index=12)
    q = to_dev(w.q_cat, "bf16")
    _, view = _views(w)
    o, lse = _run(mla, w, q, view, "bf16")
    ids = [0, 17, 40, 63]
    want, want_lse = orc.decode_sparse_ds_mla(mi.decode_f64(w.q_cat, "bf16"), w.storage, w.offset, w.num_blocks,
                                              w.page, w.strides, w.indices, w.scale, batch_ids=ids)
    check_close(to_f64(o)[ids], want, "bf16", "sparse decode, 64 x top-2048")
    _check_lse(lse[ids], want_lse, "bf16")
