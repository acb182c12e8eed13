"""mla_decode_noalloc, the decode for callers that cannot allocate device memory.

Such callers (code inside another framework's memory pool, plugins whose host
forbids cudaMalloc on the hot path, runtimes that reserve all device memory up
front) cannot provide mla_decode's workspace; this entry point keeps that
scratch in a fixed array inside the library instead. The test calls it through
the C ABI twice in a row and checks each result against the float64 oracle,
within the tolerances the other parity tests use (fp32 max-abs 1e-4; bf16
max-abs 2e-2 and relative L2 1e-2), and bit for bit against mla_decode with a
workspace (the same schedule and kernels). This file is collected last so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def _workload(which):
    if which == "v3_bf16":
        w = mi.v3_decode_small()
        q = mi.encode(mi.draw("normal", 1011, w.batch * w.geom.n_head * w.geom.entry, 0.1), "bf16")
    elif which == "v3_bf16_b64":
        # the 64-sequence batch of 1K..16K rows: the largest scratch this entry point serves
        w = mi.v3_decode_large(materialize_cache=True)
        q = mi.encode(mi.draw("normal", 3011, w.batch * w.geom.n_head * w.geom.entry, 3.0), "bf16")
    else:
        w = mi.v2_lite_decode()
        q = mi.encode(mi.draw("uniform", 11, w.batch * w.geom.n_head * w.geom.entry), "f32")
    return w, q.reshape(w.batch, w.geom.n_head, w.geom.entry)


def _oracle(w, q_bits):
    g = w.geom
    cache = w.full_cache()
    nb, page, E = cache.shape
    storage = mi.decode_f64(cache.reshape(-1), w.dtype)
    return orc.decode(mi.decode_f64(q_bits, w.dtype), storage, 0, page, (page * E, E, 1), g.kv_rank, g.d_rope,
                      w.block_table, w.seq_lens, w.scale)


@pytest.mark.parametrize("which", ["v3_bf16", "v2lite_f32", "v3_bf16_b64"])
def test_noalloc_decode_matches_oracle_twice(mla, which):
    import torch
    w, q_bits = _workload(which)
    g, dt = w.geom, w.dtype
    B, H, L, R = w.batch, g.n_head, g.kv_rank, g.d_rope
    q = to_dev(q_bits, dt)
    cache = to_dev(w.full_cache(), dt)
    table = torch.from_numpy(w.block_table).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    want, want_lse = _oracle(w, q_bits)
    # mla_decode with a workspace, for the bit-for-bit comparison
    o_ref = poisoned((B, H, L), dt)
    mla.mla_decode(o_ref, q, cache, table, lens, L, R, w.scale)
    mla.mla_device_error()
    lib = mla.lib()
    code = mla.MLA_F32 if dt == "f32" else mla.MLA_BF16
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        o = poisoned((B, H, L), dt)
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.mla_decode_noalloc(code, mla.as_mla_tensor(o), lse.data_ptr(), mla.as_mla_tensor(q),
                                    mla.as_mla_tensor(cache), table.data_ptr(), table.stride(0),
                                    table.shape[1], lens.data_ptr(), L, R, w.scale, 0, stream)
        assert st == mla.MLA_OK, lib.mla_last_error()
        mla.mla_device_error()
        check_close(to_f64(o), want, dt, f"noalloc call {call + 1} vs the oracle")
        got_lse = lse.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got_lse - want_lse)) < (1e-3 if dt == "f32" else 1.2e-2)
        assert np.array_equal(to_host_bits(o), to_host_bits(o_ref)), "noalloc differs from mla_decode"


def test_noalloc_reports_the_errors_of_mla_decode(mla):
    # One validator serves both entry points: the same malformed calls give the same codes.
    import torch
    lib = mla.lib()
    L, R, H = 512, 64, 128
    q = torch.zeros((2, H, L + R), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((2, H, L), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((4, 64, L + R), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    lens = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = torch.empty(mla.mla_decode_workspace_size(2, H, L, 0), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    T = mla.as_mla_tensor
    q_wide = torch.zeros((2, H, 1024), dtype=torch.bfloat16, device="cuda")
    o_wide = torch.zeros((2, H, 1024), dtype=torch.bfloat16, device="cuda")
    cache_wide = torch.zeros((4, 64, 1024), dtype=torch.bfloat16, device="cuda")
    huge = cache[:1].expand(2 ** 31, 64, L + R)            # more blocks than an int32 counts (stride 0)
    cases = {
        "q width != L + R": (T(o), T(q[:, :, :L]), T(cache), table.data_ptr(), 4, 4, lens.data_ptr(), L, R),
        "null block table": (T(o), T(q), T(cache), None, 4, 4, lens.data_ptr(), L, R),
        "max_blocks > stride": (T(o), T(q), T(cache), table.data_ptr(), 2, 4, lens.data_ptr(), L, R),
        "rank beyond 512": (T(o_wide), T(q_wide), T(cache_wide), table.data_ptr(), 4, 4, lens.data_ptr(), 1024, 0),
        "blocks beyond int32": (T(o), T(q), T(huge), table.data_ptr(), 4, 4, lens.data_ptr(), L, R),
    }
    for name, (ot, qt, ct, tb, stride, mb, ln, l_, r_) in cases.items():
        a = lib.mla_decode(mla.MLA_BF16, ot, None, qt, ct, tb, stride, mb, ln, l_, r_, 0.1, 0,
                           ws.data_ptr(), ws.numel(), stream)
        msg_a = lib.mla_last_error()
        b = lib.mla_decode_noalloc(mla.MLA_BF16, ot, None, qt, ct, tb, stride, mb, ln, l_, r_, 0.1, 0, stream)
        msg_b = lib.mla_last_error()
        assert a == b and a != mla.MLA_OK, (name, a, b)
        assert msg_a == msg_b, (name, msg_a, msg_b)


def test_noalloc_rejects_batches_beyond_the_static_scratch(mla):
    import torch
    B, H, L, R = 4096, 128, 512, 64                 # needs far more than the fixed scratch
    q = torch.zeros(L + R, dtype=torch.bfloat16, device="cuda").as_strided((B, H, L + R), (0, 0, 1))
    o = torch.zeros(L, dtype=torch.bfloat16, device="cuda").as_strided((B, H, L), (0, 0, 1))
    cache = torch.zeros((4, 64, L + R), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    lib = mla.lib()
    st = lib.mla_decode_noalloc(mla.MLA_BF16, mla.as_mla_tensor(o), None, mla.as_mla_tensor(q),
                                mla.as_mla_tensor(cache), table.data_ptr(), 1, 1, lens.data_ptr(), L, R,
                                0.1, 0, torch.cuda.current_stream().cuda_stream)
    assert st == mla.MLA_ERR_UNSUPPORTED
    assert b"scratch" in lib.mla_last_error()
