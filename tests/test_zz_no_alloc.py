"""mla_decode_noalloc, the decode for callers that cannot allocate device memory.

Such callers (code inside another framework's memory pool, plugins whose host
forbids cudaMalloc on the hot path, runtimes that reserve all device memory up
front) cannot provide mla_decode's workspace; this entry point keeps that
scratch in a fixed array inside the library instead. The test calls it through
the C ABI twice in a row and checks each result against mla_decode's own
output, within the tolerances the other parity tests use (fp32 max-abs 1e-4;
bf16 max-abs 2e-2 and relative L2 1e-2). This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import mla_inputs as mi
from helpers import check_close, poisoned, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _workload(which):
    if which == "v3_bf16":
        w = mi.v3_decode_small()
        q = mi.encode(mi.draw("normal", 1011, w.batch * w.geom.n_head * w.geom.entry, 0.1), "bf16")
    else:
        w = mi.v2_lite_decode()
        q = mi.encode(mi.draw("uniform", 11, w.batch * w.geom.n_head * w.geom.entry), "f32")
    return w, q.reshape(w.batch, w.geom.n_head, w.geom.entry)


@pytest.mark.parametrize("which", ["v3_bf16", "v2lite_f32"])
def test_noalloc_decode_matches_mla_decode_twice(mla, which):
    import torch
    w, q_bits = _workload(which)
    g, dt = w.geom, w.dtype
    B, H, L, R = w.batch, g.n_head, g.kv_rank, g.d_rope
    q = to_dev(q_bits, dt)
    cache = to_dev(w.full_cache(), dt)
    table = torch.from_numpy(w.block_table).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    o_ref = poisoned((B, H, L), dt)
    lse_ref = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode(o_ref, q, cache, table, lens, L, R, w.scale, lse_out=lse_ref)
    mla.mla_device_error()
    want = to_f64(o_ref)
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
        check_close(to_f64(o), want, dt, f"noalloc call {call + 1} vs mla_decode")
        assert np.max(np.abs(lse.cpu().numpy() - lse_ref.cpu().numpy())) < 1e-3


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
