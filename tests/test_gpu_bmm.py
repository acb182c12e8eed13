"""Steps 1 and 5 on the GPU: the absorption bmm's against the float64 oracle, on the
shapes and transposed views of the vllm.cpp BatchedMatmul tests and of the
workloads, NaN-poisoned, and bit-identical from run to run."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc
from helpers import check_close, poisoned, to_dev, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def _gen(dtype, seed, n, scale=1.0, kind="uniform"):
    return mi.encode(mi.draw(kind, seed, n, scale), dtype)


CASES = [  # heads, batch, K, N, what
    (16, 8, 128, 512, "V2-Lite W_UK fold"),
    (16, 8, 512, 128, "V2-Lite W_UV un-projection"),
    (128, 3, 128, 512, "V3 W_UK fold"),
    (16, 1, 512, 128, "single-token decode v-up"),
    (128, 64, 128, 512, "V3 decode batch 64 fold"),
    (128, 64, 512, 128, "V3 decode batch 64 v-up"),
    (3, 5, 12, 20, "small odd shape"),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", CASES, ids=[c[4] for c in CASES])
def test_bmm_contiguous_against_oracle_and_rerun_exact(mla, dtype, case):
    import torch
    H, B, K, N, what = case
    a = _gen(dtype, 1234, H * B * K).reshape(H, B, K)
    w = _gen(dtype, 4321, H * K * N, 1.0 / math.sqrt(K)).reshape(H, K, N)
    da, dw = to_dev(a, dtype), to_dev(w, dtype)
    out = poisoned((H, B, N), dtype)
    fn = mla.mla_absorb_q if N >= K else mla.mla_v_up
    fn(out, da, dw)
    torch.cuda.synchronize()
    want = orc.bmm(mi.decode_f64(a, dtype), mi.decode_f64(w, dtype))
    check_close(to_f64(out), want, dtype, what)
    first = to_host_bits(out)
    for _ in range(3):
        again = poisoned((H, B, N), dtype)
        fn(again, da, dw)
        torch.cuda.synchronize()
        assert np.array_equal(to_host_bits(again), first)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bmm_transposed_in_and_out_views(mla, dtype):
    # the _v_up_proj call site: input a [N,B,L] view of [B,N,L], output a [N,B,V] view of [B,N,V]
    import torch
    H, B, K, N = 16, 5, 512, 128
    raw = _gen(dtype, 2468, B * H * K).reshape(B, H, K)
    w = _gen(dtype, 8642, H * K * N, 1.0 / math.sqrt(K)).reshape(H, K, N)
    draw_t = to_dev(raw, dtype)
    a_view = draw_t.as_strided((H, B, K), (K, H * K, 1))
    out_store = poisoned((B, H, N), dtype)
    out_view = out_store.as_strided((H, B, N), (N, H * N, 1))
    mla.mla_v_up(out_view, a_view, to_dev(w, dtype))
    torch.cuda.synchronize()
    a64 = orc.strided_view(mi.decode_f64(raw, dtype).reshape(-1), 0, (H, B, K), (K, H * K, 1))
    want = orc.bmm(a64, mi.decode_f64(w, dtype))                       # [H,B,N]
    got = to_f64(out_store)                                             # [B,H,N]
    check_close(np.transpose(got, (1, 0, 2)), want, dtype, "transposed views")


def test_bmm_unscaled_pages_relative_bound(mla):
    # The vllm.cpp CUDA bound on unscaled U[-1,1) operands: |got - ref| / max(1e-2, |ref|) < 1e-2.
    import torch
    H, B, K, N = 16, 8, 128, 512
    a = _gen("bf16", 1234, H * B * K).reshape(H, B, K)
    w = _gen("bf16", 4321, H * K * N).reshape(H, K, N)
    out = poisoned((H, B, N), "bf16")
    mla.mla_absorb_q(out, to_dev(a, "bf16"), to_dev(w, "bf16"))
    torch.cuda.synchronize()
    ref = orc.bmm(mi.decode_f64(a, "bf16"), mi.decode_f64(w, "bf16"))
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref) / np.maximum(1e-2, np.abs(ref))) < 1e-2


def test_bmm_prefill_shape_sampled(mla):
    # The NoPE prefill fold: 64 heads x 8192 tokens x 256 -> 512, checked on sampled rows.
    import torch
    H, B, K, N = 64, 8192, 256, 512
    a = _gen("bf16", 11, H * B * K, kind="normal").reshape(H, B, K)
    w = _gen("bf16", 55, H * K * N, 1.0 / math.sqrt(512), kind="normal").reshape(H, K, N)
    out = poisoned((H, B, N), "bf16")
    mla.mla_absorb_q(out, to_dev(a, "bf16"), to_dev(w, "bf16"))
    torch.cuda.synchronize()
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    rows = [0, 1, 127, 128, 4095, 8191]
    want = orc.bmm(mi.decode_f64(a[:, rows], "bf16"), mi.decode_f64(w, "bf16"))
    check_close(got[:, rows], want, "bf16", "prefill fold (sampled rows)")
