"""Shared helpers of the parity tests: device transfer of generator arrays and the
tolerance checks. Expected values always come from ``oracle/``; inputs always
come from ``mla_inputs``."""
from __future__ import annotations

import numpy as np

import mla_inputs as mi

# Tolerances of the path (fp32: max-abs; bf16: max-abs and relative L2, both
# against the float64 oracle); copies and index work are bit-exact.
TOL_F32_MAX_ABS = 1e-4
TOL_BF16_MAX_ABS = 2e-2
TOL_BF16_REL_L2 = 1e-2
BF16_POISON = 0x7FC0


def torch_dtype(dtype: str):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16


def to_dev(arr: np.ndarray, dtype: str, device="cuda"):
    """A generator storage array (float32, or bf16 bits as uint16) as a device tensor."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint16).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_host_bits(t) -> np.ndarray:
    """Device tensor back to its storage representation (float32 or uint16 bits)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return mi.decode_f64(to_host_bits(t), "bf16")
    return t.detach().double().cpu().numpy()


def poisoned(shape, dtype: str, device="cuda"):
    """A NaN-poisoned output buffer: any element a kernel fails to write stays NaN."""
    import torch
    if dtype == "f32":
        return torch.full(shape, float("nan"), dtype=torch.float32, device=device)
    return torch.full(shape, BF16_POISON, dtype=torch.int16, device=device).view(torch.bfloat16)


def check_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "") -> dict:
    """Assert the path's tolerance; return the error figures for reporting."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (unwritten or overflow)"
    diff = np.abs(got - want)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.sqrt(np.sum(want * want)))
    rel_l2 = float(np.sqrt(np.sum(diff * diff)) / denom) if denom > 0 else max_abs
    scaled = max_abs / max(1.0, float(np.abs(want).max()) if want.size else 1.0)
    info = dict(max_abs=max_abs, rel_l2=rel_l2, scaled=scaled)
    if dtype == "f32":
        assert max_abs <= TOL_F32_MAX_ABS, f"{what}: fp32 max-abs {max_abs:.3e} > {TOL_F32_MAX_ABS} {info}"
    else:
        assert max_abs <= TOL_BF16_MAX_ABS, f"{what}: bf16 max-abs {max_abs:.3e} {info}"
        assert rel_l2 <= TOL_BF16_REL_L2, f"{what}: bf16 rel-L2 {rel_l2:.3e} {info}"
    return info
