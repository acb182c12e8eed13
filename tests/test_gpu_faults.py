"""Failure detection on the GPU without a fault: a bounded wait that runs out (on an
mbarrier nothing arrives on) is reported as MLA_ERR_TIMEOUT and leaves the context
usable; out-of-range block ids and sequence lengths in device memory are reported as
MLA_ERR_DEVICE_DATA by both decode paths, are never dereferenced, and do not disturb
the other sequences of the batch."""
import math

import numpy as np
import pytest

import mla_inputs as mi
from helpers import check_close, to_dev, to_f64
from test_gpu_decode import oracle_decode, run_decode

pytestmark = pytest.mark.gpu


def _batch(H, E, lens, page, seed):
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 1
    perm = mi.permutation(seed, nb)
    table = np.zeros((len(lens), max(need) + 1), np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    cache = mi.encode(mi.draw("normal", seed + 1, nb * page * E, 0.5), "bf16").reshape(nb, page, E)
    q = mi.encode(mi.draw("normal", seed + 2, len(lens) * H * E, 0.5), "bf16").reshape(len(lens), H, E)
    return table, cache, q, nb


def test_bounded_wait_runs_out_and_the_context_stays_usable(mla):
    mla.mla_check_bounded_wait(2000)                    # 2 ms on a barrier nobody arrives on
    with pytest.raises(mla.MlaError) as e:
        mla.mla_device_error()
    assert e.value.status == mla.MLA_ERR_TIMEOUT
    mla.mla_device_error()                              # reported once, then cleared
    # the device still works: a small tensor-core decode against the oracle
    H, E, L, R = 128, 576, 512, 64
    lens = [70, 130]
    table, cache, q, _ = _batch(H, E, lens, 64, 501)
    scale = 1.0 / math.sqrt(192)
    o, _ = run_decode(mla, q, cache, table, lens, "bf16", L, R, scale)
    want, _ = oracle_decode(q, cache, table, lens, "bf16", L, R, scale)
    check_close(to_f64(o), want, "bf16", "decode after a timed-out wait")


@pytest.mark.parametrize("H", [128, 16])   # the tensor-core path, the CUDA-core path
def test_decode_bad_block_id_is_reported_and_contained(mla, H):
    import torch
    L, R, page = 512, 64, 64
    E = L + R
    lens = [130, 200, 90]
    table, cache, q, nb = _batch(H, E, lens, page, 511)
    bad = table.copy()
    bad[1, 1] = nb + 9                                  # sequence 1's second page: no such block
    scale = 1.0 / math.sqrt(192)
    o = torch.zeros((len(lens), H, L), dtype=torch.bfloat16, device="cuda")
    mla.mla_decode(o, to_dev(q, "bf16"), to_dev(cache, "bf16"), torch.from_numpy(bad).cuda(),
                   torch.tensor(lens, dtype=torch.int32, device="cuda"), L, R, scale, num_splits=1)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_device_error()
    assert e.value.status == mla.MLA_ERR_DEVICE_DATA
    want, _ = oracle_decode(q, cache, table, lens, "bf16", L, R, scale, ids=[0, 2])
    check_close(to_f64(o)[[0, 2]], want, "bf16", "sequences next to the bad block id")


def test_decode_length_beyond_its_table_is_reported(mla):
    import torch
    H, L, R, page = 128, 512, 64, 64
    E = L + R
    lens = [100, 64]
    table, cache, q, _ = _batch(H, E, lens, page, 521)
    too_long = [lens[0], table.shape[1] * page + 5]    # more rows than the table can address
    scale = 1.0 / math.sqrt(192)
    o = torch.zeros((len(lens), H, L), dtype=torch.bfloat16, device="cuda")
    mla.mla_decode(o, to_dev(q, "bf16"), to_dev(cache, "bf16"), torch.from_numpy(table).cuda(),
                   torch.tensor(too_long, dtype=torch.int32, device="cuda"), L, R, scale)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_device_error()
    assert e.value.status == mla.MLA_ERR_DEVICE_DATA
    want, _ = oracle_decode(q, cache, table, lens, "bf16", L, R, scale, ids=[0])
    check_close(to_f64(o)[[0]], want, "bf16", "sequence next to the over-long one")
