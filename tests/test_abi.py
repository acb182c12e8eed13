"""The C ABI as seen from the host, without a GPU: the library loads, exports every
entry point include/mla.h declares, and rejects malformed arguments before it
touches the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mla():
    from mla_latent_kv_11_gb300 import build
    build.build()
    import mla_latent_kv_11_gb300 as m
    return m


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(mla):
    names = declared_functions()
    assert {"mla_absorb_q", "mla_concat_q", "mla_cache_write", "mla_decode", "mla_prefill",
            "mla_v_up"} <= set(names)
    lib = mla.lib()
    for n in names:
        assert hasattr(lib, n), f"libmla.so does not export {n}"
    assert lib.mla_abi_version() == 1
    assert lib.mla_status_string(2) == b"MLA_ERR_UNSUPPORTED"


def _view(shape, strides, data=0x10000):
    from mla_latent_kv_11_gb300 import MlaTensor
    t = MlaTensor()
    t.data = data
    t.rank = len(shape)
    for i, (n, s) in enumerate(zip(shape, strides)):
        t.shape[i] = n
        t.stride[i] = s
    return t


def _contig(shape, data=0x10000):
    strides, acc = [], 1
    for n in reversed(shape):
        strides.insert(0, acc)
        acc *= n
    return _view(shape, strides, data)


def test_bmm_rejects_malformed_operands_without_launching(mla):
    # vllm.cpp BatchedMatmul: inner mismatch, batch mismatch, innermost stride != 1.
    lib = mla.lib()
    o = _contig([2, 3, 4])
    assert lib.mla_absorb_q(1, o, _contig([2, 3, 4]), _contig([2, 5, 4]), None) == mla.MLA_ERR_INVALID_ARG
    assert b"inner" in lib.mla_last_error()
    assert lib.mla_absorb_q(1, o, _contig([2, 3, 4]), _contig([3, 4, 4]), None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_v_up(1, o, _view([2, 3, 4], [24, 8, 2]), _contig([2, 4, 4]), None) == mla.MLA_ERR_INVALID_ARG
    assert b"innermost" in lib.mla_last_error()
    assert lib.mla_v_up(7, o, _contig([2, 3, 4]), _contig([2, 4, 4]), None) == mla.MLA_ERR_INVALID_ARG
    # empty work is fine and launches nothing
    assert lib.mla_absorb_q(1, _contig([2, 0, 4]), _contig([2, 0, 4]), _contig([2, 4, 4]), None) == mla.MLA_OK


def test_concat_and_cache_write_validation(mla):
    lib = mla.lib()
    assert lib.mla_concat_q(1, _contig([4, 8, 10]), _contig([4, 8, 8]), _contig([4, 8, 3]), None) \
        == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_concat_q(1, _contig([4, 8, 10]), _contig([4, 8, 8]), _contig([4, 2, 2]), None) \
        == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_concat_q(1, _contig([0, 8, 10]), _contig([0, 8, 8]), _contig([0, 8, 2]), None) == mla.MLA_OK
    cache = _contig([4, 16, 10])
    assert lib.mla_cache_write(1, cache, _contig([3, 8]), _contig([3, 2]), None, 3, None) \
        == mla.MLA_ERR_INVALID_ARG                                 # null slot mapping
    assert lib.mla_cache_write(1, cache, _contig([3, 8]), _contig([3, 3]), 0x1000, 3, None) \
        == mla.MLA_ERR_INVALID_ARG                                 # entry width mismatch
    assert lib.mla_cache_write(1, cache, _contig([0, 8]), _contig([0, 2]), None, 0, None) == mla.MLA_OK


def test_decode_and_prefill_validation(mla):
    lib = mla.lib()
    B, H, L, R = 2, 16, 512, 64
    q = _contig([B, H, L + R])
    o = _contig([B, H, L])
    cache = _contig([8, 64, L + R])
    ok_args = dict(bt=0x2000, bts=4, mb=4, sl=0x3000)

    def dec(o=o, q=q, cache=cache, L=L, R=R, bt=0x2000, bts=4, mb=4, sl=0x3000, ws=0x4000, wsb=1 << 30):
        return lib.mla_decode(1, o, None, q, cache, bt, bts, mb, sl, L, R, 0.1, 0, ws, wsb, None)

    assert dec(L=500) == mla.MLA_ERR_INVALID_ARG                   # q width != L + R
    assert dec(o=_contig([B, H, L - 1])) == mla.MLA_ERR_INVALID_ARG
    assert dec(cache=_contig([8, 64, 512])) == mla.MLA_ERR_INVALID_ARG
    assert dec(bt=None) == mla.MLA_ERR_INVALID_ARG
    assert dec(bts=2) == mla.MLA_ERR_INVALID_ARG                    # stride < max_blocks
    assert dec(wsb=16) == mla.MLA_ERR_INVALID_ARG                   # workspace too small
    assert b"workspace" in lib.mla_last_error()
    assert dec(ws=0x4001) == mla.MLA_ERR_INVALID_ARG                # unaligned workspace
    assert dec(q=_view([B, H, L + R], [H * (L + R), L + R, 2])) == mla.MLA_ERR_INVALID_ARG
    assert dec(q=_contig([0, H, L + R]), o=_contig([0, H, L])) == mla.MLA_OK
    assert lib.mla_prefill(1, o, None, q, cache, 0x2000, 4, 4, None, 0x3000, 2, 1, L, R, 0.1, None, 0,
                           None) == mla.MLA_ERR_INVALID_ARG         # null cu_seqlens_q
    del ok_args


def test_bounded_wait_check_rejects_bad_limits_without_a_launch(mla):
    # checked on the host before anything reaches the device (stream 0 needs no GPU here)
    for limit in (0, 1_000_001):
        with pytest.raises(mla.MlaError) as e:
            mla.mla_check_bounded_wait(limit, stream=0)
        assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_concat_in_place_without_rope_moves_nothing(mla):
    # nope is q_cat_out's own first L columns (same data pointer and strides) and R = 0: the
    # latent columns are already in place, so the call returns without a launch
    lib = mla.lib()
    T, H, L = 4, 8, 16
    out = _contig([T, H, L])
    nope = _view([T, H, L], [H * L, L, 1], 0x10000)
    rope = _contig([T, H, 0])
    assert lib.mla_concat_q(1, out, nope, rope, None) == mla.MLA_OK
    # the same with the q_cat_out of a rope-carrying layout still validates its widths first
    assert lib.mla_concat_q(1, _contig([T, H, L + 4]), _view([T, H, L], [H * (L + 4), L + 4, 1], 0x10000),
                            _contig([T, H, 3]), None) == mla.MLA_ERR_INVALID_ARG


def test_fused_copy_fp8_sparse_and_vup_validation(mla):
    # argument checks of the later entry points, all on the host before any launch
    lib = mla.lib()
    # concat + cache write in one call: each half is checked as its own call would be
    cache = _contig([4, 16, 10])
    assert lib.mla_concat_q_cache_write(1, _contig([4, 8, 10]), _contig([4, 8, 8]), _contig([4, 8, 3]), cache,
                                        _contig([3, 8]), _contig([3, 2]), 0x1000, 3, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_concat_q_cache_write(1, _contig([4, 8, 10]), _contig([4, 8, 8]), _contig([4, 8, 2]), cache,
                                        _contig([3, 8]), _contig([3, 3]), 0x1000, 3, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_concat_q_cache_write(1, _contig([0, 8, 10]), _contig([0, 8, 8]), _contig([0, 8, 2]), cache,
                                        _contig([0, 8]), _contig([0, 2]), None, 0, None) == mla.MLA_OK
    # e4m3 cache write: the scale is required
    assert lib.mla_cache_write_fp8(1, _contig([4, 16, 10]), _contig([3, 8]), _contig([3, 2]), 0x1000, 3, None,
                                   None) == mla.MLA_ERR_INVALID_ARG
    # sparse ds_mla decode
    B, H = 2, 16
    q, o, c = _contig([B, H, 576]), _contig([B, H, 512]), _contig([8, 64, 656])

    def sparse(o=o, q=q, c=c, idx=0x2000, ids=128, topk=128, ws=0x4000, wsb=1 << 30):
        return lib.mla_decode_sparse_fp8(1, o, None, q, c, idx, ids, topk, 0.1, 0, ws, wsb, None)

    assert sparse(q=_contig([B, H, 512])) == mla.MLA_ERR_INVALID_ARG          # not a 576-wide query
    assert sparse(o=_contig([B, H, 256])) == mla.MLA_ERR_INVALID_ARG
    assert sparse(c=_contig([8, 64, 576])) == mla.MLA_ERR_INVALID_ARG         # not a 656-byte entry
    assert sparse(c=_view([8, 64, 656], [64 * 656, 656, 1], 0x10008)) == mla.MLA_ERR_INVALID_ARG   # unaligned
    assert sparse(topk=-1) == mla.MLA_ERR_INVALID_ARG
    assert sparse(idx=None) == mla.MLA_ERR_INVALID_ARG
    assert sparse(ids=64) == mla.MLA_ERR_INVALID_ARG                           # row stride < top-k
    assert sparse(wsb=16) == mla.MLA_ERR_INVALID_ARG
    assert sparse(q=_contig([0, H, 576]), o=_contig([0, H, 512])) == mla.MLA_OK
    assert lib.mla_decode_sparse_workspace_size(B, H, 128, 0) > lib.mla_decode_workspace_size(B, H, 512, 0)
    # decode with the un-projection: out and w_uv must agree with the decode's shapes
    L, R, V = 512, 64, 128
    qv, cv = _contig([B, H, L + R]), _contig([8, 64, L + R])

    def vup(out=_contig([B, H, V]), w=_contig([H, L, V]), ws=0x4000, wsb=1 << 30):
        return lib.mla_decode_v_up(1, out, None, qv, cv, 0x2000, 4, 4, 0x3000, L, R, 0.1, w, 0, ws, wsb, None)

    assert vup(out=_contig([B, H + 1, V])) == mla.MLA_ERR_INVALID_ARG
    assert vup(w=_contig([H, L, V + 8])) == mla.MLA_ERR_INVALID_ARG
    assert vup(w=_contig([H, L - 1, V])) == mla.MLA_ERR_INVALID_ARG
    assert vup(wsb=1024) == mla.MLA_ERR_INVALID_ARG
    assert b"workspace" in lib.mla_last_error()
    assert lib.mla_decode_v_up_workspace_size(B, H, L, 0) >= lib.mla_decode_workspace_size(B, H, L, 0) + B * H * L * 2


def test_absorb_concat_cache_write_validation(mla):
    # steps 1 to 3 in one call: every part is checked as its own call would be, on the host,
    # before anything is launched (all of these fail or return before touching the device)
    lib = mla.lib()
    T, H, P, L, R = 4, 8, 16, 32, 8
    q_cat = _contig([T, H, L + R])
    q_nope = _view([H, T, P], [P, H * P, 1], 0x20000)     # the transpose of a [T,H,P] buffer
    cache = _contig([4, 16, L + R])

    def call(q_cat=q_cat, q_nope=q_nope, w_uk=_contig([H, P, L]), q_pe=_contig([T, H, R]), cache=cache,
             kv_c=_contig([3, L]), k_pe=_contig([3, R]), slots=0x1000, n=3):
        return lib.mla_absorb_concat_cache_write(1, q_cat, q_nope, w_uk, q_pe, cache, kv_c, k_pe, slots, n, None)

    assert call(w_uk=_contig([H, P, L + R + 1])) == mla.MLA_ERR_INVALID_ARG   # wider than q_cat
    assert call(w_uk=_contig([H, P + 1, L])) == mla.MLA_ERR_INVALID_ARG       # inner dimension
    assert call(w_uk=_contig([H - 1, P, L])) == mla.MLA_ERR_INVALID_ARG       # heads
    assert call(q_nope=_view([H, T + 1, P], [P, H * P, 1], 0x20000)) == mla.MLA_ERR_INVALID_ARG
    assert call(q_pe=_contig([T, H, R + 1])) == mla.MLA_ERR_INVALID_ARG      # L + R != q_cat width
    assert call(k_pe=_contig([3, R + 1])) == mla.MLA_ERR_INVALID_ARG         # cache entry width
    assert call(slots=None) == mla.MLA_ERR_INVALID_ARG
    assert call(n=-1) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_absorb_concat_cache_write(3, q_cat, q_nope, _contig([H, P, L]), _contig([T, H, R]), cache,
                                             _contig([3, L]), _contig([3, R]), 0x1000, 3, None) == \
        mla.MLA_ERR_INVALID_ARG                                                 # no such dtype
    # nothing to do: no tokens, no rows to write
    assert call(q_cat=_contig([0, H, L + R]), q_nope=_view([H, 0, P], [P, H * P, 1], 0x20000),
                q_pe=_contig([0, H, R]), kv_c=_contig([0, L]), k_pe=_contig([0, R]), slots=None, n=0) == mla.MLA_OK
