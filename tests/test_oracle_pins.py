"""Pins for the double-precision oracle, checked on the CPU before any kernel.

Each test ties the oracle to something other than itself: brute-force loop
nests on tiny shapes, the absorption identity (absorbed == naive), closed
forms, invariants (softmax rows sum to one, split-combine == unsplit) and exact
bit-copy semantics. A plausible slip in the oracle (a dropped rope term, a
transposed operand, an off-by-one causal bound, a wrong block index, a wrong
LSE weight) fails at least one of them; ``test_planted_mistakes`` checks that
claim by planting such slips in a copy of the oracle.
"""
import json
import math
import os

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as orc

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _case(H, P, R, V, L, t_q, t_kv, seed):
    """Random MLA inputs at unit scale, weights ~ U[-1,1)/sqrt(L) (memra Case recipe)."""
    ws = 1.0 / math.sqrt(L)
    f = lambda k, n, s=1.0: mi.decode_f64(mi.draw("uniform", seed * 10 + k, n, s), "f32")
    return dict(
        q_nope=f(1, t_q * H * P).reshape(t_q, H, P),
        q_pe=f(2, t_q * H * R).reshape(t_q, H, R),
        c_kv=f(3, t_kv * L).reshape(t_kv, L),
        k_pe=f(4, t_kv * R).reshape(t_kv, R),
        w_uk=f(5, H * P * L, ws).reshape(H, P, L),
        w_uv=f(6, H * L * V, ws).reshape(H, L, V),
    )


def _absorbed_out(c, i, pos, scale):
    """absorb -> attend over rows 0..pos -> v_up for query row i."""
    q_lat = orc.absorb_q(c["q_nope"][i][:, None, :], c["w_uk"])[:, 0, :]
    o_lat, _ = orc.attend_absorbed(q_lat, c["q_pe"][i], c["c_kv"][: pos + 1], c["k_pe"][: pos + 1], scale)
    return orc.v_up(o_lat[:, None, :], c["w_uv"])[:, 0, :]


# --------------------------------------------------------------------------- bmm

def _loop_bmm(a_flat, a_off, a_str, b_flat, b_off, b_str, G, M, K, N):
    out = np.zeros((G, M, N))
    for g in range(G):
        for m in range(M):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += (a_flat[a_off + g * a_str[0] + m * a_str[1] + k * a_str[2]]
                            * b_flat[b_off + g * b_str[0] + k * b_str[1] + n * b_str[2]])
                out[g, m, n] = acc
    return out


def test_bmm_matches_loop_nest_on_transposed_views():
    # The up-projection call site: operand is a [N,B,K] view of a [B,N,K] buffer and
    # the output a [N,B,V] view of [B,N,V] (vllm.cpp BatchedMatmul transposed-view case).
    n_heads, batch, kdim, ndim = 5, 6, 9, 4
    src = mi.decode_f64(mi.uniform(33, batch * n_heads * kdim), "f32")
    w = mi.decode_f64(mi.uniform(44, n_heads * kdim * ndim), "f32")
    a = orc.strided_view(src, 0, (n_heads, batch, kdim), (kdim, n_heads * kdim, 1))
    b = orc.strided_view(w, 0, (n_heads, kdim, ndim), (kdim * ndim, ndim, 1))
    got = orc.bmm(a, b)
    want = _loop_bmm(src, 0, (kdim, n_heads * kdim, 1), w, 0, (kdim * ndim, ndim, 1),
                     n_heads, batch, kdim, ndim)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    # element (h, b, j) of the result lands at (b * N + h) * V + j of the [B,N,V] buffer
    flat_out = np.zeros(batch * n_heads * ndim)
    view_idx = (np.arange(batch)[None, :, None] * n_heads + np.arange(n_heads)[:, None, None]) * ndim \
        + np.arange(ndim)[None, None, :]
    flat_out[view_idx] = got
    assert flat_out[(2 * n_heads + 3) * ndim + 1] == got[3, 2, 1]


def test_bmm_identity_weight_is_identity():
    H, B, L = 3, 4, 8
    x = mi.decode_f64(mi.uniform(5, H * B * L), "f32").reshape(H, B, L)
    eye = np.broadcast_to(np.eye(L), (H, L, L))
    assert np.array_equal(orc.bmm(x, eye), x)


def test_bmm_nonsquare_orientation():
    # A transposed weight would still be the identity above; a rectangular weight with a
    # single 1 at (k0, n0) must move column k0 of the operand to column n0.
    H, B, K, N = 2, 3, 5, 7
    x = mi.decode_f64(mi.uniform(6, H * B * K), "f32").reshape(H, B, K)
    w = np.zeros((H, K, N))
    w[:, 4, 1] = 1.0
    out = orc.bmm(x, w)
    assert np.array_equal(out[:, :, 1], x[:, :, 4])
    assert np.count_nonzero(out[:, :, [0, 2, 3, 4, 5, 6]]) == 0


# --------------------------------------------------------------------------- concat

def test_concat_is_a_bit_copy_including_nan_payloads_and_negative_zero():
    T, H, L, R = 3, 4, 6, 2
    nope = mi.to_bf16_bits(mi.normal(1, T * H * L)).reshape(T, H, L)
    rope = mi.to_bf16_bits(mi.normal(2, T * H * R)).reshape(T, H, R)
    nope[0, 0, 0] = 0x8000      # -0
    nope[1, 2, 3] = 0x7FC1      # NaN with a payload
    rope[2, 3, 1] = 0xFF81      # negative NaN with a payload
    out = orc.concat_q(nope, rope)
    for t in range(T):
        for h in range(H):
            assert list(out[t, h, :L]) == list(nope[t, h])
            assert list(out[t, h, L:]) == list(rope[t, h])
    assert out[0, 0, 0] == 0x8000 and out[1, 2, 3] == 0x7FC1 and out[2, 3, L + 1] == 0xFF81


def test_concat_transposed_nope_and_broadcast_rope():
    f = FACTS["concat_cases"]
    T, H, L, R = f["transposed_nope"]["tokens"], f["transposed_nope"]["heads"], 32, 8
    raw = mi.to_bf16_bits(mi.uniform(77, H * T * L))             # [H, T, L] storage
    nope = orc.strided_view(raw, 0, (T, H, L), (L, T * L, 1))    # its [T, H, L] transpose
    rope1 = mi.to_bf16_bits(mi.uniform(88, T * R)).reshape(T, 1, R)
    out = orc.concat_q(np.ascontiguousarray(nope), rope1)
    for t in range(T):
        for h in range(H):
            assert np.array_equal(out[t, h, :L], raw[(h * T + t) * L:(h * T + t + 1) * L])
            assert np.array_equal(out[t, h, L:], rope1[t, 0])


# --------------------------------------------------------------------------- cache write

def test_cache_write_view_equals_contiguous_and_does_not_bleed():
    f = FACTS["unified_slot_write"]
    nb, page, L, R = 4, 8, 16, 4
    E, n_layers, layer = L + R, f["n_layers"], f["layer"]
    ntok = 20
    kv_c = mi.to_bf16_bits(mi.normal(1, ntok * L)).reshape(ntok, L)
    k_pe = mi.to_bf16_bits(mi.normal(2, ntok * R)).reshape(ntok, R)
    slots = mi.permutation(3, nb * page)[:ntok].copy()
    padded = int(slots[5])
    slots[5] = -1                                               # padding: writes nothing
    ref = orc.cache_write(np.zeros(nb * page * E, np.uint16), 0, nb, page, (page * E, E, 1),
                          kv_c, k_pe, slots)
    unified = np.full(nb * n_layers * page * E, 0x1234, np.uint16)   # sentinel everywhere
    after = orc.cache_write(unified, layer * page * E, nb, page, (n_layers * page * E, E, 1),
                            kv_c, k_pe, slots)
    view = orc.strided_view(after, layer * page * E, (nb, page, E), (n_layers * page * E, E, 1))
    ref3 = ref.reshape(nb, page, E)
    written = np.zeros((nb, page), bool)
    for i, s in enumerate(slots):
        if s >= 0:
            written[s // page, s % page] = True
            assert np.array_equal(view[s // page, s % page, :L], kv_c[i])
            assert np.array_equal(view[s // page, s % page, L:], k_pe[i])
    assert np.array_equal(view[written], ref3[written])
    assert np.all(view[~written] == 0x1234)                     # untouched rows keep their bits
    blocks = after.reshape(nb, n_layers, page * E)
    assert np.all(blocks[:, 0] == 0x1234) and np.all(blocks[:, 2] == 0x1234)   # no bleed
    assert not written[padded // page, padded % page]
    assert np.all(view[padded // page, padded % page] == 0x1234)


def test_paged_rows_follow_the_block_table():
    page, E, nb = 4, 3, 6
    storage = np.arange(nb * page * E, dtype=np.float64)
    table = np.array([5, 2, 0], np.int64)
    rows = orc.paged_rows(storage, 0, page, (page * E, E, 1), E, table, 10)
    for t in range(10):
        blk = table[t // page]
        assert np.array_equal(rows[t], storage[(blk * page + t % page) * E:(blk * page + t % page + 1) * E])


# --------------------------------------------------------------------------- attention

@pytest.mark.parametrize("dims_i", [0, 1, 2])
def test_absorption_identity_small_dims(dims_i):
    f = FACTS["small_dims"]
    H, P, R, V, L = f["dims"][dims_i]
    for seed in f["seeds"]:
        for t_q, t_kv in f["shapes_tq_tkv"]:
            c = _case(H, P, R, V, L, t_q, t_kv, seed + dims_i)
            scale = 1.0 / math.sqrt(P + R)
            for i in range(t_q):
                pos = t_kv - t_q + i
                got = _absorbed_out(c, i, pos, scale)
                want = orc.attend_naive(c["q_nope"][i], c["q_pe"][i], c["c_kv"][: pos + 1],
                                        c["k_pe"][: pos + 1], c["w_uk"], c["w_uv"], scale)
                assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_absorption_identity_v2_lite_decode():
    g = mi.V2_LITE
    c = _case(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank, 1, 64, 99)
    scale = 1.0 / math.sqrt(192)
    got = _absorbed_out(c, 0, 63, scale)
    want = orc.attend_naive(c["q_nope"][0], c["q_pe"][0], c["c_kv"], c["k_pe"],
                            c["w_uk"], c["w_uv"], scale)
    assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_brute_force_tiny():
    H, P, R, V, L = 2, 3, 2, 3, 4
    for T in range(1, 6):
        c = _case(H, P, R, V, L, 1, T, 500 + T)
        # scale the scores up so the softmax is far from uniform
        scale = 2.5
        bf = np.array(orc.brute_force_attention(c["q_nope"][0].tolist(), c["q_pe"][0].tolist(),
                                                c["c_kv"].tolist(), c["k_pe"].tolist(),
                                                c["w_uk"].tolist(), c["w_uv"].tolist(), scale))
        assert np.max(np.abs(_absorbed_out(c, 0, T - 1, scale) - bf)) < 1e-13
        naive = orc.attend_naive(c["q_nope"][0], c["q_pe"][0], c["c_kv"], c["k_pe"],
                                 c["w_uk"], c["w_uv"], scale)
        assert np.max(np.abs(naive - bf)) < 1e-13


def test_softmax_rows_sum_to_one():
    s = mi.decode_f64(mi.normal(9, 7 * 33), "f32").reshape(7, 33) * 20
    p = orc.softmax_rows(s)
    assert np.all(p >= 0) and np.max(np.abs(p.sum(axis=1) - 1)) < 1e-14
    # and the absorbed attention's weights are exactly those: o_lat of one-hot rows
    H, T = 3, 5
    c_kv = np.eye(T)                      # row t is e_t, so o_lat[h] = p[h, :]
    q_lat = mi.decode_f64(mi.normal(10, H * T), "f32").reshape(H, T)
    o, lse = orc.attend_absorbed(q_lat, np.zeros((H, 0)), c_kv, np.zeros((T, 0)), 1.3)
    np.testing.assert_allclose(o, orc.softmax_rows(1.3 * q_lat), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, np.log(np.exp(1.3 * q_lat).sum(axis=1)), rtol=1e-14)


@pytest.mark.parametrize("k", [1, 2, 3, 7, "len"])
def test_split_combine_equals_unsplit(k):
    H, L, R, T = 4, 16, 4, 23
    q_lat = mi.decode_f64(mi.normal(1, H * L), "f32").reshape(H, L)
    q_pe = mi.decode_f64(mi.normal(2, H * R), "f32").reshape(H, R)
    c_kv = mi.decode_f64(mi.normal(3, T * L), "f32").reshape(T, L)
    k_pe = mi.decode_f64(mi.normal(4, T * R), "f32").reshape(T, R)
    o_ref, lse_ref = orc.attend_absorbed(q_lat, q_pe, c_kv, k_pe, 0.4)
    kk = T if k == "len" else k
    bounds = sorted(set([0, T] + [round(i * T / kk) for i in range(1, kk)]))
    bounds = [0, 0] + bounds + [T]            # empty chunks at both ends
    o, lse = orc.attend_split(q_lat, q_pe, c_kv, k_pe, 0.4, bounds)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12


def test_combine_all_empty_is_zero_minus_inf():
    H, L = 2, 3
    empty = (np.zeros((H, L)), np.full(H, -np.inf))
    o, lse = orc.combine([empty, empty])
    assert np.all(o == 0) and np.all(lse == -np.inf)
    o, lse = orc.attend_absorbed(np.ones((H, L)), np.ones((H, 1)), np.zeros((0, L)), np.zeros((0, 1)), 1.0)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_closed_forms():
    H, L, R, T = 3, 8, 2, 9
    q_lat = mi.decode_f64(mi.normal(1, H * L), "f32").reshape(H, L)
    q_pe = mi.decode_f64(mi.normal(2, H * R), "f32").reshape(H, R)
    c_kv = mi.decode_f64(mi.normal(3, T * L), "f32").reshape(T, L)
    k_pe = mi.decode_f64(mi.normal(4, T * R), "f32").reshape(T, R)
    # one row: o_lat is that row, lse is its score
    o, lse = orc.attend_absorbed(q_lat, q_pe, c_kv[:1], k_pe[:1], 0.7)
    assert np.array_equal(o, np.broadcast_to(c_kv[0], (H, L)))
    np.testing.assert_allclose(lse, 0.7 * (q_lat @ c_kv[0] + q_pe @ k_pe[0]), rtol=1e-15)
    # scale 0: uniform weights, o_lat is the mean row and lse = ln T
    o, lse = orc.attend_absorbed(q_lat, q_pe, c_kv, k_pe, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(c_kv.mean(axis=0), (H, L)), atol=1e-15)
    np.testing.assert_allclose(lse, math.log(T), rtol=1e-15)
    # identical keys: uniform weights too
    same_c = np.broadcast_to(c_kv[4], (T, L)).copy()
    same_k = np.broadcast_to(k_pe[4], (T, R)).copy()
    o, _ = orc.attend_absorbed(q_lat, q_pe, same_c, same_k, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(c_kv[4], (H, L)), atol=1e-15)
    # one dominant score through the rope term alone: that row wins outright
    kp = np.zeros((T, R))
    kp[6, 0] = 1e3
    qp = np.zeros((H, R))
    qp[:, 0] = 1.0
    o, _ = orc.attend_absorbed(np.zeros((H, L)), qp, c_kv, kp, 1.0)
    assert np.array_equal(o, np.broadcast_to(c_kv[6], (H, L)))


def _paged_case(H, L, R, page, lens, seed):
    B = len(lens)
    need = [(n + page - 1) // page for n in lens]
    nb = sum(need) + 2
    perm = mi.permutation(seed, nb)
    table = np.zeros((B, max(need)), np.int64)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    E = L + R
    storage = mi.decode_f64(mi.normal(seed + 1, nb * page * E), "f32")
    return storage, table, E


def test_decode_reads_through_block_table_and_view():
    H, L, R, page = 4, 16, 4, 8
    lens = [13, 1, 24, 0]
    storage, table, E = _paged_case(H, L, R, page, lens, 40)
    q = mi.decode_f64(mi.normal(41, len(lens) * H * E), "f32").reshape(len(lens), H, E)
    o, lse = orc.decode(q, storage, 0, page, (page * E, E, 1), L, R, table, np.array(lens), 0.3)
    for b, n in enumerate(lens):
        rows = np.array([storage[(table[b, t // page] * page + t % page) * E:
                                 (table[b, t // page] * page + t % page + 1) * E] for t in range(n)]).reshape(n, E)
        o_b, lse_b = orc.attend_absorbed(q[b, :, :L], q[b, :, L:], rows[:, :L], rows[:, L:], 0.3)
        assert np.array_equal(o[b], o_b) and np.array_equal(lse[b], lse_b)
    assert np.all(o[3] == 0) and np.all(lse[3] == -np.inf)
    # the same cache seen through a layer view of a 3-layer unified buffer gives the same bits
    nb = storage.size // (page * E)
    unified = np.full(nb * 3 * page * E, 7.0)
    unified.reshape(nb, 3, page * E)[:, 1] = storage.reshape(nb, page * E)
    o2, lse2 = orc.decode(q, unified, page * E, page, (3 * page * E, E, 1), L, R, table,
                          np.array(lens), 0.3)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_prefill_query_zero_and_prefill_decode_consistency():
    H, L, R, page = 3, 8, 2, 4
    kv_lens = [9, 6]
    q_lens = [9, 3]                    # pure prefill and a suffix of a populated cache
    storage, table, E = _paged_case(H, L, R, page, kv_lens, 60)
    T = sum(q_lens)
    q = mi.decode_f64(mi.normal(61, T * H * E), "f32").reshape(T, H, E) * 3
    cu = np.array([0, 9, 12])
    o, lse = orc.prefill(q, cu, np.array(kv_lens), storage, 0, page, (page * E, E, 1), L, R, table, 0.5)
    rows0 = orc.paged_rows(storage, 0, page, (page * E, E, 1), E, table[0], 1)
    assert np.array_equal(o[0], np.broadcast_to(rows0[0, :L], (H, L)))      # query 0 sees row 0
    for r in range(T):
        b = 0 if r < 9 else 1
        i = r - cu[b]
        pos = kv_lens[b] - q_lens[b] + i
        od, ld = orc.decode(q[r][None], storage, 0, page, (page * E, E, 1), L, R,
                            table[b:b + 1], np.array([pos + 1]), 0.5)
        assert np.array_equal(o[r], od[0]) and np.array_equal(lse[r], ld[0])


def test_prefill_rows_before_the_first_cached_row_see_nothing():
    # More queries than cached rows: queries at positions below 0 attend no row (o = 0,
    # lse = -inf, as for an empty sequence); the others equal decode over their prefix.
    H, L, R, page = 2, 8, 2, 4
    kv_lens, q_lens = [3, 0], [5, 2]
    storage, table, E = _paged_case(H, L, R, page, [3, 1], 62)
    T = sum(q_lens)
    q = mi.decode_f64(mi.normal(63, T * H * E), "f32").reshape(T, H, E)
    cu = np.array([0, 5, 7])
    o, lse = orc.prefill(q, cu, np.array(kv_lens), storage, 0, page, (page * E, E, 1), L, R, table, 0.5)
    for r in range(T):
        b = 0 if r < 5 else 1
        pos = kv_lens[b] - q_lens[b] + (r - cu[b])
        if pos < 0:
            assert np.all(o[r] == 0) and np.all(lse[r] == -np.inf)
        else:
            od, ld = orc.decode(q[r][None], storage, 0, page, (page * E, E, 1), L, R,
                                table[b:b + 1], np.array([pos + 1]), 0.5)
            assert np.array_equal(o[r], od[0]) and np.array_equal(lse[r], ld[0])
    assert sum(kv_lens[b] - q_lens[b] + i < 0 for b in range(2) for i in range(q_lens[b])) == 4


def test_stepwise_decode_through_appended_cache():
    # Rows are appended one step at a time; each step equals a full recompute (memra gate 2).
    H, P, R, V, L = 4, 24, 8, 32, 64
    f = FACTS["stepwise_decode"]
    total = f["prefill"] + f["steps"]
    c = _case(H, P, R, V, L, total, total, 77)
    page, E = 4, L + R
    table = np.array([[2, 0, 1]], np.int64)
    storage = np.zeros(3 * page * E)
    slot_of = lambda t: table[0, t // page] * page + t % page
    storage = orc.cache_write(storage, 0, 3, page, (page * E, E, 1), c["c_kv"][:f["prefill"]],
                              c["k_pe"][:f["prefill"]], np.array([slot_of(t) for t in range(f["prefill"])]))
    scale = 1.0 / math.sqrt(P + R)
    for step in range(f["steps"]):
        pos = f["prefill"] + step
        out, _, _, storage = orc.decode_step(
            c["q_nope"][pos][None], c["q_pe"][pos][None], c["w_uk"], c["w_uv"],
            c["c_kv"][pos][None], c["k_pe"][pos][None], np.array([slot_of(pos)]),
            storage, 0, page, (page * E, E, 1), table, np.array([pos + 1]), scale)
        want = orc.attend_naive(c["q_nope"][pos], c["q_pe"][pos], c["c_kv"][: pos + 1],
                                c["k_pe"][: pos + 1], c["w_uk"], c["w_uv"], scale)
        assert np.max(np.abs(out[0] - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


# --------------------------------------------------------------------------- the pins bite

def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible slips in the oracle (on the CPU) and check a pin fails each time."""
    H, P, R, V, L, T = 2, 3, 2, 3, 4, 5
    c = _case(H, P, R, V, L, 1, T, 505)
    bf = np.array(orc.brute_force_attention(c["q_nope"][0].tolist(), c["q_pe"][0].tolist(),
                                            c["c_kv"].tolist(), c["k_pe"].tolist(),
                                            c["w_uk"].tolist(), c["w_uv"].tolist(), 2.5))
    good = orc.attend_absorbed

    def dropped_rope(q_lat, q_pe, c_kv, k_pe, scale):
        return good(q_lat, q_pe * 0, c_kv, k_pe, scale)

    def no_scale(q_lat, q_pe, c_kv, k_pe, scale):
        return good(q_lat, q_pe, c_kv, k_pe, 1.0)

    def off_by_one(q_lat, q_pe, c_kv, k_pe, scale):
        return good(q_lat, q_pe, c_kv[:-1] if len(c_kv) > 1 else c_kv, k_pe[:-1] if len(k_pe) > 1 else k_pe, scale)

    for bad in (dropped_rope, no_scale, off_by_one):
        monkeypatch.setattr(orc, "attend_absorbed", bad)
        assert np.max(np.abs(_absorbed_out(c, 0, T - 1, 2.5) - bf)) > 1e-6, bad.__name__
    monkeypatch.setattr(orc, "attend_absorbed", good)

    # transposed weight: a square-per-head but non-symmetric W_UK fold must differ
    good_bmm = orc.bmm
    monkeypatch.setattr(orc, "bmm", lambda a, b: good_bmm(a, np.swapaxes(b, 1, 2)) if a.shape[2] == b.shape[2] else good_bmm(a, b))
    cc = _case(2, 4, 2, 4, 4, 1, T, 506)
    bf2 = np.array(orc.brute_force_attention(cc["q_nope"][0].tolist(), cc["q_pe"][0].tolist(),
                                             cc["c_kv"].tolist(), cc["k_pe"].tolist(),
                                             cc["w_uk"].tolist(), cc["w_uv"].tolist(), 2.5))
    assert np.max(np.abs(_absorbed_out(cc, 0, T - 1, 2.5) - bf2)) > 1e-6
    monkeypatch.setattr(orc, "bmm", good_bmm)

    # a wrong LSE weight in the combine (forgetting to subtract the max) is harmless
    # mathematically but a dropped exp is not: check the split pin catches it
    good_combine = orc.combine

    def linear_combine(parts):
        lses = np.stack([p[1] for p in parts])
        os_ = np.stack([p[0] for p in parts])
        w = np.where(np.isfinite(lses), lses - lses.min(), 0.0)
        return np.einsum("kh,khl->hl", w, os_) / w.sum(axis=0)[:, None], lses.max(axis=0)

    monkeypatch.setattr(orc, "combine", linear_combine)
    q_lat = mi.decode_f64(mi.normal(1, 4 * 16), "f32").reshape(4, 16)
    q_pe = mi.decode_f64(mi.normal(2, 4 * 4), "f32").reshape(4, 4)
    c_kv = mi.decode_f64(mi.normal(3, 23 * 16), "f32").reshape(23, 16)
    k_pe = mi.decode_f64(mi.normal(4, 23 * 4), "f32").reshape(23, 4)
    o_ref, _ = good(q_lat, q_pe, c_kv, k_pe, 0.4)
    o, _ = orc.attend_split(q_lat, q_pe, c_kv, k_pe, 0.4, [0, 7, 15, 23])
    assert np.max(np.abs(o - o_ref)) > 1e-6
    monkeypatch.setattr(orc, "combine", good_combine)

    # a block-table slip (using the logical block number) breaks the view pin
    good_rows = orc.paged_rows

    def ignore_table(storage, offset, page, strides, entry, block_row, length):
        return good_rows(storage, offset, page, strides, entry, np.arange(len(block_row)), length)

    storage, table, E = _paged_case(2, 8, 2, 4, [10], 70)
    o_good, _ = orc.decode(np.ones((1, 2, E)), storage, 0, 4, (4 * E, E, 1), 8, 2, table, np.array([10]), 0.5)
    monkeypatch.setattr(orc, "paged_rows", ignore_table)
    o_bad, _ = orc.decode(np.ones((1, 2, E)), storage, 0, 4, (4 * E, E, 1), 8, 2, table, np.array([10]), 0.5)
    assert not np.array_equal(o_good, o_bad)


# --------------------------------------------------------------------------- the recipes

def test_generator_is_the_pages_lcg():
    f = FACTS["lcg"]
    s, out = 1234, []
    for _ in range(64):
        s = (s * f["a"] + f["c"]) & 0xFFFFFFFF
        out.append((s >> f["shift"]) / f["denominator"] * 2.0 - 1.0)
    assert np.array_equal(mi.uniform(1234, 64).astype(np.float64), np.array(out))


def test_workload_geometry_matches_the_pages():
    f = FACTS
    g = mi.V2_LITE
    assert (g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank) == tuple(
        f["v2_lite"][k] for k in ("n_head", "d_nope", "d_rope", "d_v", "kv_rank"))
    assert mi.V3.n_head == f["v3"]["n_head"] and mi.V3.entry == f["dense_decode_view"]["head_dim"]
    n = mi.NOPE_64
    assert (n.n_head, n.d_nope, n.d_rope, n.d_v, n.kv_rank) == tuple(
        f["nope_64"][k] for k in ("n_head", "d_nope", "d_rope", "d_v", "kv_rank"))
    u = f["unified_slot_write"]
    assert u["n_layers"] * u["page"] * u["entry"] == u["stride0"]
    assert u["layer"] * u["page"] * u["entry"] == u["offset"]
    w = mi.write_concat_workload()
    assert w.kv_c.shape == (u["ntok"], u["kv_lora_rank"]) and w.k_pe.shape == (u["ntok"], u["pe"])
    assert len(set(w.slots.tolist())) == u["ntok"] and w.slots.max() < u["num_blocks"] * u["page"]


# ---------------------------------------------------------------------------- fp8 (e4m3) cache

def test_e4m3_values_are_the_formats():
    # 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals at exponent 0, no
    # infinities, NaN only where every exponent and mantissa bit is set
    v = orc.e4m3_value(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x30] == 0.5
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0            # largest finite
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9     # smallest normal, smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9                          # largest subnormal
    assert v[0x00] == 0.0 and np.signbit(v[0x80]) and v[0x80] == 0.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.sum(np.isnan(v)) == 2
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                          # codes 0..126 are ascending


def test_e4m3_round_trip_and_torch_agree():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    v = orc.e4m3_value(codes)
    fin = ~np.isnan(v)
    assert np.array_equal(orc.e4m3_code(v[fin].astype(np.float32)), codes[fin])   # exact values
    x = (mi.draw("normal", 7001, 200000) * 60.0).astype(np.float32)
    x = x[np.abs(x) < 448]                                    # torch's cast does not saturate
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_code(x), t)


def test_e4m3_ties_to_even_and_saturation():
    c = orc.e4m3_code(np.array([1 + 1 / 16, 1 + 3 / 16, 2.0 ** -10, 3 * 2.0 ** -10,
                                449.0, 464.0, 1e6, -1e6, -0.0, np.nan], np.float32))
    assert c.tolist() == [0x38, 0x3A, 0x00, 0x02, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x7F]


def test_fp8_cache_write_is_the_scaled_code_and_does_not_bleed():
    T, L, R, page, nb, layers, layer = 9, 16, 8, 4, 6, 3, 1
    E = L + R
    kv = mi.decode_f64(mi.draw("normal", 7011, T * L, 3.0), "f32").reshape(T, L)
    kp = mi.decode_f64(mi.draw("normal", 7012, T * R, 3.0), "f32").reshape(T, R)
    slots = np.array([5, -1, 0, 23, 7, 12, -3, 1, 18], np.int64)
    storage = mi.permutation(7013, nb * layers * page * E).astype(np.uint8)   # sentinel bytes
    strides = (layers * page * E, E, 1)
    out = orc.cache_write_fp8(storage, layer * page * E, nb, page, strides, kv, kp, slots, 0.5)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        base = layer * page * E + (s // page) * strides[0] + (s % page) * E
        row = np.concatenate([kv[i], kp[i]]).astype(np.float32) / np.float32(0.5)
        assert np.array_equal(out[base:base + E], orc.e4m3_code(row))
        assert np.allclose(orc.e4m3_value(out[base:base + E]) * 0.5,
                           np.concatenate([kv[i], kp[i]]), rtol=2 ** -4, atol=2 ** -10)
    written = np.zeros(storage.size, bool)
    for s in slots[slots >= 0]:
        base = layer * page * E + (s // page) * strides[0] + (s % page) * E
        written[base:base + E] = True
    assert np.array_equal(out[~written], storage[~written])   # no bleed


def test_fp8_decode_equals_decode_on_the_same_values():
    # a cache whose values are exactly e4m3-representable, stored once as codes and once as
    # float64 values: the fp8 decode with descale 1 is the plain decode of those values; an
    # exact power-of-two descale_k scales the cache, descale_q scales the scores like the
    # softmax scale
    H, L, R, page, lens = 4, 8, 4, 4, [5, 9, 1]
    E = L + R
    nb = sum((n + page - 1) // page for n in lens) + 1
    codes = mi.permutation(7021, 256 * ((nb * page * E) // 256 + 1))[: nb * page * E].astype(np.uint8)
    codes = np.where((codes & 0x7F) == 0x7F, 0x38, codes).astype(np.uint8)       # no NaN codes
    codes = np.where((codes >> 3 & 0xF) >= 11, codes & 0x87, codes).astype(np.uint8)   # keep |v| < 16
    vals = orc.e4m3_value(codes)
    perm = mi.permutation(7022, nb)
    need = [(n + page - 1) // page for n in lens]
    table = np.zeros((len(lens), max(need)), np.int64)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    q = mi.decode_f64(mi.draw("normal", 7023, len(lens) * H * E), "f32").reshape(len(lens), H, E)
    args = (0, page, (page * E, E, 1), L, R, table, np.array(lens))
    o1, l1 = orc.decode_fp8(q, codes, *args, 0.3, 1.0, 1.0)
    o0, l0 = orc.decode(q, vals, *args, 0.3)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)
    o4, _ = orc.decode_fp8(q, codes, *args, 0.3, 1.0, 4.0)
    o4b, _ = orc.decode(q, vals * 4.0, *args, 0.3)
    assert np.allclose(o4, o4b, rtol=1e-13, atol=1e-13)
    o2, l2 = orc.decode_fp8(q, codes, *args, 0.3, 2.0, 1.0)
    o2b, l2b = orc.decode(q, vals, *args, 0.6)
    assert np.allclose(o2, o2b, rtol=1e-13, atol=1e-13) and np.allclose(l2, l2b, rtol=1e-13)


def test_fp8_planted_mistakes_are_caught(monkeypatch):
    # a wrong exponent bias, rounding by truncation, or a dropped descale must fail a pin
    good_value = orc.e4m3_value
    monkeypatch.setattr(orc, "e4m3_value", lambda c: good_value(c) * 2.0)   # bias off by one
    with pytest.raises(AssertionError):
        test_e4m3_values_are_the_formats()
    monkeypatch.setattr(orc, "e4m3_value", good_value)
    good_code = orc.e4m3_code

    def truncating(x):
        x = np.asarray(x, np.float32)
        c = good_code(x)
        over = np.abs(orc.e4m3_value(c)) > np.abs(x.astype(np.float64))
        return np.where(over & ((c & 0x7F) > 0), c - 1, c).astype(np.uint8)

    monkeypatch.setattr(orc, "e4m3_code", truncating)
    with pytest.raises(AssertionError):
        test_e4m3_round_trip_and_torch_agree()
    monkeypatch.setattr(orc, "e4m3_code", good_code)
    good_dec = orc.decode_fp8
    monkeypatch.setattr(orc, "decode_fp8", lambda *a, **k: good_dec(*a[:10], 1.0, 1.0, *a[12:], **k))
    with pytest.raises(AssertionError):
        test_fp8_decode_equals_decode_on_the_same_values()
    monkeypatch.setattr(orc, "decode_fp8", good_dec)


# ---------------------------------------------------------------------------- fp8 ds_mla sparse decode

def _ds_mla_values_by_library(entries):
    """The entries' values by other routes: torch's e4m3 and bf16 decoders, numpy's
    little-endian float32 reader, and an explicit loop over the four 128-column groups."""
    import torch
    e = np.ascontiguousarray(entries, dtype=np.uint8).reshape(-1, 656)
    n = e.shape[0]
    codes = torch.from_numpy(e[:, :512].copy()).view(torch.float8_e4m3fn).double().numpy()
    scales = np.frombuffer(e[:, 512:528].tobytes(), dtype="<f4").reshape(n, 4).astype(np.float64)
    rope = torch.from_numpy(e[:, 528:].copy()).view(torch.bfloat16).double().numpy()
    c_kv = codes.copy()
    for g in range(4):
        c_kv[:, 128 * g:128 * (g + 1)] *= scales[:, g:g + 1]
    return c_kv, rope


def test_ds_mla_entry_values_follow_the_byte_layout():
    ent = mi.ds_mla_entries(8101, 40)
    c_kv, k_pe = orc.ds_mla_values(ent)
    want_c, want_r = _ds_mla_values_by_library(ent)
    assert c_kv.shape == (40, 512) and k_pe.shape == (40, 64)
    assert np.array_equal(c_kv, want_c) and np.array_equal(k_pe, want_r)
    # a hand-built entry: code 0x38 (1.0) in column 130 (group 1, scale 0.25), code 0xC0
    # (-2.0) in column 511 (group 3, scale 3.0), rope column 5 = bf16 0x4040 (3.0)
    e = np.zeros((1, 656), np.uint8)
    e[0, 130], e[0, 511] = 0x38, 0xC0
    e[0, 512:528] = np.array([1.0, 0.25, 1.0, 3.0], "<f4").view(np.uint8)
    e[0, 528 + 10], e[0, 528 + 11] = 0x40, 0x40
    c, r = orc.ds_mla_values(e)
    assert c[0, 130] == 0.25 and c[0, 511] == -6.0 and np.count_nonzero(c) == 2
    assert r[0, 5] == 3.0 and np.count_nonzero(r) == 1


def _sparse_small(pattern, unit_scales, batch=3, heads=4, topk=96, num_blocks=12, page=16, seed_cfg=7):
    w = mi.sparse_decode_workload(batch=batch, heads=heads, topk=topk, num_blocks=num_blocks, page=page,
                                  pattern=pattern, unit_scales=unit_scales, config_index=seed_cfg)
    q = mi.decode_f64(w.q_cat, "bf16")
    return w, q


@pytest.mark.parametrize("pattern,unit_scales", [("blocks", True), ("scattered", False)])
def test_sparse_decode_equals_paged_decode_of_the_listed_rows(pattern, unit_scales):
    # page-1 paged decode whose block table is the list of valid slots, over float64 values of
    # the contiguous layer decoded by the library routes
    w, q = _sparse_small(pattern, unit_scales)
    layer = w.storage.reshape(w.num_blocks, w.n_layers, w.page, 656)[:, w.layer].reshape(-1, 656)
    c_kv, k_pe = _ds_mla_values_by_library(layer)
    values = np.concatenate([c_kv, k_pe], axis=1).reshape(-1)
    valid = [w.indices[b][w.indices[b] >= 0].astype(np.int64) for b in range(q.shape[0])]
    table = np.zeros((q.shape[0], max(1, max(v.size for v in valid))), np.int64)
    for b, v in enumerate(valid):
        table[b, :v.size] = v
    lens = np.array([v.size for v in valid])
    o_d, l_d = orc.decode(q, values, 0, 1, (576, 576, 1), 512, 64, table, lens, w.scale)
    o_s, l_s = orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides,
                                        w.indices, w.scale)
    assert np.array_equal(o_s, o_d) and np.array_equal(l_s, l_d)
    assert np.isfinite(o_s).all() or (lens == 0).any()


def test_sparse_decode_is_order_free_and_skips_padding():
    w, q = _sparse_small("scattered", False, batch=4)
    o0, l0 = orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides, w.indices, w.scale)
    idx = w.indices[:, ::-1].copy()                                   # reversed
    idx = np.concatenate([np.full((idx.shape[0], 7), -1, np.int32), idx], axis=1)   # more padding
    o1, l1 = orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides, idx, w.scale)
    assert np.allclose(o1, o0, rtol=1e-12, atol=1e-14) and np.allclose(l1, l0, rtol=1e-13)


def test_sparse_decode_duplicate_listing_doubles_the_weight():
    w, q = _sparse_small("blocks", False, batch=1, heads=3)
    a, b = 5, 17
    o, lse = orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides,
                                      np.array([[a, -1, b, a]]), w.scale)
    layer = w.storage.reshape(w.num_blocks, w.n_layers, w.page, 656)[:, w.layer].reshape(-1, 656)
    c_kv, k_pe = _ds_mla_values_by_library(layer[[a, b]])
    k = np.concatenate([c_kv, k_pe], axis=1)
    s = w.scale * (q[0] @ k.T)                                        # [H, 2]
    wa, wb = 2 * np.exp(s[:, 0]), np.exp(s[:, 1])
    want = (wa[:, None] * c_kv[0] + wb[:, None] * c_kv[1]) / (wa + wb)[:, None]
    assert np.allclose(o[0], want, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse[0], np.log(wa + wb), rtol=1e-13)


def test_sparse_decode_empty_single_and_out_of_range():
    w, q = _sparse_small("blocks", False, batch=2, heads=3)
    idx = np.array([[-1, -1, -1], [-1, 40, -1]])
    o, lse = orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides, idx, w.scale)
    assert np.array_equal(o[0], np.zeros((3, 512))) and np.all(lse[0] == -np.inf)
    layer = w.storage.reshape(w.num_blocks, w.n_layers, w.page, 656)[:, w.layer].reshape(-1, 656)
    c_kv, k_pe = _ds_mla_values_by_library(layer[[40]])
    assert np.allclose(o[1], np.broadcast_to(c_kv[0], (3, 512)), rtol=1e-14, atol=0)
    s = w.scale * (q[1] @ np.concatenate([c_kv[0], k_pe[0]]))
    assert np.allclose(lse[1], s, rtol=1e-13)
    with pytest.raises(ValueError):
        orc.decode_sparse_ds_mla(q, w.storage, w.offset, w.num_blocks, w.page, w.strides,
                                 np.array([[0, w.num_blocks * w.page], [1, 2]]), w.scale)


def test_sparse_planted_mistakes_are_caught(monkeypatch):
    good_values = orc.ds_mla_values

    def groups_reversed(entries):
        e = np.ascontiguousarray(entries, dtype=np.uint8).reshape(-1, 656).copy()
        sc = e[:, 512:528].reshape(-1, 4, 4)[:, ::-1].reshape(-1, 16)
        e[:, 512:528] = sc
        return good_values(e)

    def rope_big_endian(entries):
        e = np.ascontiguousarray(entries, dtype=np.uint8).reshape(-1, 656).copy()
        e[:, 528:] = e[:, 528:].reshape(-1, 64, 2)[:, :, ::-1].reshape(-1, 128)
        return good_values(e)

    for bad in (groups_reversed, rope_big_endian):
        monkeypatch.setattr(orc, "ds_mla_values", bad)
        with pytest.raises(AssertionError), np.errstate(invalid="ignore"):   # swapped bytes make NaNs
            test_ds_mla_entry_values_follow_the_byte_layout()
    monkeypatch.setattr(orc, "ds_mla_values", good_values)
    good_dec = orc.decode_sparse_ds_mla

    def padding_as_slot_zero(q, st, off, nb, page, strides, idx, scale, batch_ids=None):
        return good_dec(q, st, off, nb, page, strides, np.maximum(idx, 0), scale, batch_ids)

    def row_and_block_swapped(q, st, off, nb, page, strides, idx, scale, batch_ids=None):
        idx = np.asarray(idx)
        sw = np.where(idx >= 0, (idx % page) * page + idx // page, idx) if nb == page else idx
        s0, s1, s2 = strides
        return good_dec(q, st, off, nb, page, (s1, s0, s2), idx, scale, batch_ids) if nb != page else \
            good_dec(q, st, off, nb, page, strides, sw, scale, batch_ids)

    monkeypatch.setattr(orc, "decode_sparse_ds_mla", padding_as_slot_zero)
    with pytest.raises(AssertionError):
        test_sparse_decode_is_order_free_and_skips_padding()
    monkeypatch.setattr(orc, "decode_sparse_ds_mla", row_and_block_swapped)
    with pytest.raises((AssertionError, IndexError)):
        test_sparse_decode_equals_paged_decode_of_the_listed_rows("scattered", False)
    monkeypatch.setattr(orc, "decode_sparse_ds_mla", good_dec)
