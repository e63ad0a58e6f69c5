"""Pins of the oracle's W8A8 projections (the INT8 mode of the Linear step,
PyPTO-Gym AT-10 article, section 四: AT-05 per-token quant of the input,
int32 matmul, AT-06 dequant) against facts fixed outside the oracle: closed
forms of integer sums, the BF16 mode on inputs where both modes are exact,
the quantisation error bound against the real-valued product, and the
properties every per-token code row has."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from mla_attention_prolog_gb300 import workloads as wl


def f32(b):
    return wl.bf16_bits_to_f32(np.asarray(b, np.uint16))


def bf16_bits(v):
    """FP32 values -> BF16 bits by torch's conversion (round to nearest even)."""
    return torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _case(name, T=None, flags=0, seed=0, **over):
    w = wl.WORKLOADS[name]
    d = dataclasses.replace(w.dims, flags=w.dims.flags | wl.W8A8 | flags, **over)
    if T is not None:
        d = d.with_T(T)
    inp = wl.make_inputs(w, d, seed=seed)
    ww = wl.make_w8a8_weights(w, d, seed=seed)
    return d, inp, ww


def _run(d, inp, ww, **kw):
    return oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin,
                                  taps=True, **kw)


# ---------------------------------------------------------------- int32 matmul

def test_integer_dot_closed_forms():
    K = 7168
    a = np.full(K, 127, np.int8)
    # the largest magnitude a row of codes reaches: K * 127^2
    assert oracle.dot_i8(a, np.full(K, -127, np.int8)) == -K * 127 * 127
    alt = np.where(np.arange(K) % 2 == 0, 1, -1)
    assert oracle.dot_i8((alt * 127).astype(np.int8), (alt * 3).astype(np.int8)) == 381 * K
    # a[k] = (k mod 255) - 127 against w = 1: every full period of 255 sums
    # to 0, the last 28 entries are -127 .. -100
    ramp = ((np.arange(K) % 255) - 127).astype(np.int8)
    r = K % 255
    assert oracle.dot_i8(ramp, np.ones(K, np.int8)) == sum(range(-127, -127 + r))
    # against w[k] = k mod 3 - 1 (a transposed or shifted index changes it)
    w3 = ((np.arange(K) % 3) - 1).astype(np.int8)
    want = sum(((k % 255) - 127) * ((k % 3) - 1) for k in range(K))
    assert oracle.dot_i8(ramp, w3) == want


def test_dequant_converts_then_scales():
    # (float)y rounds to nearest: 2^24 + 1 -> 2^24, 2^24 + 3 -> 2^24 + 4
    assert oracle.dequant(2 ** 24 + 1, 1.0, 1.0) == 2.0 ** 24
    assert oracle.dequant(2 ** 24 + 3, 1.0, 1.0) == 2.0 ** 24 + 4
    assert oracle.dequant(-6, 0.5, 0.25) == -0.75
    assert oracle.dequant(0, 3.0, 7.0) == 0.0
    # scales are applied (a dropped scale would give 100 or 10)
    assert oracle.dequant(100, 0.1, 0.5) == pytest.approx(5.0, rel=1e-6)


def test_project_w8a8_uses_rows_of_w():
    """Out n takes row n of W (not column n) and scale n."""
    W = np.array([[1, 2, 3], [4, 5, 6]], np.int8)
    a = np.array([1, 0, -1], np.int8)
    out = oracle.project_w8a8(a, W, 2.0, np.array([1.0, 10.0], np.float32))
    assert out.tolist() == [(1 - 3) * 2.0, (4 - 6) * 2.0 * 10.0]


# ------------------------------------------------------- the whole prolog

def test_compression_equals_bf16_mode_where_both_are_exact():
    """x rows of integers whose largest magnitude is 127 quantise to
    themselves with scale 1; with weight scales 1 the W8A8 compression is the
    exact sum rounded once to BF16 -- the BF16 mode's definition."""
    d, inp, ww = _case("tiny_q")
    rng = np.random.default_rng(5)
    xi = rng.integers(-127, 128, size=(d.T, d.D)).astype(np.float32)
    xi[:, 0] = 127.0  # amax 127 in every row
    inp = dataclasses.replace(inp, x=bf16_bits(xi))
    ww = dataclasses.replace(ww, w_scale=np.ones_like(ww.w_scale))
    got = _run(d, inp, ww)
    assert np.array_equal(got["x_codes"], xi.astype(np.int8))
    assert np.all(got["x_scale"] == 1.0)
    d16 = dataclasses.replace(d, flags=d.flags & ~wl.W8A8)
    ref = oracle.mla_prolog(d16, inp.x, inp.gamma, bf16_bits(ww.W_a.astype(np.float32)),
                            bf16_bits(ww.W_b.astype(np.float32)), inp.positions, inp.cos_sin, taps=True)
    assert np.array_equal(got["c"], ref["c"])
    assert np.array_equal(got["normed"], ref["normed"])
    assert np.array_equal(got["out_kpe"], ref["out_kpe"])


def test_worst_case_magnitude_is_exact():
    """Every code 127 against every weight code 127: c = bf16(D * 127^2 * s)."""
    d, inp, ww = _case("tiny", D=7168)
    inp = dataclasses.replace(inp, x=bf16_bits(np.full((d.T, d.D), 127.0, np.float32)))
    s = np.float32(2.0 ** -20)
    ww = dataclasses.replace(ww, W_a=np.full_like(ww.W_a, 127), w_scale=np.full_like(ww.w_scale, s))
    got = _run(d, inp, ww)
    v = float(d.D * 127 * 127) * 2.0 ** -20  # exact in FP32: 17 significant bits times a power of 2
    assert np.all(got["c"] == bf16_bits([v])[0])


def _bound_check(y, a_vals, a_scale, W_codes, w_scale, bf16_out):
    """|y - a . (W_codes * w_scale)| stays within the quantisation error of the
    input row (|a - code * s_a| <= s_a / 2 per entry) plus the output rounding
    (BF16 half-ulp, else a few FP32 ulps) and the FP32 steps."""
    W = W_codes.astype(np.float64) * w_scale.astype(np.float64)[:, None]
    exact = W @ a_vals.astype(np.float64)
    qerr = 0.5 * float(a_scale) * np.abs(W).sum(axis=1)
    rnd = (2.0 ** -8 if bf16_out else 2.0 ** -22) * (np.abs(exact) + qerr)
    assert np.all(np.abs(y.astype(np.float64) - exact) <= qerr * 1.0001 + rnd + 1e-30)
    return exact


@pytest.mark.parametrize("name", ["tiny", "tiny_q"])
def test_projections_within_the_quantisation_bound(name):
    d, inp, ww = _case(name, seed=3)
    got = _run(d, inp, ww)
    Lq, Lkv, R, H, Dn, Dv = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim, d.v_dim
    NQw = d.n_q if Lq else 0
    s_a = ww.w_scale[:d.n_a]
    s_q = ww.w_scale[d.n_a:d.n_a + NQw]
    s_kv = ww.w_scale[d.n_a + NQw:]
    W_qb = ww.W_b[:NQw * Lq].reshape(NQw, Lq)
    W_kvb = ww.W_b[NQw * Lq:].reshape(d.n_kv, Lkv)
    X = f32(inp.x).reshape(d.T, d.D)
    for t in range(d.T):
        _bound_check(f32(got["c"][t]), X[t], got["x_scale"][t], ww.W_a, s_a, True)
        nrm = f32(got["normed"][t])
        kv = _bound_check(np.concatenate([np.concatenate([f32(got["out_k"][t, h, :Dn]), f32(got["out_v"][t, h])])
                                          for h in range(H)]),
                          nrm[Lq:], got["n_scale"][t, 1], W_kvb, s_kv, True)
        assert np.abs(kv).max() > 0
        if Lq:
            q = got["q"][t].reshape(H, Dn + R)
            rows = np.concatenate([np.arange(h * (Dn + R), h * (Dn + R) + Dn) for h in range(H)])
            _bound_check(q[:, :Dn].reshape(-1), nrm[:Lq], got["n_scale"][t, 0], W_qb[rows], s_q[rows], False)


def test_code_rows_are_per_token_quantisations():
    d, inp, ww = _case("tiny_q", seed=4)
    got = _run(d, inp, ww)
    X = f32(inp.x).reshape(d.T, d.D)
    for t in range(d.T):
        for vals, codes, s in ((X[t], got["x_codes"][t], got["x_scale"][t]),
                               (f32(got["normed"][t, :d.q_lora_rank]), got["n_codes"][t, :d.q_lora_rank],
                                got["n_scale"][t, 0]),
                               (f32(got["normed"][t, d.q_lora_rank:]), got["n_codes"][t, d.q_lora_rank:],
                                got["n_scale"][t, 1])):
            amax = np.abs(vals).max()
            assert s == pytest.approx(amax / 127, rel=1e-6)
            assert np.abs(codes.astype(np.int32)).max() == 127
            assert np.all(np.abs(codes * np.float64(s) - vals) <= 0.5 * s * (1 + 1e-5) + 1e-30)


def test_zero_row_and_bad_position():
    d, inp, ww = _case("tiny_q", seed=6)
    x = inp.x.reshape(d.T, d.D).copy()
    x[1] = 0
    pos = inp.positions.copy()
    pos[2] = d.max_pos  # out of range
    got = _run(d, dataclasses.replace(inp, x=x.reshape(-1) if inp.x.ndim == 1 else x, positions=pos), ww)
    assert np.all(got["x_codes"][1] == 0) and got["x_scale"][1] == 0.0
    assert np.all(f32(got["c"][1]) == 0.0)
    assert got["bad_positions"] == 1
    assert np.all(got["out_k"][2] == 0) and np.all(got["out_q_int8"][2] == 0)
    assert np.all(got["n_codes"][2] == 0) and np.all(got["n_scale"][2] == 0)


def test_flag_and_weights_must_agree():
    d, inp, ww = _case("tiny")
    with pytest.raises(ValueError):  # BF16 entry with the W8A8 flag
        oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    d16 = dataclasses.replace(d, flags=d.flags & ~wl.W8A8)
    with pytest.raises(ValueError):  # W8A8 entry without the flag
        oracle.mla_prolog_w8a8(d16, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin)


def _f32_rn(q):
    """The FP32 value nearest to the rational q (ties to even), by exact arithmetic."""
    from fractions import Fraction
    q = Fraction(q)
    if q == 0:
        return 0.0
    lo = float(np.float32(float(q)))  # within one FP32 ulp of q
    cands = sorted({lo, float(np.nextafter(np.float32(lo), np.float32(np.inf))),
                    float(np.nextafter(np.float32(lo), np.float32(-np.inf)))})
    best = min(cands, key=lambda c: (abs(Fraction(c) - q), int(np.array([c], np.float32).view(np.uint32)[0]) & 1))
    return best


def test_worked_example_by_hand():
    """A projection worked by hand (AT-05, int32 matmul, AT-06):
    x = (1, -0.5, 0.25, 2): amax 2, inv = 127/2 = 63.5 exactly, x * inv =
    (63.5, -31.75, 15.875, 127) -> rint half-even (64, -32, 16, 127), scale
    s_x = fl(2/127).  W rows (1, 2, 3, 4) and (-1, 0, 1, 0): integer sums
    64 - 64 + 48 + 508 = 556 and -64 + 16 = -48.  Dequant with w_scale
    (0.5, 0.25): fl(fl(556 * s_x) * 0.5), fl(fl(-48 * s_x) * 0.25)."""
    from fractions import Fraction
    x = np.array([1.0, -0.5, 0.25, 2.0], np.float32)
    codes, s_x = oracle.quant_row(x)
    assert codes.tolist() == [64, -32, 16, 127]
    assert s_x == _f32_rn(Fraction(2, 127))
    W = np.array([[1, 2, 3, 4], [-1, 0, 1, 0]], np.int8)
    assert [oracle.dot_i8(codes, W[0]), oracle.dot_i8(codes, W[1])] == [556, -48]
    y = oracle.project_w8a8(codes, W, s_x, np.array([0.5, 0.25], np.float32))
    want = [_f32_rn(Fraction(_f32_rn(556 * Fraction(s_x))) * Fraction(1, 2)),
            _f32_rn(Fraction(_f32_rn(-48 * Fraction(s_x))) * Fraction(1, 4))]
    assert y.tolist() == want
    # and it approximates the real-valued product x . W[n] * w_scale[n] within
    # s_x / 2 * sum |W[n]| * w_scale[n] (rows 0 and 1: sum |W| = 10 and 2)
    exact = [float(np.dot(x.astype(np.float64), W[0].astype(np.float64))) * 0.5,
             float(np.dot(x.astype(np.float64), W[1].astype(np.float64))) * 0.25]
    assert abs(y[0] - exact[0]) <= 0.5 * s_x * 10 * 0.5 + 1e-6
    assert abs(y[1] - exact[1]) <= 0.5 * s_x * 2 * 0.25 + 1e-6


def test_given_codes_feed_the_expansions():
    """The given-codes input (used to check a candidate's steps after its own
    normed-row codes): the oracle's own codes give its own outputs bit for
    bit; a code moved by one changes only that token's outputs, and its
    k_nope and value are the AT-06 product of the moved codes, formed here
    with numpy's integer dot, FP32 multiplies and torch's BF16 conversion."""
    d, inp, ww = _case("tiny_q", T=6, max_pos=8)
    own = _run(d, inp, ww)
    again = _run(d, inp, ww, given_codes=own["n_codes"], given_scale=own["n_scale"])
    for k in ("out_k", "out_v", "out_kpe", "out_q_int8", "out_scale"):
        assert np.array_equal(again[k], own[k]), k
    Lq, Lkv, H, Dn, Dv, R = d.q_lora_rank, d.kv_lora_rank, d.num_heads, d.nope_dim, d.v_dim, d.rope_dim
    codes = own["n_codes"].copy()
    j, k = 2, Lq + 5
    codes[j, k] += 1 if codes[j, k] < 127 else -1
    moved = _run(d, inp, ww, given_codes=codes, given_scale=own["n_scale"])
    for t in range(d.T):
        if t == j:
            continue
        for name in ("out_k", "out_v", "out_q_int8", "out_scale"):
            assert np.array_equal(moved[name][t], own[name][t]), (name, t)
    NQ = H * (Dn + R)
    W_kv = ww.W_b[NQ * Lq:].reshape(H * (Dn + Dv), Lkv).astype(np.int64)
    s_kv = ww.w_scale[d.n_a + NQ:]
    acc = (W_kv @ codes[j, Lq:].astype(np.int64)).astype(np.float32)
    kv = (acc * np.float32(own["n_scale"][j, 1])) * s_kv
    kv = bf16_bits(kv).reshape(H, Dn + Dv)
    assert np.array_equal(moved["out_k"][j][:, :Dn], kv[:, :Dn])
    assert np.array_equal(moved["out_v"][j], kv[:, Dn:])
    assert not np.array_equal(moved["out_v"][j], own["out_v"][j])
    assert np.array_equal(moved["out_kpe"][j], own["out_kpe"][j])  # k_pe does not pass through the codes
    with pytest.raises(ValueError):
        _run(d, inp, ww, given_codes=codes)
