"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each pin takes an independent route: exact rational arithmetic, a library
routine (torch / numpy), a closed form, an invariant of the mathematics, or a
hand-derived worked example under ``tests/golden/``.  They are chosen so that
a plausible slip in the oracle (a dropped term, a wrong sign or pairing, a
transposed operand, the wrong rounding rule) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from mla_attention_prolog_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def bits_to_f32(b):
    return wl.bf16_bits_to_f32(np.asarray(b, np.uint16))


def nearest_bf16_exact(v: float) -> int:
    """Nearest BF16 to the real number v (ties to even), by exact rationals."""
    if v == 0:
        return 0x8000 if math.copysign(1, v) < 0 else 0
    fv = Fraction(v)
    # candidate bit patterns around the FP32 truncation of v
    f32 = np.float32(v)
    base = int(np.array([f32], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for b in range(max(base - 2, 0), min(base + 3, 0xFFFF)):
        c = float(bits_to_f32([b])[0])
        if not math.isfinite(c) or (c == 0 and b not in (0, 0x8000)):
            continue
        if (c < 0) != (v < 0) and c != 0:
            continue
        err = abs(Fraction(c) - fv)
        key = (err, b & 1)  # ties go to the even mantissa
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


# ----------------------------------------------------------------- BF16 casts

def test_f32_to_bf16_matches_torch(oracle_lib):
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(500) * 1e-39).astype(np.float32),   # subnormals
        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 65504.0, 3.0e38], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_lib.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_bf16_ties_to_even(oracle_lib):
    assert oracle_lib.f32_to_bf16(1.0 + 2**-8) == 0x3F80       # tie -> even (1.0)
    assert oracle_lib.f32_to_bf16(1.0 + 3 * 2**-8) == 0x3F82   # tie -> even (1 + 2^-6)
    assert oracle_lib.f32_to_bf16(1.0 + 2**-8 + 2**-20) == 0x3F81


def test_f64_to_bf16_exact_rationals(oracle_lib):
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000))
    vals += [1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-40, -(1.0 + 2**-8 + 2**-40)]
    for v in vals:
        assert oracle_lib.f64_to_bf16(v) == nearest_bf16_exact(v), v


# ----------------------------------------------------------------- projection

def _rand_bf16(shape, std=1.0):
    return wl._bf16_bits(torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)))


def test_projection_one_hot_reproduces_weight_column(oracle_lib):
    N, K = 40, 96
    W = _rand_bf16((N, K), 0.02)
    for j in (0, 17, K - 1):
        x = np.zeros(K, np.uint16)
        x[j] = 0x3F80  # 1.0
        got = oracle_lib.project_bf16(x, W)
        assert np.array_equal(got, W[:, j]), j       # [N, K] layout: column j, not row j
    # two-hot: the sum of two columns, rounded once
    x = np.zeros(K, np.uint16)
    x[3] = 0x3F80
    x[50] = 0x4000  # 2.0
    want = [nearest_bf16_exact(float(a) + 2.0 * float(b))
            for a, b in zip(bits_to_f32(W[:, 3]), bits_to_f32(W[:, 50]))]
    assert np.array_equal(oracle_lib.project_bf16(x, W), np.array(want, np.uint16))


def test_projection_matches_library_matmul(oracle_lib):
    N, K = 64, 512
    W = _rand_bf16((N, K), 0.02)
    x = _rand_bf16((K,), 1.0)
    ref = torch.from_numpy(bits_to_f32(W).astype(np.float64)) @ torch.from_numpy(bits_to_f32(x).astype(np.float64))
    want = np.array([nearest_bf16_exact(float(v)) for v in ref.numpy()], np.uint16)
    assert np.array_equal(oracle_lib.project_bf16(x, W), want)
    got32 = oracle_lib.project_f32(x, W)
    assert np.array_equal(got32, ref.numpy().astype(np.float32))


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_matches_torch_rms_norm(oracle_lib):
    for L in (64, 512, 1536):
        x = _rand_bf16((L,), 1.3)
        g = wl._bf16_bits(torch.from_numpy((1 + 0.1 * rng.standard_normal(L)).astype(np.float32)))
        y32, y16 = oracle_lib.rmsnorm_row(x, g, 1e-6)
        ref = torch.nn.functional.rms_norm(
            torch.from_numpy(bits_to_f32(x).astype(np.float64))[None], (L,),
            weight=torch.from_numpy(bits_to_f32(g).astype(np.float64)), eps=1e-6)[0].numpy()
        # FP32 sequential sum of L positive terms: relative error <= (L-1)*2^-24, plus a
        # few roundings after it; a dropped term would move rstd by ~1/(2L), far above.
        np.testing.assert_allclose(y32, ref, rtol=(L + 8) * 2.0**-24, atol=0)
        # BF16 output is the rounding of the FP32 result: within one BF16 step of the exact
        diff = np.abs(bits_to_f32(y16).astype(np.float64) - ref)
        assert np.all(diff <= np.abs(ref) * (2**-8 + (L + 8) * 2.0**-24))


def test_rmsnorm_unit_gamma_closed_form(oracle_lib):
    for L, scale in ((512, 1.0), (1536, 0.05), (64, 30.0)):
        x = _rand_bf16((L,), scale)
        xf = bits_to_f32(x).astype(np.float64)
        ms = np.mean(xf * xf)
        y32, _ = oracle_lib.rmsnorm_row(x, None, 1e-6)
        rms = math.sqrt(np.mean(y32.astype(np.float64) ** 2))
        assert abs(rms - math.sqrt(ms / (ms + 1e-6))) <= 1e-6


def test_rmsnorm_constant_row(oracle_lib):
    for c in (0.5, -3.0, 1e-3):
        x = np.full(256, oracle_lib.f32_to_bf16(c), np.uint16)
        cb = float(bits_to_f32(x[:1])[0])
        y32, _ = oracle_lib.rmsnorm_row(x, None, 1e-6)
        np.testing.assert_allclose(y32, cb / math.sqrt(cb * cb + 1e-6), rtol=1e-6)


def test_rmsnorm_scale_invariance_eps0(oracle_lib):
    x = _rand_bf16((512,), 1.0)
    y_a, _ = oracle_lib.rmsnorm_row(x, None, 0.0)
    x4 = wl._bf16_bits(torch.from_numpy(bits_to_f32(x) * np.float32(16.0)))  # exact 2^4 scaling
    y_b, _ = oracle_lib.rmsnorm_row(x4, None, 0.0)
    assert np.array_equal(y_a, y_b)


# ----------------------------------------------------------------- RoPE

def _table(max_pos=64, R=16):
    return wl.cos_sin_table(max_pos, R)


def test_rope_identity_at_position_zero(oracle_lib):
    tab = _table()
    x = rng.standard_normal(16).astype(np.float32)
    assert np.array_equal(tab[0, :8], np.ones(8, np.float32))
    assert np.array_equal(tab[0, 8:], np.zeros(8, np.float32))
    assert np.array_equal(oracle_lib.rope(x, tab[0]), x)


def test_rope_unit_vectors_rotate_half_pairing(oracle_lib):
    R, tab = 16, _table()
    p = 7
    c, s = tab[p, :8], tab[p, 8:]
    for i in range(8):
        e = np.zeros(R, np.float32)
        e[i] = 1
        out = oracle_lib.rope(e, tab[p])
        want = np.zeros(R, np.float32)
        want[i], want[i + 8] = c[i], s[i]
        assert np.array_equal(out, want)
        e = np.zeros(R, np.float32)
        e[i + 8] = 1
        out = oracle_lib.rope(e, tab[p])
        want = np.zeros(R, np.float32)
        want[i], want[i + 8] = -s[i], c[i]
        assert np.array_equal(out, want)


def test_rope_matches_complex_rotation(oracle_lib):
    R, tab = 64, wl.cos_sin_table(4096, 64)
    for p in (1, 100, 4095):
        x = rng.standard_normal(R).astype(np.float32)
        z = x[:32].astype(np.float64) + 1j * x[32:].astype(np.float64)
        theta = 10000.0 ** (-2.0 * np.arange(32) / R)
        w = z * np.exp(1j * p * theta)
        out = oracle_lib.rope(x, tab[p]).astype(np.float64)
        np.testing.assert_allclose(out[:32], w.real, atol=2e-6 * np.abs(z).max())
        np.testing.assert_allclose(out[32:], w.imag, atol=2e-6 * np.abs(z).max())


def test_rope_preserves_pair_norms_and_composes(oracle_lib):
    R, tab = 64, wl.cos_sin_table(8192, 64)
    x = rng.standard_normal(R).astype(np.float32)
    for p1, p2 in ((3, 5), (1000, 2000), (4000, 4095)):
        a = oracle_lib.rope(x, tab[p1])
        n0 = np.hypot(x[:32].astype(np.float64), x[32:])
        n1 = np.hypot(a[:32].astype(np.float64), a[32:])
        np.testing.assert_allclose(n1, n0, rtol=1e-6)
        b = oracle_lib.rope(a, tab[p2])
        c = oracle_lib.rope(x, tab[p1 + p2])
        np.testing.assert_allclose(b, c, atol=1e-5 * np.abs(x).max() * 10)


# ----------------------------------------------------------------- quant

def test_quant_worked_examples(oracle_lib):
    cases = json.load(open(os.path.join(GOLDEN, "quant_worked_example.json")))["cases"]
    for cs in cases:
        codes, scale = oracle_lib.quant_row(np.array(cs["y"], np.float32))
        assert codes.tolist() == cs["codes"]
        assert scale == cs["scale"]


def _brute_quant(y32):
    """Independent route: numpy FP32 ops and Python's round() (ties to even)."""
    amax = np.float32(np.max(np.abs(y32)))
    if amax == 0:
        return np.zeros(len(y32), np.int8), 0.0
    inv = np.float32(127.0) / amax
    prods = (y32 * inv).astype(np.float32)
    codes = np.array([max(-127, min(127, round(float(v)))) for v in prods], np.int8)
    return codes, float(amax / np.float32(127.0))


def test_quant_brute_force_and_invariants(oracle_lib):
    for n, s in ((24576, 0.3), (1000, 1e-4), (77, 50.0)):
        y = (rng.standard_normal(n) * s).astype(np.float32)
        codes, scale = oracle_lib.quant_row(y)
        bc, bs = _brute_quant(y)
        assert np.array_equal(codes, bc) and scale == bs
        assert np.max(np.abs(codes.astype(int))) == 127
        err = np.abs(y.astype(np.float64) - codes.astype(np.float64) * scale)
        assert np.all(err <= scale * (0.5 + 1e-4))
        c2, s2 = oracle_lib.quant_row(-y)
        assert np.array_equal(c2, -codes) and s2 == scale
        c3, s3 = oracle_lib.quant_row(y * np.float32(8.0))
        assert np.array_equal(c3, codes) and s3 == scale * 8.0


# ----------------------------------------------------------------- whole op

def _small_dims(**kw):
    base = dict(T=6, D=128, q_lora_rank=32, kv_lora_rank=64, rope_dim=16, num_heads=3,
                nope_dim=32, v_dim=16, max_pos=32, flags=wl.QUANT_Q)
    base.update(kw)
    return wl.Dims(**base)


def _independent_chain(d, inp):
    """The prolog re-expressed with library routines (torch float64/float32,
    complex rotation, Python round) as a brute-force cross-check on tiny sizes."""
    f = lambda a: torch.from_numpy(bits_to_f32(a).astype(np.float64))
    x = f(inp.x).reshape(d.T, d.D)
    Wa = f(inp.W_a).reshape(d.n_a, d.D)
    g = bits_to_f32(inp.gamma)
    Lq, Lkv, R, H, Dn, Dv = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim, d.v_dim
    C = (x @ Wa.T).numpy()
    Cb = np.vectorize(lambda v: float(bits_to_f32([nearest_bf16_exact(v)])[0]))(C)
    def norm(blk, gam):
        t = torch.from_numpy(blk.astype(np.float32))
        y = torch.nn.functional.rms_norm(t, (blk.shape[1],), weight=torch.from_numpy(gam), eps=d.eps)
        return y.to(torch.bfloat16).to(torch.float64).numpy()
    nq = norm(Cb[:, :Lq], g[:Lq]) if Lq else None
    nkv = norm(Cb[:, Lq:Lq + Lkv], g[Lq:])
    tab = inp.cos_sin[inp.positions].astype(np.float64)
    half = R // 2
    def rot(v):  # v [T, ..., R] float64
        z = v[..., :half] + 1j * v[..., half:]
        w = z * (tab[:, None, :half] + 1j * tab[:, None, half:]) if v.ndim == 3 else \
            z * (tab[:, :half] + 1j * tab[:, half:])
        return np.concatenate([w.real, w.imag], -1)
    kpe = rot(Cb[:, Lq + Lkv:])
    Wb = bits_to_f32(inp.W_b).astype(np.float64)
    Wkv = Wb[d.n_q * Lq:].reshape(d.n_kv, Lkv)
    KV = (nkv @ Wkv.T).reshape(d.T, H, Dn + Dv)
    res = {"kpe": kpe, "k_nope": KV[:, :, :Dn], "v": KV[:, :, Dn:], "Cb": Cb, "nkv": nkv}
    if Lq:
        Wq = Wb[:d.n_q * Lq].reshape(d.n_q, Lq)
        Q = (nq @ Wq.T).reshape(d.T, H, Dn + R)
        Q[:, :, Dn:] = rot(Q[:, :, Dn:])
        res["q"] = Q.reshape(d.T, -1)
    return res


@pytest.mark.parametrize("name", ["tiny", "tiny_q"])
def test_whole_op_against_independent_chain(oracle_lib, name):
    w = wl.WORKLOADS[name]
    d = w.dims
    inp = wl.make_inputs(w)
    o = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, taps=True)
    ref = _independent_chain(d, inp)
    assert o["bad_positions"] == 0
    assert np.array_equal(bits_to_f32(o["c"]), ref["Cb"].astype(np.float32))
    nk = bits_to_f32(o["normed"][:, d.q_lora_rank:]).astype(np.float64)
    assert np.all(np.abs(nk - ref["nkv"]) <= np.abs(ref["nkv"]) * 2**-7)  # <= 1 BF16 step
    kpe = bits_to_f32(o["out_kpe"]).astype(np.float64)
    assert np.all(np.abs(kpe - ref["kpe"]) <= np.abs(ref["kpe"]) * 2**-8 + 1e-6)
    ok = bits_to_f32(o["out_k"]).astype(np.float64)
    ov = bits_to_f32(o["out_v"]).astype(np.float64)
    tol = lambda r: 1e-2 + 1e-2 * np.abs(r)
    assert np.all(np.abs(ok[:, :, :d.nope_dim] - ref["k_nope"]) <= tol(ref["k_nope"]))
    assert np.all(np.abs(ov - ref["v"]) <= tol(ref["v"]))
    for h in range(d.num_heads):  # K assembles the shared rotated k_pe into every head
        assert np.array_equal(o["out_k"][:, h, d.nope_dim:], o["out_kpe"])
    if d.q_lora_rank:
        np.testing.assert_allclose(o["q"], ref["q"], rtol=2e-2, atol=2e-3)
        q8 = o["out_q_int8"].reshape(d.T, -1)
        for t in range(d.T):
            c, s = _brute_quant(o["q"][t])
            assert np.array_equal(q8[t], c) and o["out_scale"][t] == s


def test_whole_op_shapes_mla_prolog_001(oracle_lib):
    g = json.load(open(os.path.join(GOLDEN, "shapes_mla_prolog_001.json")))
    d = wl.Dims(max_pos=8, **g["dims"])
    inp = wl.make_inputs(wl.Workload("case001", d, positions="arange"))
    pl = g["page_layout"]
    assert list(inp.x.reshape(1, 1, -1).shape) == pl["hidden_states"]
    assert [d.D, d.n_a] == pl["kv_a_weight"]                 # the page passes it pre-transposed
    assert [d.kv_lora_rank, d.n_kv] == pl["kv_b_weight"]
    assert [d.kv_lora_rank] == pl["ln_weight"] and d.eps == pl["eps"]
    o = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    b, h, s, dn = pl["k_nope"]
    assert o["out_k"][:, :, :d.nope_dim].shape == (b * s, h, dn)
    assert o["out_v"].shape == (pl["value"][0] * pl["value"][2], pl["value"][1], pl["value"][3])
    assert o["out_kpe"].shape == (1, pl["k_pe"][3])


def test_whole_op_token_subset_and_threads(oracle_lib):
    d = _small_dims()
    inp = wl.make_inputs(wl.Workload("s", d, positions="uniform"))
    oracle_lib.set_threads(1)
    full = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    oracle_lib.set_threads(4)
    full4 = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    sub = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin,
                                tokens=[5, 0, 2])
    for k in ("out_k", "out_v", "out_kpe", "out_q_int8", "out_scale"):
        assert np.array_equal(full[k], full4[k])
        assert np.array_equal(sub[k], full[k][[5, 0, 2]])


def test_whole_op_bad_position_zero_fills(oracle_lib):
    d = _small_dims()
    inp = wl.make_inputs(wl.Workload("s", d, positions="uniform"))
    pos = inp.positions.copy()
    pos[1] = d.max_pos   # one past the table
    pos[4] = -1
    o = oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, pos, inp.cos_sin)
    assert o["bad_positions"] == 2
    for t in (1, 4):
        for k in ("out_k", "out_v", "out_kpe", "out_q_int8"):
            assert not np.any(o[k][t])
        assert o["out_scale"][t] == 0
    assert np.any(o["out_k"][0])


def test_whole_op_zero_x_row(oracle_lib):
    """x = 0 gives c = 0, normed = 0 (eps > 0), all outputs 0, scale 0."""
    d = _small_dims(T=2)
    inp = wl.make_inputs(wl.Workload("s", d, positions="arange"))
    x = inp.x.copy()
    x[0] = 0
    o = oracle_lib.mla_prolog(d, x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    assert not np.any(o["out_k"][0]) and not np.any(o["out_v"][0]) and not np.any(o["out_q_int8"][0])
    assert o["out_scale"][0] == 0.0 and o["out_scale"][1] > 0
