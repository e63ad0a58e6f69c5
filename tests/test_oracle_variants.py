"""Pins of the oracle's variant steps (interleaved RoPE, per-head q RMSNorm,
per-(token, head) quant, latent KV-cache scatter) against facts fixed outside
the oracle: library reshapes and norms, complex rotation, exact invariances,
and identities with the base path on permuted weights.
"""
import numpy as np
import pytest
import torch

from mla_attention_prolog_gb300 import workloads as wl

rng = np.random.default_rng(4321)


def f32(bits):
    return wl.bf16_bits_to_f32(np.asarray(bits, np.uint16))


def _dims(**kw):
    base = dict(T=5, D=128, q_lora_rank=32, kv_lora_rank=64, rope_dim=16, num_heads=3,
                nope_dim=32, v_dim=16, max_pos=32, flags=wl.QUANT_Q)
    base.update(kw)
    return wl.Dims(**base)


def _run(oracle_lib, d, inp, W_a=None, W_b=None, taps=False):
    return oracle_lib.mla_prolog(d, inp.x, inp.gamma, inp.W_a if W_a is None else W_a,
                                 inp.W_b if W_b is None else W_b, inp.positions, inp.cos_sin, taps=taps)


# ------------------------------------------------------------ interleaved RoPE

def test_deinterleave_is_the_chunk2_transpose(oracle_lib):
    """[R/2, 2] viewed and transposed to [2, R/2] (numpy's reshape/transpose)."""
    for R in (16, 64):
        x = rng.standard_normal(R).astype(np.float32)
        want = x.reshape(R // 2, 2).T.reshape(R)
        assert np.array_equal(oracle_lib.deinterleave(x), want)


def test_interleaved_rope_rotates_adjacent_pairs(oracle_lib):
    """De-interleave + rotate-half == complex rotation of (x[2i], x[2i+1])."""
    R, tab = 64, wl.cos_sin_table(4096, 64)
    theta = 10000.0 ** (-2.0 * np.arange(R // 2) / R)
    for p in (0, 1, 77, 4095):
        x = rng.standard_normal(R).astype(np.float32)
        out = oracle_lib.rope(oracle_lib.deinterleave(x), tab[p]).astype(np.float64)
        z = x[0::2].astype(np.float64) + 1j * x[1::2].astype(np.float64)
        w = z * np.exp(1j * p * theta)
        np.testing.assert_allclose(out[:R // 2], w.real, atol=2e-6 * np.abs(z).max())
        np.testing.assert_allclose(out[R // 2:], w.imag, atol=2e-6 * np.abs(z).max())


def _deinterleave_perm(R):
    return np.concatenate([np.arange(0, R, 2), np.arange(1, R, 2)])


@pytest.mark.parametrize("extra", [0, wl.QUANT_PER_HEAD, wl.Q_HEAD_NORM | wl.QUANT_PER_HEAD])
def test_interleaved_whole_op_equals_base_op_on_permuted_rope_rows(oracle_lib, extra):
    """The interleaved variant on W equals the base path on W with the rope
    output rows (k_pe rows of W_a, each head's rope rows of W_q_b) permuted by
    the de-interleave: every output bit-identical (with the per-head norm, up
    to the order in which the head's squares are summed)."""
    d = _dims(flags=wl.QUANT_Q | extra)
    inp = wl.make_inputs(wl.Workload("v", d, positions="uniform"))
    Lq, Lkv, R, H, Dn = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim
    perm = _deinterleave_perm(R)
    Wa = inp.W_a.reshape(d.n_a, d.D).copy()
    Wa[Lq + Lkv:] = Wa[Lq + Lkv:][perm]
    Wb = inp.W_b.copy()
    Wq = Wb[:d.n_q * Lq].reshape(H, Dn + R, Lq)
    Wq[:, Dn:] = Wq[:, Dn:][:, perm]
    base = _run(oracle_lib, d, inp, W_a=Wa.reshape(-1), W_b=Wb)
    di = wl.Dims(**{**d.__dict__, "flags": d.flags | wl.ROPE_INTERLEAVED})
    inter = _run(oracle_lib, di, inp)
    exact = ("out_k", "out_v", "out_kpe") if extra & wl.Q_HEAD_NORM else \
        ("out_k", "out_v", "out_kpe", "out_q_int8", "out_scale")
    for k in exact:
        assert np.array_equal(base[k], inter[k]), k
    if extra & wl.Q_HEAD_NORM:
        np.testing.assert_allclose(inter["out_scale"], base["out_scale"], rtol=1e-6)
        diff = np.abs(inter["out_q_int8"].astype(int) - base["out_q_int8"].astype(int))
        assert diff.max() <= 1 and diff.mean() <= 1e-2


# ------------------------------------------------------- per-head q RMSNorm

def test_rmsnorm_f32_row_against_torch_and_closed_form(oracle_lib):
    for L, eps, s in ((192, 1e-6, 1.0), (512, 1e-6, 3e-3), (64, 0.0, 40.0)):
        x = (rng.standard_normal(L) * s).astype(np.float32)
        y = oracle_lib.rmsnorm_f32_row(x, eps).astype(np.float64)
        t = torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (L,), eps=eps).numpy()
        np.testing.assert_allclose(y, t, rtol=4e-6, atol=1e-30)
        ms = np.mean(x.astype(np.float64) ** 2)
        assert abs(np.mean(y ** 2) - ms / (ms + eps)) <= 1e-5


def test_rmsnorm_f32_row_power_of_two_invariance(oracle_lib):
    x = rng.standard_normal(192).astype(np.float32)
    y = oracle_lib.rmsnorm_f32_row(x, 0.0)
    for k in (-6, 3, 10):
        assert np.array_equal(oracle_lib.rmsnorm_f32_row(x * np.float32(2.0 ** k), 0.0), y)


def test_head_norm_whole_op_against_independent_chain(oracle_lib):
    """q with the per-head norm: torch float64 projection of the oracle's own
    normed c_q, torch rms_norm per head, complex rotation of the rope slice."""
    d = _dims(flags=wl.QUANT_Q | wl.Q_HEAD_NORM)
    inp = wl.make_inputs(wl.Workload("v", d, positions="uniform"))
    o = _run(oracle_lib, d, inp, taps=True)
    Lq, R, H, Dn = d.q_lora_rank, d.rope_dim, d.num_heads, d.nope_dim
    nq = torch.from_numpy(f32(o["normed"][:, :Lq]).astype(np.float64))
    Wq = torch.from_numpy(f32(inp.W_b[:d.n_q * Lq]).astype(np.float64).reshape(d.n_q, Lq))
    Q = (nq @ Wq.T).reshape(d.T, H, Dn + R)
    ms_pre = (Q ** 2).mean(-1).numpy()
    Q = torch.nn.functional.rms_norm(Q, (Dn + R,), eps=d.eps).numpy()
    tab = inp.cos_sin[inp.positions].astype(np.float64)
    z = Q[:, :, Dn:Dn + R // 2] + 1j * Q[:, :, Dn + R // 2:]
    w = z * (tab[:, None, :R // 2] + 1j * tab[:, None, R // 2:])
    Q[:, :, Dn:] = np.concatenate([w.real, w.imag], -1)
    np.testing.assert_allclose(o["q"].reshape(d.T, H, -1), Q, rtol=1e-4, atol=1e-5)
    # every head row's mean square is ms / (ms + eps) (RoPE keeps the head's
    # sum of squares)
    ms = np.mean(o["q"].reshape(d.T, H, -1).astype(np.float64) ** 2, -1)
    np.testing.assert_allclose(ms, ms_pre / (ms_pre + d.eps), atol=1e-5)


# ------------------------------------------------- per-(token, head) quant

def test_per_head_quant_against_per_token_quant(oracle_lib):
    """Per head row: |code| reaches 127; the head holding the token's max |q|
    gets exactly the per-token codes and scale."""
    d = _dims(T=6)
    dh = wl.Dims(**{**d.__dict__, "flags": d.flags | wl.QUANT_PER_HEAD})
    inp = wl.make_inputs(wl.Workload("v", d, positions="uniform"))
    tok = _run(oracle_lib, d, inp, taps=True)
    hd = _run(oracle_lib, dh, inp, taps=True)
    assert hd["out_scale"].shape == (d.T, d.num_heads)
    assert np.array_equal(tok["q"], hd["q"])
    for t in range(d.T):
        for h in range(d.num_heads):
            c = hd["out_q_int8"][t, h].astype(int)
            if hd["out_scale"][t, h] > 0:
                assert np.abs(c).max() == 127
        top = int(np.argmax(hd["out_scale"][t]))
        assert hd["out_scale"][t, top] == tok["out_scale"][t]
        assert np.array_equal(hd["out_q_int8"][t, top], tok["out_q_int8"][t, top])


# --------------------------------------------------------- KV-cache scatter

def test_scatter_kv_cache_rows_and_skips(oracle_lib):
    d = _dims(T=6)
    inp = wl.make_inputs(wl.Workload("v", d, positions="uniform"))
    o = _run(oracle_lib, d, inp, taps=True)
    num_slots, W = 16, d.kv_lora_rank + d.rope_dim
    cache = np.full((num_slots, W), 0xBEEF, np.uint16)
    slots = np.array([7, -1, 0, 15, 16, 3], np.int32)
    bad = oracle_lib.scatter_kv_cache(cache, slots, o["normed"], o["out_kpe"], d.q_lora_rank)
    assert bad == 1
    written = {7: 0, 0: 2, 15: 3, 3: 5}
    for s in range(num_slots):
        if s in written:
            j = written[s]
            assert np.array_equal(cache[s, :d.kv_lora_rank], o["normed"][j, d.q_lora_rank:])
            assert np.array_equal(cache[s, d.kv_lora_rank:], o["out_kpe"][j])
        else:
            assert np.all(cache[s] == 0xBEEF)


def test_scatter_kv_cache_against_torch_index_copy(oracle_lib):
    """An independent route to the same cache: torch's index_copy_ of the rows
    [normed c_kv | k_pe_rot] at the valid slots (those in [0, num_slots));
    padding (-1) and out-of-range slots are left out of the index list."""
    d = _dims(T=40)
    inp = wl.make_inputs(wl.Workload("v", d, positions="uniform"))
    o = _run(oracle_lib, d, inp, taps=True)
    num_slots, W = 64, d.kv_lora_rank + d.rope_dim
    rng = np.random.default_rng(5)
    slots = rng.permutation(num_slots + 8)[:d.T].astype(np.int32)  # distinct, some >= num_slots
    slots[rng.choice(d.T, 6, replace=False)] = -1
    cache = np.full((num_slots, W), 0xBEEF, np.uint16)
    bad = oracle_lib.scatter_kv_cache(cache, slots, o["normed"], o["out_kpe"], d.q_lora_rank)
    keep = (slots >= 0) & (slots < num_slots)
    assert bad == int((slots >= num_slots).sum())
    rows = torch.from_numpy(np.concatenate([o["normed"][:, d.q_lora_rank:], o["out_kpe"]], axis=1)
                            .astype(np.int32))
    want = torch.full((num_slots, W), 0xBEEF, dtype=torch.int32)
    want.index_copy_(0, torch.from_numpy(slots[keep].astype(np.int64)), rows[torch.from_numpy(keep)])
    assert np.array_equal(cache.astype(np.int32), want.numpy())
