"""GPU parity of the W8A8 prolog (MLA_PROLOG_W8A8) against the oracle.

What is integer work, or FP32 work on exact integers in the same order on
both sides, is compared bit for bit: x's per-token codes and scales and the
rotated k_pe (from the exactly dequantised compression).  The normed rows
come out of an FP32 sum of squares whose order differs between the two
sides (the BF16 mode's RMSNorm), so their codes may differ by one: they are
held to the INT8 bar (<= 1 on <= 0.1 %), and at least 95 % of the tokens must
carry exactly the oracle's codes.  From there on every token is checked step
for step: the oracle, fed the kernel's own normed codes and scales, must give
K, V, the q codes and the q scales bit for bit.  The outputs are also held to
the parity bar against the oracle's own results (K and V for every token;
the INT8 codes and scales for the tokens that carry the oracle's normed
codes).  A deterministic case with every code at +-127 checks the
integer products at their largest magnitudes (past 2^24 in one chain).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import alloc_outputs, bf16_within, device_inputs, quant_within
from mla_attention_prolog_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from mla_attention_prolog_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _w8(name, T=None, **over):
    w = wl.WORKLOADS[name]
    d = dataclasses.replace(w.dims, flags=w.dims.flags | wl.W8A8, **over)
    return w, (d.with_T(T) if T else d)


def _run_gpu(d, inp, ww, cache=None):
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.load_w8a8(torch.from_numpy(ww.W_a).to(DEV), torch.from_numpy(ww.W_b).to(DEV),
                torch.from_numpy(ww.w_scale).to(DEV))
    args = (dins["x"], dins["gamma"], None, None, dins["positions"], dins["cos_sin"],
            outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t,
            outs["out_q_int8"].t if "out_q_int8" in outs else None,
            outs["out_scale"].t if "out_scale" in outs else None)
    if cache is None:
        p.run(*args)
    else:
        p.run_cached(*args, cache[0], cache[1])
    status = p.device_status()
    taps = {
        "x_codes": p.tap(binding.TAP_X_CODES).float().cpu().numpy(),
        "x_scale": p.tap(binding.TAP_X_SCALE).cpu().numpy(),
        "n_codes": p.tap(binding.TAP_NORMED).float().cpu().numpy(),
        "n_scale": p.tap(binding.TAP_NORM_SCALE).cpu().numpy(),
    }
    names = p.kernel_names()
    p.close()
    for k, g in outs.items():
        assert g.guards_intact(), f"{k}: write outside the buffer"
    return status, outs, taps, names


def _sample(T, n, seed=7):
    if T <= n:
        return None
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.arange(1, T - 1), n - 2, replace=False)
    return np.array(sorted({0, T - 1} | set(int(i) for i in rest)), np.int32)


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else \
        t.cpu().numpy()


def check_w8a8(d, inp, ww, sample=384):
    status, outs, taps, names = _run_gpu(d, inp, ww)
    assert names[0] == "mla_quant_x_kernel"
    tok = _sample(d.T, sample)
    ref = oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin,
                                 tokens=tok, taps=True)
    rows = np.arange(d.T) if tok is None else tok
    sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
    # x's codes and scales: bit-exact
    assert np.array_equal(taps["x_codes"][rows], ref["x_codes"].astype(np.float32))
    assert np.array_equal(taps["x_scale"][rows], ref["x_scale"])
    # rotated k_pe: from the exact compression, same FP32 RoPE -> bit-exact
    assert np.array_equal(_bits(outs["out_kpe"].t[sel]), ref["out_kpe"])
    # normed-row codes against the oracle's own: the RMSNorm's FP32 sum of
    # squares runs in another order, which may move a BF16 normed value by an
    # ulp and its code by one -- held to the INT8 bar (<= 1 on <= 0.1 %), the
    # scale to one BF16 ulp of the row's largest magnitude
    nc, nref = taps["n_codes"][rows], ref["n_codes"].astype(np.float32)
    dq = np.abs(nc - nref)
    assert dq.max() <= 1 and (dq > 0).mean() <= 1e-3, (dq.max(), (dq > 0).mean())
    ns = taps["n_scale"][rows]
    rel = np.abs(ns - ref["n_scale"]) / np.maximum(ref["n_scale"], 1e-30)
    assert np.all(rel <= 2.0 ** -7), rel.max()
    same = np.all(nc == nref, axis=1) & np.all(ns == ref["n_scale"], axis=1)
    assert same.mean() >= 0.95, f"only {same.mean():.3f} of the tokens have the oracle's normed codes"
    # every token, step for step from the kernel's own normed codes: the
    # integer products, AT-06, RoPE, split / assemble and the q quant are
    # then the same FP32 work in the same order on both sides -> bit-exact
    given = oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin,
                                   tokens=tok, given_codes=nc.astype(np.int8), given_scale=ns)
    ok_k, ok_v = _bits(outs["out_k"].t[sel]), _bits(outs["out_v"].t[sel])
    assert np.array_equal(ok_k, given["out_k"])
    assert np.array_equal(ok_v, given["out_v"])
    # and against the oracle's own results: K and V within the BF16 bar for
    # every token; q within the INT8 bar for the tokens that carry the
    # oracle's own normed codes (a token with a legitimately different normed
    # row has another, equally valid q row -- one normed code moves a head's
    # largest |q|, and so a per-head scale, by up to ~1e-3 -- and is held to
    # the step-for-step check above instead)
    bf16_within(outs["out_k"].t[sel], ref["out_k"], "out_k")
    bf16_within(outs["out_v"].t[sel], ref["out_v"], "out_v")
    if d.q_lora_rank:
        qc, qs = outs["out_q_int8"].t[sel], outs["out_scale"].t[sel]
        assert np.array_equal(qc.cpu().numpy(), given["out_q_int8"])
        assert np.array_equal(qs.cpu().numpy(), given["out_scale"])
        keep = torch.from_numpy(same).to(DEV)
        quant_within(qc[keep], qs[keep], ref["out_q_int8"][same], ref["out_scale"][same])
    return status, outs, ref, same


@pytest.mark.parametrize("name,T", [("tiny", 0), ("tiny_q", 0), ("v2lite_decode", 0), ("v2lite_prefill", 0),
                                    ("v3_decode", 0), ("v3_decode", 200), ("v3_prefill", 1000),
                                    ("v3_prefill", 0)])
def test_w8a8_parity(name, T):
    w, d = _w8(name, T)
    inp = wl.make_inputs(w, d)
    ww = wl.make_w8a8_weights(w, d)
    status, _, _, same = check_w8a8(d, inp, ww, sample=256 if d.T > 4096 else 384)
    print(f"{name} T={d.T}: {same.mean():.3f} of the tokens bit-exact end to end")
    assert status == 0


@pytest.mark.parametrize("name,T", [("v3_decode", 0), ("v2lite_prefill", 300)])
def test_w8a8_zero_rows_of_x(name, T):
    """Tokens whose x row is zero: AT-05 gives scale 0 and codes 0, so the
    compression, the normed rows and their codes (scale 0), K, V, k_pe and
    q are zero -- every token compared with the oracle as in the parity
    test, and the zero tokens' outputs exactly zero."""
    w, d = _w8(name, T)
    inp = wl.make_inputs(w, d)
    zero = [0, d.T // 2, d.T - 1]
    x = inp.x.copy()
    x[zero] = 0
    inp = dataclasses.replace(inp, x=x)
    ww = wl.make_w8a8_weights(w, d)
    status, outs, ref, _ = check_w8a8(d, inp, ww, sample=384)
    assert status == 0
    for t in zero:
        for k in ("out_k", "out_v", "out_kpe"):
            assert not outs[k].t[t].float().abs().sum().item(), (k, t)
        if d.q_lora_rank:
            assert not outs["out_q_int8"].t[t].abs().sum().item()
            assert outs["out_scale"].t[t].item() == 0.0


@pytest.mark.parametrize("extra", [wl.ROPE_INTERLEAVED, wl.QUANT_PER_HEAD, wl.Q_HEAD_NORM])
def test_w8a8_q_variants(extra):
    w, d = _w8("v3_prefill", 300)
    d = dataclasses.replace(d, flags=d.flags | extra)
    inp = wl.make_inputs(w, d)
    same = check_w8a8(d, inp, wl.make_w8a8_weights(w, d))[3]
    print(f"variant {extra}: {same.mean():.3f} of the tokens bit-exact end to end")


@pytest.mark.parametrize("over", [dict(nope_dim=32, num_heads=8, D=1024, q_lora_rank=512, kv_lora_rank=256),
                                  dict(nope_dim=64, rope_dim=32, v_dim=64, num_heads=16, D=2048)],
                         ids=["dn32_r64", "dn64_r32"])
def test_w8a8_unusual_shapes(over):
    """Heads whose nope part is narrower than the rope slice (the q epilogue
    then reads across the warps' column halves) and narrow heads."""
    w, d = _w8("v3_prefill", 300, **over)
    inp = wl.make_inputs(w, d)
    check_w8a8(d, inp, wl.make_w8a8_weights(w, d))


@pytest.mark.parametrize("T", [130, 300])
def test_w8a8_largest_codes_are_exact(T):
    """Every code +-127 (x rows constant, every weight code 127, gamma 1):
    the compression sums D 127^2 = 115,612,672 and the q expansion
    Lq 127^2 = 24,774,144, past 2^24, so one FP32 accumulation chain would
    round; the weight scales make the compression 2^26 exactly, so the norm
    gives exactly 1.0 whatever its sum order, and every output is fixed."""
    w, d = _w8("v3_prefill", T, num_heads=4, max_pos=T)
    inp = wl.make_inputs(w, d)
    x = np.full((d.T, d.D), 127.0, np.float32)
    x[1::2] *= -1.0  # sign per row: codes +-127, x scale 1
    bits = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    one = np.full_like(inp.gamma, 0x3F80)  # BF16 1.0
    inp = dataclasses.replace(inp, x=bits, gamma=one)
    ww = wl.make_w8a8_weights(w, d)
    s = np.float32(2.0 ** 26 / (d.D * 127 * 127))
    ww = dataclasses.replace(ww, W_a=np.full_like(ww.W_a, 127), W_b=np.full_like(ww.W_b, 127),
                             w_scale=np.full_like(ww.w_scale, s))
    status, outs, taps, _ = _run_gpu(d, inp, ww)
    ref = oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin,
                                 taps=True)
    assert np.all(np.abs(ref["n_codes"]) == 127)
    assert np.array_equal(taps["n_codes"], ref["n_codes"].astype(np.float32))
    assert np.array_equal(taps["n_scale"], ref["n_scale"])
    for k in ("out_k", "out_v", "out_kpe"):
        assert np.array_equal(_bits(outs[k].t), ref[k]), k
    assert np.array_equal(outs["out_q_int8"].t.cpu().numpy(), ref["out_q_int8"])
    assert np.array_equal(outs["out_scale"].t.cpu().numpy(), ref["out_scale"])
    assert status == 0


def test_w8a8_cache_and_bad_positions():
    w, d = _w8("v3_decode", 64)
    inp = wl.make_inputs(w, d)
    inp.positions[3] = d.max_pos
    inp.positions[9] = -1
    ww = wl.make_w8a8_weights(w, d)
    slots = torch.arange(d.T, dtype=torch.int32, device=DEV).flip(0)
    cache = torch.zeros((d.T + 5, d.kv_lora_rank + d.rope_dim), dtype=torch.bfloat16, device=DEV)
    status, outs, taps, _ = _run_gpu(d, inp, ww, cache=(slots, cache))
    assert status & binding.STATUS_POSITION_RANGE
    ref = oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions, inp.cos_sin,
                                 taps=True)
    for t in (3, 9):
        assert torch.count_nonzero(outs["out_k"].t[t]) == 0 and np.all(taps["n_scale"][t] == 0)
    want = np.zeros((d.T + 5, d.kv_lora_rank + d.rope_dim), np.uint16)
    oracle.scatter_kv_cache(want, slots.cpu().numpy(), ref["normed"], ref["out_kpe"], d.q_lora_rank)
    bf16_within(cache, want, "kv_cache")


def test_w8a8_run_needs_loaded_weights_and_null_pointers():
    w, d = _w8("tiny")
    p = binding.MlaProlog.from_dims(d)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    with pytest.raises(binding.MlaPrologError):  # nothing loaded yet
        p.run(dins["x"], dins["gamma"], None, None, dins["positions"], dins["cos_sin"],
              outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t)
    with pytest.raises(ValueError):  # BF16 weights on a W8A8 handle
        p.run(dins["x"], dins["gamma"], dins["W_a"], dins["W_b"], dins["positions"], dins["cos_sin"],
              outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t)
    d16 = dataclasses.replace(d, flags=0)
    p16 = binding.MlaProlog.from_dims(d16)
    ww = wl.make_w8a8_weights(w, d)
    with pytest.raises(binding.MlaPrologError):  # not a W8A8 handle
        p16.load_w8a8(torch.from_numpy(ww.W_a).to(DEV), torch.from_numpy(ww.W_b).to(DEV),
                      torch.from_numpy(ww.w_scale).to(DEV))
    p.close()
    p16.close()


@pytest.mark.parametrize("T", [1000, 4096])
def test_w8a8_kv_resident_matches_pair_kernel(T):
    """The W8A8 kv tiles on the kv-resident pair kernel (normed c_kv codes
    resident, one exact chain, each warp dequantising the columns it stores)
    give the same bytes as on the pair expansion kernel; the quant beside
    the kv kernel too."""
    w, d = _w8("v3_prefill", T)
    inp = wl.make_inputs(w, d)
    ww = wl.make_w8a8_weights(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.load_w8a8(torch.from_numpy(ww.W_a).to(DEV), torch.from_numpy(ww.W_b).to(DEV),
                torch.from_numpy(ww.w_scale).to(DEV))
    got = []
    for kvres, overlap in ((0, 0), (1, 0), (1, 1)):
        p.set_tuning(binding.TUNE_KV_RESIDENT, kvres)
        p.set_tuning(binding.TUNE_QUANT_OVERLAP, overlap)
        assert ("mla_expand_kv_pair_kernel" in p.kernel_names()) == bool(kvres)
        outs = alloc_outputs(d, DEV)
        p.run(dins["x"], dins["gamma"], None, None, dins["positions"], dins["cos_sin"],
              outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t, outs["out_q_int8"].t, outs["out_scale"].t)
        assert p.device_status() == 0
        for k, g in outs.items():
            assert g.guards_intact(), k
        got.append({k: _bits(g.t) for k, g in outs.items()})
    p.close()
    for other in got[1:]:
        for k in got[0]:
            assert np.array_equal(got[0][k], other[k]), k
