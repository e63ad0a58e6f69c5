"""GPU parity of the fused prolog against the CPU oracle, through the C ABI.

Small and ragged cases are compared on every element; the full-size
workloads on a seeded sample of tokens that always includes the first and
last token (and, for the long prefill, every token whose x row was scaled
x20).  Tolerances are the parity bar: BF16 outputs |d| <= 1e-2 + 1e-2 |ref|,
scales relative <= 1e-3, INT8 codes differ by <= 1 on <= 0.1% of elements,
and the quant step bit-exact on the oracle's own FP32 q.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import alloc_outputs, bf16_within, device_inputs, quant_within, rope_within, run_prolog
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


def _sample(w: wl.Workload, inp: wl.Inputs, n: int):
    T = inp.dims.T
    if T <= n:
        return None
    rng = np.random.default_rng(7)
    must = {0, T - 1} | set(int(i) for i in inp.boosted_rows)
    n = max(n, len(must) + 16)  # every boosted row, and some others
    if T <= n:
        return None
    rest = rng.choice(np.setdiff1d(np.arange(T), np.array(sorted(must))), n - len(must), replace=False)
    return np.array(sorted(must | set(int(i) for i in rest)), np.int32)


def check_against_oracle(w: wl.Workload, dims=None, sample=512, positions=None, tunings=((),)):
    """Runs the prolog once per entry of `tunings` (each a sequence of
    (tuning key, value) pairs set on one handle, in order) and holds every
    run to the oracle on the same sampled tokens."""
    inp = wl.make_inputs(w, dims)
    if positions is not None:
        inp.positions[:] = positions
    d = inp.dims
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    tok = _sample(w, inp, sample)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok,
                            taps=True)
    sel = slice(None) if tok is None else torch.from_numpy(tok.astype(np.int64)).to(DEV)
    Dn, R, H = d.nope_dim, d.rope_dim, d.num_heads
    n = ref["out_kpe"].shape[0]
    rows = np.arange(d.T) if tok is None else tok
    pos = np.clip(inp.positions[rows], 0, d.max_pos - 1)
    cs = inp.cos_sin[pos]
    kpe_in = ref["c"][:, d.q_lora_rank + d.kv_lora_rank:]
    il = bool(d.flags & wl.ROPE_INTERLEAVED)
    status = 0
    for tune in tunings:
        for key, value in tune:
            p.set_tuning(key, value)
        outs = alloc_outputs(d, DEV)
        run_prolog(p, dins, outs)
        status |= p.device_status()
        # K's nope columns and V to the BF16 bar; the rotated k_pe (K's rope
        # slices, out_kpe) to that bar widened by a one-ulp rounding of its inputs
        k_got = outs["out_k"].t[sel].reshape(n, H, Dn + R)
        k_want = ref["out_k"].reshape(n, H, Dn + R)
        bf16_within(k_got[:, :, :Dn], np.ascontiguousarray(k_want[:, :, :Dn]), f"out_k nope {tune}")
        bf16_within(outs["out_v"].t[sel], ref["out_v"], f"out_v {tune}")
        rope_within(k_got[:, :, Dn:], np.ascontiguousarray(k_want[:, :, Dn:]), kpe_in, cs[:, :R // 2],
                    cs[:, R // 2:], il, f"out_k rope {tune}")
        rope_within(outs["out_kpe"].t[sel], ref["out_kpe"].reshape(n, R), kpe_in, cs[:, :R // 2], cs[:, R // 2:],
                    il, f"out_kpe {tune}")
        if d.q_lora_rank:
            quant_within(outs["out_q_int8"].t[sel], outs["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        for k, g in outs.items():
            assert g.guards_intact(), f"{k}: write outside the buffer"
    p.close()
    return status, ref, outs


@pytest.mark.parametrize("name", ["tiny", "tiny_q", "v2lite_decode", "v2lite_prefill", "v3_decode", "v3_prefill"])
def test_workload_parity(name):
    status, ref, _ = check_against_oracle(wl.WORKLOADS[name])
    assert status == 0 and ref["bad_positions"] == 0


RAGGED = wl.Dims(T=300, D=512, q_lora_rank=64, kv_lora_rank=128, rope_dim=32, num_heads=5,
                 nope_dim=64, v_dim=48, max_pos=512, flags=wl.QUANT_Q)


@pytest.mark.parametrize("dims", [
    RAGGED,                                               # 3 token tiles, ragged tail, q path
    dataclasses.replace(RAGGED, T=1),                     # one token (decode schedule)
    dataclasses.replace(RAGGED, T=129),                   # decode, two tiles, 1-row tail
    dataclasses.replace(RAGGED, T=257, q_lora_rank=0, flags=0),   # prefill, KV only
    dataclasses.replace(RAGGED, T=200, D=1024, kv_lora_rank=512, rope_dim=64, num_heads=3,
                        nope_dim=128, v_dim=128, q_lora_rank=0, flags=0),   # decode, narrow kv tiles
    dataclasses.replace(RAGGED, T=96, D=2048, q_lora_rank=96, rope_dim=16, nope_dim=16, v_dim=16,
                        num_heads=7),                     # narrow heads, Lq not a multiple of 64
    dataclasses.replace(RAGGED, T=40, max_pos=1),         # one rope position: every token at 0, RoPE = identity
    dataclasses.replace(RAGGED, num_heads=1),             # one head
    dataclasses.replace(RAGGED, T=260, D=64),             # the hidden size one K block
], ids=["ragged300q", "T1", "T129", "prefill257", "decode200", "narrow_heads", "max_pos1", "one_head", "D64"])
def test_ragged_parity(dims):
    w = wl.Workload("ragged", dims, positions="uniform")
    status, ref, _ = check_against_oracle(w)
    assert status == 0 and ref["bad_positions"] == 0


def test_v3_prefill_beyond_32bit_offsets():
    """The largest batch tested: the V3 prolog at T = 65536 (4x the
    workload, near its size rule T * H * (Dn + R + Dv) <= 4e9), where the
    FP32 q workspace is 6.4 GB, so byte offsets pass 2^32, and out_k's pass
    2^31 -- every output within the bar of the oracle on sampled tokens up
    to the last one, guard bands intact."""
    w = wl.WORKLOADS["v3_prefill"]
    d = dataclasses.replace(w.dims.with_T(65536), max_pos=65536)
    assert d.T * d.n_q * 4 > 2**32 and d.T * d.num_heads * (d.nope_dim + d.rope_dim) * 2 > 2**31
    status, ref, _ = check_against_oracle(w, dims=d, sample=1024)
    assert status == 0 and ref["bad_positions"] == 0


@pytest.mark.parametrize("name,T", [("v3_decode", 0), ("v3_prefill", 640), ("v2lite_prefill", 300)])
def test_compression_chain_and_drain_settings(name, T):
    """The compression's accumulation chain length (MLA_TUNE_COMPRESS_GROUP:
    1, 2, 4, 8 K blocks) and its drained sums with or without TwoSum
    (MLA_TUNE_COMPRESS_COMPENSATED) change rounding only: every setting
    within the bar of the oracle on every token; out-of-range values are
    refused."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    G, C = binding.TUNE_COMPRESS_GROUP, binding.TUNE_COMPRESS_COMPENSATED
    tunings = [((G, g), (C, c)) for g in (1, 2, 4, 8) for c in (0, 1)]
    status, _, _ = check_against_oracle(w, dims=d, sample=d.T, tunings=tunings)
    assert status == 0
    p = binding.MlaProlog.from_dims(d)
    for key, bad in ((G, 0), (G, 65), (C, 2)):
        with pytest.raises(binding.MlaPrologError):
            p.set_tuning(key, bad)
    p.close()


@pytest.mark.parametrize("name,T", [("v3_prefill", 640), ("v3_decode", 0), ("v2lite_prefill", 300)])
def test_zero_rows_of_x(name, T):
    """Tokens whose x row is all zero: C = 0, so the RMSNorm (eps > 0) gives
    zero rows, K, V and the rotated k_pe are zero, q is zero and its amax 0
    -- codes 0 and scale 0 (the quant step's zero row) -- while the other
    tokens stay within the bar of the oracle."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    inp = wl.make_inputs(w, d)
    zero = np.array([0, 1, d.T // 2, d.T - 1], np.int64)
    x = inp.x.copy()
    x[zero] = 0
    inp = dataclasses.replace(inp, x=x)
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    run_prolog(p, dins, outs)
    assert p.device_status() == 0
    tok = np.unique(np.concatenate([zero, np.linspace(0, d.T - 1, 24).astype(np.int64)])).astype(np.int32)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(outs[k].t[sel], ref[k], k)
        for t in zero:
            assert not outs[k].t[int(t)].float().abs().sum().item(), (k, int(t))
    if d.q_lora_rank:
        quant_within(outs["out_q_int8"].t[sel], outs["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        for t in zero:
            assert not outs["out_q_int8"].t[int(t)].abs().sum().item()
            assert outs["out_scale"].t[int(t)].item() == 0.0
    for k, g in outs.items():
        assert g.guards_intact(), k
    p.close()


def test_out_of_range_positions_zero_fill_and_status():
    d = dataclasses.replace(RAGGED, T=40)
    w = wl.Workload("badpos", d, positions="uniform")
    inp = wl.make_inputs(w)
    pos = inp.positions.copy()
    pos[3] = d.max_pos
    pos[17] = -5
    status, ref, outs = check_against_oracle(w, positions=pos)
    assert status & binding.STATUS_POSITION_RANGE
    assert ref["bad_positions"] == 2
    for t in (3, 17):
        assert not outs["out_k"].t[t].float().abs().sum().item()
        assert not outs["out_q_int8"].t[t].abs().sum().item()
        assert outs["out_scale"].t[t].item() == 0


def test_quant_step_bit_exact_on_oracle_q():
    w = wl.WORKLOADS["v3_decode"]
    inp = wl.make_inputs(w)
    d = inp.dims
    tok = np.arange(0, d.T, 4, dtype=np.int32)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin,
                            tokens=tok, taps=True)
    q = torch.from_numpy(ref["q"]).to(DEV)
    q[1].zero_()  # an all-zero row: codes 0, scale 0
    codes = torch.empty(q.shape, dtype=torch.int8, device=DEV)
    scale = torch.empty(q.shape[0], dtype=torch.float32, device=DEV)
    binding.quant_rows(q, codes, scale)
    torch.cuda.synchronize()
    qh = q.cpu().numpy()
    for i in range(qh.shape[0]):
        c, s = oracle.quant_row(qh[i])
        assert np.array_equal(codes[i].cpu().numpy(), c), i
        assert scale[i].item() == s, i
    assert scale[1].item() == 0.0 and not codes[1].abs().sum().item()


def test_runs_are_deterministic():
    w = wl.WORKLOADS["v3_decode"]
    inp = wl.make_inputs(w)
    d = inp.dims
    dins = device_inputs(inp, DEV)
    a, b = alloc_outputs(d, DEV), alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    run_prolog(p, dins, a)
    run_prolog(p, dins, b)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k].t.view(torch.uint8) if a[k].t.dtype != torch.float32 else a[k].t,
                           b[k].t.view(torch.uint8) if b[k].t.dtype != torch.float32 else b[k].t), k
    p.close()


def test_empty_batch_is_a_no_op():
    d = dataclasses.replace(RAGGED, T=0)
    p = binding.MlaProlog.from_dims(d)
    dins = device_inputs(wl.make_inputs(wl.Workload("e", dataclasses.replace(d, T=1), positions="uniform")), DEV)
    rc = binding.lib().mla_prolog_run(p.handle, *([None] * 12))
    assert rc == 0
    assert p.device_status() == 0
    p.close()
    del dins


def test_bounded_wait_selftest_reports_timeout():
    p = binding.MlaProlog.from_dims(wl.WORKLOADS["tiny"].dims)
    p.selftest_wait_timeout(2_000_000)  # 2 ms
    assert p.device_status() & binding.STATUS_WAIT_TIMEOUT
    # the context stays usable
    check_against_oracle(wl.WORKLOADS["tiny"])
    p.close()


def test_timing_events_hook():
    w = wl.WORKLOADS["v2lite_decode"]
    inp = wl.make_inputs(w)
    d = inp.dims
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    names = p.kernel_names()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
    p.set_timing_events(ev)
    run_prolog(p, dins, outs)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(names))]
    assert all(t >= 0 for t in times)
    p.set_timing_events([])
    p.close()


@pytest.mark.parametrize("name", ["tiny_q", "v2lite_decode", "v3_decode"])
def test_fused_decode_kernel_matches_four_kernels(name):
    """The cooperative decode kernel runs the same arithmetic as the four
    standalone kernels, so their outputs must be bit-identical."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = inp.dims
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    if p.kernel_names()[0] == "mla_compress_norm_kernel":  # the cluster schedule is this size's default
        p.set_tuning(binding.TUNE_CLUSTER_NORM, 0)
    assert p.kernel_names()[0] == "mla_compress_kernel"
    p.set_tuning(binding.TUNE_DECODE_FUSED, 1)
    assert p.kernel_names() == ["mla_decode_kernel"]
    a = alloc_outputs(d, DEV)
    run_prolog(p, dins, a)
    assert p.device_status() == 0
    p.set_tuning(binding.TUNE_DECODE_FUSED, 0)
    assert p.kernel_names()[0] == "mla_compress_kernel"
    b = alloc_outputs(d, DEV)
    run_prolog(p, dins, b)
    assert p.device_status() == 0
    for k in a:
        x, y = a[k].t, b[k].t
        if x.dtype != torch.float32:
            x, y = x.view(torch.uint8), y.view(torch.uint8)
        assert torch.equal(x, y), k
    p.close()


V2L = wl.WORKLOADS["v2lite_decode"]


@pytest.mark.parametrize("T", [1, 17, 64, 100, 128])
def test_cluster_compression_parity(T):
    """The compression and the norm in one thread-block cluster (partials
    summed in distributed shared memory): parity with the oracle at every
    owner split of the tokens, and the same outputs within the bar as the
    split-K path."""
    d = V2L.dims.with_T(T)
    w = wl.Workload("v2l", d, positions="uniform")
    inp = wl.make_inputs(w)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.set_tuning(binding.TUNE_CLUSTER_NORM, 1)
    assert p.kernel_names()[0] == "mla_compress_norm_kernel", p.kernel_names()
    a = alloc_outputs(d, DEV)
    run_prolog(p, dins, a)
    assert p.device_status() == 0
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t, ref[k], k)
        assert a[k].guards_intact(), k
    p.set_tuning(binding.TUNE_CLUSTER_NORM, 0)
    assert p.kernel_names()[0] == "mla_compress_kernel"
    b = alloc_outputs(d, DEV)
    run_prolog(p, dins, b)
    assert p.device_status() == 0
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t, b[k].t.view(torch.int16).cpu().numpy().view(np.uint16), k + " (split-K path)")
    p.set_tuning(binding.TUNE_CLUSTER_NORM, 1)
    c = alloc_outputs(d, DEV)
    run_prolog(p, dins, c)
    torch.cuda.synchronize()
    for k in a:  # deterministic
        assert torch.equal(a[k].t.view(torch.int16), c[k].t.view(torch.int16)), k
    p.close()


def test_cluster_compression_bad_positions():
    d = V2L.dims.with_T(48)
    w = wl.Workload("v2l", d, positions="uniform")
    inp = wl.make_inputs(w)
    inp.positions[7] = d.max_pos
    inp.positions[40] = -3
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.set_tuning(binding.TUNE_CLUSTER_NORM, 1)
    run_prolog(p, dins, outs)
    assert p.device_status() & binding.STATUS_POSITION_RANGE
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    assert ref["bad_positions"] == 2
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(outs[k].t, ref[k], k)
    for t in (7, 40):
        assert not outs["out_k"].t[t].float().abs().sum().item()
    p.close()


@pytest.mark.parametrize("name", ["tiny", "tiny_q"])
def test_cluster_compression_is_the_default_for_tiny_batches(name):
    p = binding.MlaProlog.from_dims(wl.WORKLOADS[name].dims)
    assert p.kernel_names()[0] == "mla_compress_norm_kernel"
    p.close()
    p = binding.MlaProlog.from_dims(V2L.dims)
    assert p.kernel_names()[0] == "mla_compress_kernel"  # split-K measured faster at this size
    p.close()


@pytest.mark.parametrize("name,T,extra", [
    ("v2lite_prefill", 0, 0),
    ("v2lite_prefill", 300, 0),                                      # the odd CTA of the last pair all out of range
    ("v3_prefill", 640, 0),
    ("v3_prefill", 385, wl.ROPE_INTERLEAVED | wl.Q_HEAD_NORM),
], ids=["v2l_full", "v2l_T300", "v3_T640", "v3_T385_variants"])
def test_pair_expansion_matches_single_cta(name, T, extra):
    """Prefill runs the expansion on CTA pairs (tcgen05 cta_group::2, M = 256):
    parity with the oracle, and the same outputs within the bar as the
    one-CTA kernel (the accumulation order per output is the same, so they
    are expected to agree bit for bit)."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    d = dataclasses.replace(d, flags=d.flags | extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    assert p.kernel_names()[2] == ("mla_expand_pair_kernel" if d.q_lora_rank else "mla_expand_kernel")
    p.set_tuning(binding.TUNE_PAIR_EXPAND, 1)
    assert p.kernel_names()[2] == "mla_expand_pair_kernel", p.kernel_names()
    a = alloc_outputs(d, DEV)
    run_prolog(p, dins, a)
    assert p.device_status() == 0
    p.set_tuning(binding.TUNE_PAIR_EXPAND, 0)
    assert p.kernel_names()[2] == "mla_expand_kernel"
    b = alloc_outputs(d, DEV)
    run_prolog(p, dins, b)
    assert p.device_status() == 0
    torch.cuda.synchronize()
    tok = np.unique(np.linspace(0, d.T - 1, min(d.T, 96)).astype(np.int32))
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t[sel], ref[k], k)
        bf16_within(a[k].t, b[k].t.view(torch.int16).cpu().numpy().view(np.uint16), k + " vs one-CTA")
    if d.q_lora_rank:
        quant_within(a["out_q_int8"].t[sel], a["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        quant_within(a["out_q_int8"].t, a["out_scale"].t, b["out_q_int8"].t.cpu().numpy(),
                     b["out_scale"].t.cpu().numpy())
    same = all(torch.equal(a[k].t.view(torch.uint8) if a[k].t.dtype != torch.float32 else a[k].t,
                           b[k].t.view(torch.uint8) if b[k].t.dtype != torch.float32 else b[k].t) for k in a)
    print(f"pair vs one-CTA outputs bit-identical: {same}")
    for k, g in a.items():
        assert g.guards_intact(), k
    p.close()


@pytest.mark.parametrize("name,T", [("v2lite_prefill", 0), ("v2lite_prefill", 300), ("v3_prefill", 640),
                                    ("v3_prefill", 257)], ids=["v2l_full", "v2l_T300", "v3_T640", "v3_T257"])
def test_pair_compression_matches_single_cta(name, T):
    """The compression on CTA pairs (opt-in; M = 256, the odd CTA of a ragged
    last tile has no token rows): parity with the oracle, and the
    outputs within the bar of the one-CTA compression (bit-identical when both
    use the same split-K factor)."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    assert p.kernel_names()[0] == "mla_compress_kernel"  # one CTA per tile measured faster
    p.set_tuning(binding.TUNE_PAIR_COMPRESS, 1)
    assert p.kernel_names()[0] == "mla_compress_pair_kernel", p.kernel_names()
    a = alloc_outputs(d, DEV)
    run_prolog(p, dins, a)
    assert p.device_status() == 0
    p.set_tuning(binding.TUNE_PAIR_COMPRESS, 0)
    assert p.kernel_names()[0] == "mla_compress_kernel"
    b = alloc_outputs(d, DEV)
    run_prolog(p, dins, b)
    assert p.device_status() == 0
    torch.cuda.synchronize()
    tok = np.unique(np.concatenate([np.linspace(0, d.T - 1, min(d.T, 96)).astype(np.int32), inp.boosted_rows[:8]]))
    tok = tok.astype(np.int32)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t[sel], ref[k], k)
        bf16_within(a[k].t, b[k].t.view(torch.int16).cpu().numpy().view(np.uint16), k + " vs one-CTA")
    if d.q_lora_rank:
        quant_within(a["out_q_int8"].t[sel], a["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        quant_within(a["out_q_int8"].t, a["out_scale"].t, b["out_q_int8"].t.cpu().numpy(),
                     b["out_scale"].t.cpu().numpy())
    same = all(torch.equal(a[k].t.view(torch.uint8) if a[k].t.dtype != torch.float32 else a[k].t,
                           b[k].t.view(torch.uint8) if b[k].t.dtype != torch.float32 else b[k].t) for k in a)
    print(f"pair vs one-CTA compression outputs bit-identical: {same}")
    for k, g in a.items():
        assert g.guards_intact(), k
    p.close()


@pytest.mark.parametrize("name,T,extra,pair", [
    ("v2lite_prefill", 0, 0, 0),
    ("v2lite_prefill", 300, 0, 0),                                    # last tile ragged, one warp's rows all past T
    ("v3_prefill", 640, 0, 1),
    ("v3_prefill", 385, wl.ROPE_INTERLEAVED | wl.Q_HEAD_NORM, 1),
    ("v3_prefill", 300, wl.QUANT_PER_HEAD, 1),                        # kv tiles only through the store ring
    ("v3_prefill", 385, 0, 0),                                        # one CTA per tile, q and kv tiles
], ids=["v2l_full", "v2l_T300", "v3_T640", "v3_T385_variants", "v3_T300_per_head", "v3_T385_one_cta"])
def test_tma_store_matches_thread_stores(name, T, extra, pair):
    """The expansion epilogue's bulk tensor stores (the default where the dims
    allow them) write the same bytes as per-thread stores, nothing outside
    the outputs (guard bands intact), and stay within the bar of the oracle."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    d = dataclasses.replace(d, flags=d.flags | extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    if d.q_lora_rank:
        p.set_tuning(binding.TUNE_PAIR_EXPAND, pair)
    outs = []
    for ts in (1, 0):
        p.set_tuning(binding.TUNE_TMA_STORE, ts)
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    a, b = outs
    _bits_equal(a, b)
    tok = np.unique(np.linspace(0, d.T - 1, min(d.T, 64)).astype(np.int32))
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t[sel], ref[k], k)
    if d.q_lora_rank:
        quant_within(a["out_q_int8"].t[sel], a["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
    for o in outs:
        for k, g in o.items():
            assert g.guards_intact(), k
    p.close()


def _bits_equal(a, b):
    for k in a:
        x, y = a[k].t, b[k].t
        if x.dtype != torch.float32:
            x, y = x.view(torch.uint8), y.view(torch.uint8)
        assert torch.equal(x, y), k


@pytest.mark.parametrize("name,T", [("v2lite_prefill", 0), ("v2lite_prefill", 300), ("v3_prefill", 640),
                                    ("v3_prefill", 385)], ids=["v2l_full", "v2l_T300", "v3_T640", "v3_T385"])
def test_compression_tile_widths(name, T):
    """Every compression tile width (128 with TwoSum draining; 144, 192 and
    256 with plain FP32 draining, 144 on the 192-wide kernel, ragged last
    weight tiles) within the bar of the oracle, with the guard bands intact."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    tok = np.unique(np.concatenate([np.linspace(0, d.T - 1, min(d.T, 64)).astype(np.int32), inp.boosted_rows[:8]]))
    tok = tok.astype(np.int32)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    for tile in (128, 144, 192, 256):
        p.set_tuning(binding.TUNE_COMPRESS_TILE, tile)
        assert p.schedule()["bn_a"] == tile
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        torch.cuda.synchronize()
        for k in ("out_k", "out_v", "out_kpe"):
            bf16_within(o[k].t[sel], ref[k], f"{k} (tile {tile})")
        if d.q_lora_rank:
            quant_within(o["out_q_int8"].t[sel], o["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        for k, g in o.items():
            assert g.guards_intact(), k
    with pytest.raises(binding.MlaPrologError):
        p.set_tuning(binding.TUNE_COMPRESS_TILE, 160)
    p.close()


@pytest.mark.parametrize("name", ["v3_decode", "v2lite_decode"])
def test_l2_fetch_keeps_outputs(name):
    """Fetching the expansion weights into L2 during the decode compression
    changes no output bit; prefill handles refuse the switch."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = inp.dims
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    outs = []
    for f in (1, 0):
        p.set_tuning(binding.TUNE_L2_FETCH, f)
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    _bits_equal(outs[0], outs[1])
    for o in outs:
        for k, g in o.items():
            assert g.guards_intact(), k
    p.close()
    q = binding.MlaProlog.from_dims(wl.WORKLOADS["v2lite_prefill"].dims.with_T(300))
    with pytest.raises(binding.MlaPrologError):
        q.set_tuning(binding.TUNE_L2_FETCH, 1)
    q.close()


@pytest.mark.parametrize("T,extra", [(640, 0), (385, wl.ROPE_INTERLEAVED), (0, 0)], ids=["T640", "T385_il", "full"])
def test_wide_q_tiles_match_head_tiles(T, extra):
    """q tiles of 256 columns across head boundaries (CTA pairs, per-token q
    path) give the same bytes as one head per tile, within the bar of the
    oracle, guard bands intact."""
    w = wl.WORKLOADS["v3_prefill"]
    d = w.dims.with_T(T) if T else w.dims
    d = dataclasses.replace(d, flags=d.flags | extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    outs = []
    for f in (1, 0):
        p.set_tuning(binding.TUNE_Q_WIDE, f)
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    _bits_equal(outs[0], outs[1])
    tok = np.unique(np.concatenate([np.linspace(0, d.T - 1, min(d.T, 48)).astype(np.int32), inp.boosted_rows[:4]]))
    tok = tok.astype(np.int32)
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    a = outs[0]
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t[sel], ref[k], k)
    quant_within(a["out_q_int8"].t[sel], a["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
    for o in outs:
        for k, g in o.items():
            assert g.guards_intact(), k
    p.close()
    q = binding.MlaProlog.from_dims(dataclasses.replace(d, flags=d.flags | wl.QUANT_PER_HEAD))
    with pytest.raises(binding.MlaPrologError):
        q.set_tuning(binding.TUNE_Q_WIDE, 1)
    q.close()


@pytest.mark.parametrize("name,T,extra", [("v3_prefill", 640, 0), ("v3_prefill", 385, wl.QUANT_PER_HEAD),
                                          ("v2lite_prefill", 300, 0), ("v2lite_prefill", 0, 0)],
                         ids=["v3_T640", "v3_T385_per_head", "v2l_T300", "v2l_full"])
def test_kv_resident_matches_pair_kernel(name, T, extra):
    """The kv tiles on the kv-resident pair kernel (activations loaded once per
    group of kv tiles) give the same bytes as on the pair expansion kernel,
    within the bar of the oracle, guard bands intact."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    d = dataclasses.replace(d, flags=d.flags | extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.set_tuning(binding.TUNE_PAIR_EXPAND, 1)
    outs = []
    for f in (1, 0):
        p.set_tuning(binding.TUNE_KV_RESIDENT, f)
        names = p.kernel_names()
        assert ("mla_expand_kv_pair_kernel" in names) == bool(f), names
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    _bits_equal(outs[0], outs[1])
    tok = np.unique(np.linspace(0, d.T - 1, min(d.T, 48)).astype(np.int32))
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)
    a = outs[0]
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(a[k].t[sel], ref[k], k)
    if d.q_lora_rank:
        quant_within(a["out_q_int8"].t[sel], a["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
    for o in outs:
        for k, g in o.items():
            assert g.guards_intact(), k
    p.close()


def test_quant_beside_kv_kernel_keeps_outputs():
    """The per-token quant on the side stream beside the kv-resident kernel
    (forked and joined with events, also inside a CUDA graph) writes the same
    bytes as the quant after it, and the caller's stream sees them."""
    w = wl.WORKLOADS["v3_prefill"]
    d = w.dims.with_T(4096)  # enough (token tile, kv group) jobs for the kv-resident kernel
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    assert "mla_expand_kv_pair_kernel" in p.kernel_names(), p.kernel_names()
    outs = []
    for f in (1, 0):
        p.set_tuning(binding.TUNE_QUANT_OVERLAP, f)
        o = alloc_outputs(d, DEV)
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            run_prolog(p, dins, o)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                run_prolog(p, dins, o)
            o["out_q_int8"].t.zero_()
            g.replay()
        st.synchronize()
        assert p.device_status() == 0
        outs.append(o)
    _bits_equal(outs[0], outs[1])
    for o in outs:
        for k, gd in o.items():
            assert gd.guards_intact(), k
    p.close()


@pytest.mark.parametrize("name,T,variant", [("v2lite_prefill", 0, 0), ("v2lite_prefill", 4000, 0),
                                            ("v2lite_prefill", 0, wl.W8A8), ("v3_prefill", 4096, 0),
                                            ("v3_prefill", 0, 0), ("v3_prefill", 4096, wl.W8A8)],
                         ids=["v2l_full", "v2l_T4000", "v2l_w8a8", "v3_T4096", "v3_full", "v3_T4096_w8a8"])
def test_kv_half_tiles_keep_outputs(name, T, variant):
    """The last round of kv jobs as half jobs (MLA_TUNE_KV_HALVES): on the
    KV-only prefill's one-CTA kernel half tiles (128 of 256 columns; 56 of
    512 jobs would otherwise run alone), on the kv-resident pair kernel half
    super-jobs (4 of 8 kv tiles; V3: 36 of 1024) -- the same bytes as whole
    jobs; the key is refused where there is no such round."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    d = dataclasses.replace(d, flags=d.flags | variant)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    if variant & wl.W8A8:
        ww = wl.make_w8a8_weights(w, d)
        p.load_w8a8(torch.from_numpy(ww.W_a).to(DEV), torch.from_numpy(ww.W_b).to(DEV),
                    torch.from_numpy(ww.w_scale).to(DEV))
        dins["W_a"] = dins["W_b"] = None
    outs = []
    for f in (1, 0, 1):
        p.set_tuning(binding.TUNE_KV_HALVES, f)
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    _bits_equal(outs[0], outs[1])
    _bits_equal(outs[0], outs[2])
    for o in outs:
        for k, g in o.items():
            assert g.guards_intact(), k
    p.close()
    q = binding.MlaProlog.from_dims(w.dims.with_T(300))  # 48 jobs: no second round
    with pytest.raises(binding.MlaPrologError):
        q.set_tuning(binding.TUNE_KV_HALVES, 1)
    q.close()


def test_kv_group_sizes_keep_outputs():
    """The kv-resident kernel's super-job size (MLA_TUNE_KV_GROUP: 1, 2, 4,
    8, 16 kv tiles per token tile; the last round's half super-jobs planned
    again for each) writes the same bytes as the default; sizes outside
    1 .. the kv tile count are refused."""
    w = wl.WORKLOADS["v3_prefill"]
    d = w.dims.with_T(4096)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    assert "mla_expand_kv_pair_kernel" in p.kernel_names()
    base = alloc_outputs(d, DEV)
    run_prolog(p, dins, base)
    assert p.device_status() == 0
    for g in (1, 2, 4, 16, 8):
        p.set_tuning(binding.TUNE_KV_GROUP, g)
        for halves in (1, 0):
            try:
                p.set_tuning(binding.TUNE_KV_HALVES, halves)
            except binding.MlaPrologError:
                assert halves == 1  # this group size leaves no short last round
                continue
            o = alloc_outputs(d, DEV)
            run_prolog(p, dins, o)
            torch.cuda.synchronize()
            assert p.device_status() == 0, (g, halves)
            _bits_equal(base, o)
            del o
    n_tiles = d.num_heads * (d.nope_dim + d.v_dim) // 256
    for bad in (0, n_tiles + 1):
        with pytest.raises(binding.MlaPrologError):
            p.set_tuning(binding.TUNE_KV_GROUP, bad)
    p.close()


# Unusual shapes for the prefill paths: smaller ranks, few heads, 64-wide nope
# and value (two heads per 256-column kv tile), ragged token counts.
_ODD_PREFILL = [
    wl.Dims(T=700, D=1024, q_lora_rank=512, kv_lora_rank=256, rope_dim=64, num_heads=8, nope_dim=128,
            v_dim=128, max_pos=4096, flags=wl.QUANT_Q),
    wl.Dims(T=1100, D=768, q_lora_rank=256, kv_lora_rank=512, rope_dim=64, num_heads=16, nope_dim=64,
            v_dim=64, max_pos=4096, flags=wl.QUANT_Q),
]


@pytest.mark.parametrize("d", _ODD_PREFILL, ids=["lkv256_h8", "dn64_h16"])
def test_prefill_paths_on_unusual_shapes(d):
    """Every prefill path on shapes other than the V2-Lite / V3 ones: the
    compression tile widths, one head per q tile vs 256-column q tiles, kv
    tiles on the pair kernel vs resident, the quant after vs beside the kv
    kernel -- each within the bar of the oracle, the expansion variants bit
    for bit equal, guard bands intact."""
    w = wl.Workload("odd", d, positions="uniform", seed=3)
    inp = wl.make_inputs(w)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    tok = np.unique(np.linspace(0, d.T - 1, 40).astype(np.int32))
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)
    sel = torch.from_numpy(tok.astype(np.int64)).to(DEV)

    def run_and_check():
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        torch.cuda.synchronize()
        for k in ("out_k", "out_v", "out_kpe"):
            bf16_within(o[k].t[sel], ref[k], k)
        quant_within(o["out_q_int8"].t[sel], o["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
        for k, g in o.items():
            assert g.guards_intact(), k
        return o

    for tile in (128, 144, 192, 256):
        p.set_tuning(binding.TUNE_COMPRESS_TILE, tile)
        run_and_check()
    p.set_tuning(binding.TUNE_PAIR_EXPAND, 1)
    base = None
    for q_wide, kvres, overlap in ((0, 0, 0), (1, 0, 0), (1, 1, 0), (1, 1, 1), (0, 1, 1)):
        p.set_tuning(binding.TUNE_Q_WIDE, q_wide)
        p.set_tuning(binding.TUNE_KV_RESIDENT, kvres)
        if kvres:
            p.set_tuning(binding.TUNE_QUANT_OVERLAP, overlap)
        o = run_and_check()
        if base is None:
            base = o
        else:
            _bits_equal(base, o)
    p.close()


@pytest.mark.parametrize("name,T", [("v3_prefill", 4096), ("v3_decode", 0), ("v2lite_prefill", 0),
                                    ("v2lite_decode", 0)])
def test_l2_policy_keeps_outputs(name, T):
    """The L2 eviction priorities of the bulk copies (MLA_TUNE_L2_POLICY:
    weights / activations evict last, output stores evict first) change only
    which lines L2 keeps: every policy writes the same bytes; out-of-range
    policies are refused."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    outs = []
    for pol in (0, 1, 2, 4, 7):
        p.set_tuning(binding.TUNE_L2_POLICY, pol)
        o = alloc_outputs(d, DEV)
        run_prolog(p, dins, o)
        assert p.device_status() == 0
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs[1:]:
        _bits_equal(outs[0], o)
    for bad in (-1, 8):
        with pytest.raises(binding.MlaPrologError):
            p.set_tuning(binding.TUNE_L2_POLICY, bad)
    p.close()
