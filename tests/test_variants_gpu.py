"""GPU parity of the prolog's variants against the CPU oracle, through the C ABI.

Variants: interleaved RoPE (QuantRope3D's de-interleave), the per-head q
RMSNorm of the DeepSeek-V4 q path, the per-(token, head) INT8 quant fused
into the expansion kernel, and the latent KV-cache write of
``mla_prolog_run_cached``.  Same bar as the base path: BF16 outputs
|d| <= 1e-2 + 1e-2 |ref|, scales relative <= 1e-3, INT8 codes differ by <= 1
on <= 0.1% of elements; the fused per-head quant is also held bit-exact to
the standalone quant step applied to the kernel's own FP32 q.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import alloc_outputs, bf16_within, device_inputs, quant_within, run_prolog
from mla_attention_prolog_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
IL, HN, PH = wl.ROPE_INTERLEAVED, wl.Q_HEAD_NORM, wl.QUANT_PER_HEAD


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from mla_attention_prolog_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _with_flags(dims: wl.Dims, extra: int) -> wl.Dims:
    return dataclasses.replace(dims, flags=dims.flags | extra)


def _sample(inp: wl.Inputs, n: int):
    T = inp.dims.T
    if T <= n:
        return None
    rng = np.random.default_rng(11)
    must = {0, T - 1} | set(int(i) for i in inp.boosted_rows)
    rest = rng.choice(np.setdiff1d(np.arange(T), np.array(sorted(must))), n - len(must), replace=False)
    return np.array(sorted(must | set(int(i) for i in rest)), np.int32)


def _compare(d, inp, outs, tok):
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok,
                            taps=True)
    sel = slice(None) if tok is None else torch.from_numpy(tok.astype(np.int64)).to(DEV)
    bf16_within(outs["out_k"].t[sel], ref["out_k"], "out_k")
    bf16_within(outs["out_v"].t[sel], ref["out_v"], "out_v")
    bf16_within(outs["out_kpe"].t[sel], ref["out_kpe"], "out_kpe")
    if d.q_lora_rank:
        quant_within(outs["out_q_int8"].t[sel], outs["out_scale"].t[sel], ref["out_q_int8"], ref["out_scale"])
    for k, g in outs.items():
        assert g.guards_intact(), f"{k}: write outside the buffer"
    return ref


def run_variant(w: wl.Workload, extra: int, dims=None, sample=512):
    d = _with_flags(dims or w.dims, extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    run_prolog(p, dins, outs)
    status = p.device_status()
    ref = _compare(d, inp, outs, _sample(inp, sample))
    p.close()
    return status, ref, outs


RAGGED = wl.Dims(T=300, D=512, q_lora_rank=64, kv_lora_rank=128, rope_dim=32, num_heads=5,
                 nope_dim=64, v_dim=48, max_pos=512, flags=wl.QUANT_Q)


@pytest.mark.parametrize("extra", [IL, HN, PH, HN | PH, IL | HN | PH],
                         ids=["interleaved", "head_norm", "per_head", "head_norm+per_head", "all"])
@pytest.mark.parametrize("name", ["tiny_q", "v3_decode"])
def test_q_variants(name, extra):
    status, ref, _ = run_variant(wl.WORKLOADS[name], extra)
    assert status == 0 and ref["bad_positions"] == 0


@pytest.mark.parametrize("name", ["tiny", "v2lite_decode", "v2lite_prefill"])
def test_interleaved_kv_only(name):
    status, ref, _ = run_variant(wl.WORKLOADS[name], IL)
    assert status == 0 and ref["bad_positions"] == 0


def test_all_variants_v3_prefill_sampled():
    """Full-size V3 prefill (16384 tokens) with every q variant; 512 sampled
    tokens, including every x20 row."""
    status, ref, _ = run_variant(wl.WORKLOADS["v3_prefill"], IL | HN | PH)
    assert status == 0 and ref["bad_positions"] == 0


@pytest.mark.parametrize("dims", [
    RAGGED,                                                # prefill, 3 token tiles, ragged tail
    dataclasses.replace(RAGGED, T=129),                    # decode, two tiles
    dataclasses.replace(RAGGED, T=1),                      # one token
    dataclasses.replace(RAGGED, T=96, D=2048, q_lora_rank=96, rope_dim=16, nope_dim=16, v_dim=16,
                        num_heads=7),                      # narrow heads, Lq not a multiple of 64
    dataclasses.replace(RAGGED, T=40, rope_dim=128, nope_dim=64),   # wide rope slice (R > 64)
], ids=["ragged300", "T129", "T1", "narrow_heads", "rope128"])
def test_ragged_variants(dims):
    w = wl.Workload("ragged", dims, positions="uniform")
    status, ref, _ = run_variant(w, IL | HN | PH)
    assert status == 0 and ref["bad_positions"] == 0


def test_bad_positions_with_per_head_quant():
    d = _with_flags(dataclasses.replace(RAGGED, T=40), IL | HN | PH)
    w = wl.Workload("badpos", d, positions="uniform")
    inp = wl.make_inputs(w)
    inp.positions[5] = d.max_pos + 3
    inp.positions[22] = -1
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    run_prolog(p, dins, outs)
    assert p.device_status() & binding.STATUS_POSITION_RANGE
    ref = _compare(d, inp, outs, None)
    assert ref["bad_positions"] == 2
    for t in (5, 22):
        assert not outs["out_q_int8"].t[t].abs().sum().item()
        assert not outs["out_scale"].t[t].abs().sum().item()
    p.close()


@pytest.mark.parametrize("name,extra", [("tiny_q", HN), ("v3_decode", IL | HN), ("v3_decode", 0)])
def test_fused_per_head_quant_bit_exact(name, extra):
    """The per-head quant inside the expansion epilogue equals the standalone
    quant step (mla_prolog_quant_rows) on the same kernel's FP32 q, read from
    a per-token run of the same dims (its q tap), bit for bit."""
    w = wl.WORKLOADS[name]
    d_tok = _with_flags(w.dims, extra)
    d_head = _with_flags(w.dims, extra | PH)
    inp = wl.make_inputs(w, d_tok)
    dins = device_inputs(inp, DEV)
    p_tok = binding.MlaProlog.from_dims(d_tok)
    o_tok = alloc_outputs(d_tok, DEV)
    run_prolog(p_tok, dins, o_tok)
    q = p_tok.tap(binding.TAP_Q)
    p_head = binding.MlaProlog.from_dims(d_head)
    o_head = alloc_outputs(d_head, DEV)
    run_prolog(p_head, dins, o_head)
    H, HD = d_head.num_heads, d_head.nope_dim + d_head.rope_dim
    rows = q.view(d_tok.T * H, HD).contiguous()
    codes = torch.empty(rows.shape, dtype=torch.int8, device=DEV)
    scale = torch.empty(rows.shape[0], dtype=torch.float32, device=DEV)
    binding.quant_rows(rows, codes, scale)
    torch.cuda.synchronize()
    assert p_tok.device_status() == 0 and p_head.device_status() == 0
    assert torch.equal(o_head["out_q_int8"].t.reshape(-1, HD), codes)
    assert torch.equal(o_head["out_scale"].t.reshape(-1), scale)
    # the K / V outputs do not depend on the quant granularity
    for k in ("out_k", "out_v", "out_kpe"):
        assert torch.equal(o_head[k].t.view(torch.int16), o_tok[k].t.view(torch.int16)), k
    with pytest.raises(binding.MlaPrologError):
        p_head.tap(binding.TAP_Q)
    p_tok.close()
    p_head.close()


@pytest.mark.parametrize("name,extra", [("tiny_q", IL | HN | PH), ("v3_decode", IL | HN | PH),
                                        ("v2lite_decode", IL)])
def test_fused_decode_kernel_matches_four_kernels(name, extra):
    w = wl.WORKLOADS[name]
    d = _with_flags(w.dims, extra)
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    p = binding.MlaProlog.from_dims(d)
    p.set_tuning(binding.TUNE_DECODE_FUSED, 1)   # also turns the cluster compression off
    a = alloc_outputs(d, DEV)
    run_prolog(p, dins, a)
    assert p.device_status() == 0
    p.set_tuning(binding.TUNE_DECODE_FUSED, 0)
    b = alloc_outputs(d, DEV)
    run_prolog(p, dins, b)
    assert p.device_status() == 0
    for k in a:
        x, y = a[k].t, b[k].t
        if x.dtype != torch.float32:
            x, y = x.view(torch.uint8), y.view(torch.uint8)
        assert torch.equal(x, y), k
    p.close()


# ------------------------------------------------------------ latent KV cache

CACHE_SENTINEL = 0x7FB3  # a NaN pattern no kernel writes


def _slots(T: int, num_slots: int, seed: int) -> np.ndarray:
    """Distinct slots for most tokens, -1 (padding) for a few."""
    rng = np.random.default_rng(seed)
    s = rng.choice(num_slots, T, replace=False).astype(np.int32)
    s[rng.random(T) < 0.1] = -1
    return s


def run_cached(d, inp, slots: np.ndarray, num_slots: int, fused: bool = False, cluster: bool = False):
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    cache = torch.full((num_slots, d.kv_lora_rank + d.rope_dim), CACHE_SENTINEL, dtype=torch.int16,
                       device=DEV).view(torch.bfloat16)
    slot_t = torch.from_numpy(slots).to(DEV)
    p = binding.MlaProlog.from_dims(d)
    if fused:
        p.set_tuning(binding.TUNE_DECODE_FUSED, 1)
    if cluster:
        p.set_tuning(binding.TUNE_CLUSTER_NORM, 1)
    p.run_cached(dins["x"], dins["gamma"], dins["W_a"], dins["W_b"], dins["positions"], dins["cos_sin"],
                 outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t,
                 outs["out_q_int8"].t if "out_q_int8" in outs else None,
                 outs["out_scale"].t if "out_scale" in outs else None, slot_t, cache)
    status = p.device_status()
    normed = p.tap(binding.TAP_NORMED)
    torch.cuda.synchronize()
    # the same outputs as a run without the cache
    plain = alloc_outputs(d, DEV)
    run_prolog(p, dins, plain)
    torch.cuda.synchronize()
    for k in outs:
        x, y = outs[k].t, plain[k].t
        if x.dtype != torch.float32:
            x, y = x.view(torch.uint8), y.view(torch.uint8)
        assert torch.equal(x, y), k
    p.close()
    return status, outs, cache, normed


def check_cache(d, inp, slots, cache, outs, normed):
    """Written rows: the oracle's normed c_kv | k_pe_rot within the BF16 bar and
    the kernel's own normed row and out_kpe bit for bit; other rows untouched."""
    num_slots = cache.shape[0]
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, taps=True)
    want = np.full((num_slots, d.kv_lora_rank + d.rope_dim), CACHE_SENTINEL, np.uint16)
    bad = oracle.scatter_kv_cache(want, slots, ref["normed"], ref["out_kpe"], d.q_lora_rank)
    got = cache.view(torch.int16).cpu().numpy().view(np.uint16)
    written = np.array(sorted(set(int(s) for s in slots if 0 <= s < num_slots)), np.int64)
    untouched = np.setdiff1d(np.arange(num_slots), written)
    assert np.all(got[untouched] == CACHE_SENTINEL)
    if len(written):
        bf16_within(cache[torch.from_numpy(written).to(DEV)], want[written], "kv_cache")
    own = torch.cat([normed[:, d.q_lora_rank:], outs["out_kpe"].t], dim=1).view(torch.int16).cpu().numpy()
    for t, s in enumerate(slots):
        if 0 <= s < num_slots:
            assert np.array_equal(got[s].view(np.int16), own[t]), t
    return bad


@pytest.mark.parametrize("dims", [
    RAGGED,                                                # prefill norm kernel (warp per token)
    dataclasses.replace(RAGGED, T=129),                    # decode norm kernel (split-K)
    dataclasses.replace(RAGGED, T=77, q_lora_rank=0, flags=0),   # KV only
], ids=["prefill300", "decode129", "kv_only77"])
@pytest.mark.parametrize("extra", [0, IL], ids=["rotate_half", "interleaved"])
def test_kv_cache_write(dims, extra):
    d = _with_flags(dims, extra)
    inp = wl.make_inputs(wl.Workload("cache", d, positions="uniform"), d)
    num_slots = 2 * d.T + 13
    slots = _slots(d.T, num_slots, 3)
    status, outs, cache, normed = run_cached(d, inp, slots, num_slots)
    assert status == 0
    assert check_cache(d, inp, slots, cache, outs, normed) == 0


@pytest.mark.parametrize("name", ["v2lite_decode", "v3_decode", "tiny_q"])
def test_kv_cache_write_workloads(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = inp.dims
    num_slots = 4 * d.T
    slots = _slots(d.T, num_slots, 5)
    status, outs, cache, normed = run_cached(d, inp, slots, num_slots)
    assert status == 0
    check_cache(d, inp, slots, cache, outs, normed)


@pytest.mark.parametrize("name", ["tiny_q", "v3_decode"])
def test_kv_cache_write_fused_decode_kernel(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = inp.dims
    num_slots = 3 * d.T
    slots = _slots(d.T, num_slots, 9)
    status, outs, cache, normed = run_cached(d, inp, slots, num_slots, fused=True)
    assert status == 0
    check_cache(d, inp, slots, cache, outs, normed)


def test_kv_cache_slot_range_and_bad_positions():
    d = dataclasses.replace(RAGGED, T=50)
    inp = wl.make_inputs(wl.Workload("cache", d, positions="uniform"), d)
    num_slots = 64
    slots = _slots(d.T, num_slots, 21)
    slots[4] = num_slots          # past the cache: skipped, reported
    slots[9] = num_slots + 1000
    inp.positions[12] = d.max_pos  # a bad position writes a zero row
    if slots[12] < 0:
        slots[12] = next(s for s in range(num_slots) if s not in set(slots.tolist()))
    status, outs, cache, normed = run_cached(d, inp, slots, num_slots)
    assert status & binding.STATUS_SLOT_RANGE
    assert status & binding.STATUS_POSITION_RANGE
    assert check_cache(d, inp, slots, cache, outs, normed) == 2
    assert not cache[int(slots[12])].float().abs().sum().item()


def test_kv_cache_empty_batch_and_bad_arguments():
    d = dataclasses.replace(RAGGED, T=0)
    p = binding.MlaProlog.from_dims(d)
    cache = torch.zeros((4, d.kv_lora_rank + d.rope_dim), dtype=torch.bfloat16, device=DEV)
    slots = torch.zeros((1,), dtype=torch.int32, device=DEV)
    L = binding.lib()
    assert L.mla_prolog_run_cached(p.handle, *([None] * 11), slots.data_ptr(), cache.data_ptr(), 4, None) == 0
    # null cache / null slots / negative size are rejected before any launch
    assert L.mla_prolog_run_cached(p.handle, *([None] * 11), slots.data_ptr(), None, 4, None) == -1
    assert L.mla_prolog_run_cached(p.handle, *([None] * 11), None, cache.data_ptr(), 4, None) == -1
    assert L.mla_prolog_run_cached(p.handle, *([None] * 11), slots.data_ptr(), cache.data_ptr(), -1, None) == -1
    assert p.device_status() == 0
    p.close()


@pytest.mark.parametrize("extra", [0, IL], ids=["rotate_half", "interleaved"])
def test_kv_cache_write_cluster_compression(extra):
    """The cache rows written by the cluster kernel's norm groups."""
    w = wl.WORKLOADS["v2lite_decode"]
    d = _with_flags(w.dims, extra)
    inp = wl.make_inputs(w, d)
    num_slots = 3 * d.T
    slots = _slots(d.T, num_slots, 13)
    status, outs, cache, normed = run_cached(d, inp, slots, num_slots, cluster=True)
    assert status == 0
    check_cache(d, inp, slots, cache, outs, normed)
    _compare(d, inp, outs, None)
