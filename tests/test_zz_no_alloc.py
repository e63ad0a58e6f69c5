"""GPU tests of mla_prolog_run_noalloc, the entry point for callers that cannot
call cudaMalloc (e.g. a plugin inside an inference runtime that reserves the
device memory pool up front, or a caller that cannot accept cudaMalloc's
implicit device synchronisation).  It runs the whole prolog with its scratch
in a static device array of the library.  Its outputs must equal those of the
handle-based mla_prolog_run() on the same inputs, call after call: bit for
bit where both launch the same kernels, within the parity bar where the
handle picks other kernels (the cluster compression of tiny batches).  The
small q-path case is also held to the CPU oracle, and a bad position must
show in the status word of that call only.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import alloc_outputs, bf16_within, device_inputs, quant_within, run_prolog
from mla_attention_prolog_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
SCRATCH_BYTES = 32 << 20  # the static scratch array's size


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from mla_attention_prolog_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _cdims(d):
    return binding.MlaPrologDims(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads,
                                 d.nope_dim, d.v_dim, d.max_pos, d.eps, d.flags)


def _noalloc(d, dins, outs, status):
    dims = _cdims(d)
    ptr = lambda k: outs[k].t.data_ptr() if k in outs else None
    return binding.lib().mla_prolog_run_noalloc(
        ctypes.byref(dims), dins["x"].data_ptr(), dins["gamma"].data_ptr(), dins["W_a"].data_ptr(),
        dins["W_b"].data_ptr(), dins["positions"].data_ptr(), dins["cos_sin"].data_ptr(),
        ptr("out_k"), ptr("out_v"), ptr("out_kpe"), ptr("out_q_int8"), ptr("out_scale"),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _scratch_need(d, sms):
    """Bytes of scratch the entry point needs for dims d (the handle's
    workspace blocks, each rounded up to 256 bytes)."""
    al = lambda b: (b + 255) & ~255
    p = binding.plan(d, sms)
    NQ = d.num_heads * (d.nope_dim + d.rope_dim)
    return (al(p["splits_a"] * d.T * d.n_a * 4) + al(d.T * (d.q_lora_rank + d.kv_lora_rank) * 2) +
            (al(d.T * NQ * 4) if d.q_lora_rank else 0) + al(d.T * 4) + 256)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _case(name, T=None, **over):
    w = wl.WORKLOADS[name]
    d = w.dims if T is None else w.dims.with_T(T)
    if over:
        d = dataclasses.replace(d, **over)
    return w, d


# (workload, T, extra dims, bit-exact against mla_prolog_run)
CASES = [
    ("tiny_q", None, {}, False),              # the handle runs the cluster compression here
    ("tiny", 512, {"max_pos": 512}, True),    # prefill schedule on a tiny shape
    ("v2lite_decode", None, {}, True),
    ("v2lite_prefill", 300, {}, True),         # prefill schedule with split-K
    ("v2lite_prefill", None, {}, True),        # the full V2-Lite prefill, T = 4096
    ("v3_decode", None, {}, True),
    ("v3_decode", 246, {}, True),              # two token tiles, the largest V3 batch that fits
]


@pytest.mark.parametrize("name,T,over,exact", CASES,
                         ids=[f"{c[0]}-T{c[1] or 'cfg'}" for c in CASES])
def test_noalloc_matches_run_on_two_calls(name, T, over, exact):
    w, d = _case(name, T, **over)
    if _scratch_need(d, _sms()) > SCRATCH_BYTES:
        pytest.skip("does not fit the static scratch on this device's SM count")
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    ref = alloc_outputs(d, DEV)
    p = binding.MlaProlog.from_dims(d)
    run_prolog(p, dins, ref)
    assert p.device_status() == 0
    p.close()
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for call in range(2):
        outs = alloc_outputs(d, DEV)
        assert _noalloc(d, dins, outs, status) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert status.item() == 0
        for k in ("out_k", "out_v", "out_kpe"):
            if exact:
                assert np.array_equal(_bits(outs[k].t), _bits(ref[k].t)), f"{k} (call {call})"
            else:
                bf16_within(outs[k].t, _bits(ref[k].t), f"{k} (call {call})")
        if d.q_lora_rank:
            if exact:
                assert torch.equal(outs["out_q_int8"].t, ref["out_q_int8"].t), f"q codes (call {call})"
                assert torch.equal(outs["out_scale"].t, ref["out_scale"].t), f"q scales (call {call})"
            else:
                quant_within(outs["out_q_int8"].t, outs["out_scale"].t,
                             ref["out_q_int8"].t.cpu().numpy(), ref["out_scale"].t.cpu().numpy())
        for k, g in outs.items():
            assert g.guards_intact(), k


def test_noalloc_tiny_q_against_the_oracle():
    w, d = _case("tiny_q")
    inp = wl.make_inputs(w, d)
    dins = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    assert _noalloc(d, dins, outs, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin)
    for k in ("out_k", "out_v", "out_kpe"):
        bf16_within(outs[k].t, ref[k], k)
    quant_within(outs["out_q_int8"].t, outs["out_scale"].t, ref["out_q_int8"], ref["out_scale"])


def test_noalloc_status_word_is_per_call():
    """A position outside the table sets MLA_STATUS_POSITION_RANGE and
    zero-fills that token's outputs; the next call, with good positions,
    starts from a clear status word (the shared scratch is reset per call)."""
    w, d = _case("tiny_q")
    inp = wl.make_inputs(w, d)
    bad = inp.positions.copy()
    bad[1] = d.max_pos
    dins = device_inputs(dataclasses.replace(inp, positions=bad), DEV)
    outs = alloc_outputs(d, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    assert _noalloc(d, dins, outs, status) == 0
    torch.cuda.synchronize()
    assert status.item() == binding.STATUS_POSITION_RANGE
    for k in ("out_k", "out_v", "out_kpe", "out_q_int8"):
        assert torch.count_nonzero(outs[k].t[1]) == 0, k
        assert torch.count_nonzero(outs[k].t[0]) > 0, k
    assert outs["out_scale"].t[1].item() == 0.0
    good = device_inputs(inp, DEV)
    outs = alloc_outputs(d, DEV)
    assert _noalloc(d, good, outs, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 0


@pytest.mark.parametrize("name,T", [("v3_prefill", None), ("v3_decode", 256), ("v3_decode", 247),
                                    ("v2lite_prefill", 12288)])
def test_noalloc_rejects_dims_beyond_its_scratch(name, T):
    w, d = _case(name, T)
    if _scratch_need(d, _sms()) <= SCRATCH_BYTES:
        pytest.skip("fits the static scratch on this device's SM count")
    dims = _cdims(d)
    rc = binding.lib().mla_prolog_run_noalloc(ctypes.byref(dims), *([None] * 12), None)
    assert rc == -2  # MLA_ERR_UNSUPPORTED_DIMS: its workspace exceeds the static scratch
