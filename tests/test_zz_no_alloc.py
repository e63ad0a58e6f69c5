"""GPU test of mla_prolog_run_noalloc, the entry point for callers that cannot
call cudaMalloc (e.g. a plugin inside an inference runtime that reserves the
device memory pool up front).  It runs the whole prolog with its scratch in a
static device array of the library, and must give the outputs of the
handle-based mla_prolog_run() on the same inputs, call after call.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import alloc_outputs, bf16_within, device_inputs, quant_within, run_prolog
from mla_attention_prolog_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    from mla_attention_prolog_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _noalloc(d, dins, outs, status):
    dims = binding.MlaPrologDims(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads,
                                 d.nope_dim, d.v_dim, d.max_pos, d.eps, d.flags)
    ptr = lambda k: outs[k].t.data_ptr() if k in outs else None
    return binding.lib().mla_prolog_run_noalloc(
        ctypes.byref(dims), dins["x"].data_ptr(), dins["gamma"].data_ptr(), dins["W_a"].data_ptr(),
        dins["W_b"].data_ptr(), dins["positions"].data_ptr(), dins["cos_sin"].data_ptr(),
        ptr("out_k"), ptr("out_v"), ptr("out_kpe"), ptr("out_q_int8"), ptr("out_scale"),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["tiny_q", "v2lite_decode", "v3_decode"])
def test_noalloc_matches_run_on_two_calls(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = inp.dims
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
            bf16_within(outs[k].t, _bits(ref[k].t), f"{k} (call {call})")
        if d.q_lora_rank:
            quant_within(outs["out_q_int8"].t, outs["out_scale"].t,
                         ref["out_q_int8"].t.cpu().numpy(), ref["out_scale"].t.cpu().numpy())
        for k, g in outs.items():
            assert g.guards_intact(), k


def test_noalloc_rejects_dims_beyond_its_scratch():
    d = wl.WORKLOADS["v3_prefill"].dims
    dims = binding.MlaPrologDims(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads,
                                 d.nope_dim, d.v_dim, d.max_pos, d.eps, d.flags)
    rc = binding.lib().mla_prolog_run_noalloc(ctypes.byref(dims), *([None] * 12), None)
    assert rc == -2  # MLA_ERR_UNSUPPORTED_DIMS: its workspace exceeds the 32 MiB static scratch
