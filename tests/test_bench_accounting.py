"""bench.py's work accounting (no GPU): the per-kernel algorithmic bytes of
every workload and variant add up to the whole op's, and the W8A8 mode
counts its INT8 weights at one byte plus their row scales."""
import dataclasses
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from mla_attention_prolog_gb300 import workloads as wl  # noqa: E402

VARIANTS = [0, wl.ROPE_INTERLEAVED, wl.QUANT_PER_HEAD, wl.Q_HEAD_NORM | wl.QUANT_PER_HEAD, wl.W8A8,
            wl.W8A8 | wl.QUANT_PER_HEAD]


@pytest.mark.parametrize("name", ["tiny", "tiny_q", "v2lite_decode", "v2lite_prefill", "v3_decode", "v3_prefill"])
@pytest.mark.parametrize("flags", VARIANTS)
@pytest.mark.parametrize("cache", [False, True])
def test_kernel_bytes_add_up(name, flags, cache):
    d0 = wl.WORKLOADS[name].dims
    if flags & (wl.QUANT_PER_HEAD | wl.Q_HEAD_NORM) and not d0.q_lora_rank:
        pytest.skip("a q variant without a q path")
    d = dataclasses.replace(d0, flags=d0.flags | flags)
    names = ["mla_quant_x_kernel", "mla_compress_kernel", "mla_norm_rope_kernel", "mla_expand_kernel",
             "mla_quant_kernel"]
    b, f = bench.kernel_work(d, cache, names)  # asserts the per-kernel bytes sum to the whole op's
    assert all(v >= 0 for v in b.values())
    assert sum(f[k] for k in names) == wl.algorithmic_flops(d)
    if not d.w8a8:
        assert b["mla_quant_x_kernel"] == 0
    b2, _ = bench.kernel_work(d, cache, names + ["mla_expand_kv_pair_kernel"])
    assert b2["mla_expand_pair_kernel"] + b2["mla_expand_kv_pair_kernel"] == b["mla_expand_kernel"]


@pytest.mark.parametrize("name", ["v2lite_prefill", "v3_decode", "v3_prefill"])
def test_w8a8_counts_weights_at_one_byte(name):
    d = wl.WORKLOADS[name].dims
    d8 = dataclasses.replace(d, flags=d.flags | wl.W8A8)
    weights = d.n_a * d.D + d.w_b_elems
    assert wl.algorithmic_bytes(d) - wl.algorithmic_bytes(d8) == weights - 4 * d8.n_w_scales
    assert wl.algorithmic_flops(d8) == wl.algorithmic_flops(d)
