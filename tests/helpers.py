"""Shared helpers of the GPU tests: device copies of the seeded inputs,
guard-banded output buffers, and the tolerance checks of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

from mla_attention_prolog_gb300 import workloads as wl

GUARD = 64  # elements of sentinel before and after every output buffer
SENTINEL_BF16 = 0x7FA1  # a NaN pattern no kernel writes
SENTINEL_I8 = 0x5A


def bf16_dev(a: np.ndarray, shape, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).reshape(shape).to(dev)


def device_inputs(inp: wl.Inputs, dev):
    d = inp.dims
    return dict(
        x=bf16_dev(inp.x, (d.T, d.D), dev),
        gamma=bf16_dev(inp.gamma, (-1,), dev),
        W_a=bf16_dev(inp.W_a, (d.n_a, d.D), dev),
        W_b=bf16_dev(inp.W_b, (-1,), dev),
        positions=torch.from_numpy(inp.positions).to(dev),
        cos_sin=torch.from_numpy(inp.cos_sin).to(dev),
    )


class Guarded:
    """An output tensor with sentinel guard bands around it."""

    def __init__(self, shape, dtype, dev):
        n = int(np.prod(shape))
        self.n = n
        if dtype == torch.bfloat16:
            self.buf = torch.full((n + 2 * GUARD,), SENTINEL_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
        elif dtype == torch.int8:
            self.buf = torch.full((n + 2 * GUARD,), SENTINEL_I8, dtype=torch.int8, device=dev)
        else:
            self.buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=dtype, device=dev)
        # keep the payload 16-byte aligned: GUARD elements of >= 1 byte, 64 * size % 16 == 0
        self.t = self.buf[GUARD:GUARD + n].view(shape)

    def guards_intact(self) -> bool:
        b = self.buf
        if b.dtype == torch.bfloat16:
            g = torch.cat([b[:GUARD], b[-GUARD:]]).view(torch.int16)
            return bool((g == SENTINEL_BF16).all())
        if b.dtype == torch.int8:
            g = torch.cat([b[:GUARD], b[-GUARD:]])
            return bool((g == SENTINEL_I8).all())
        g = torch.cat([b[:GUARD], b[-GUARD:]])
        return bool(torch.isnan(g).all())


def alloc_outputs(d: wl.Dims, dev):
    H, Dn, Dv, R = d.num_heads, d.nope_dim, d.v_dim, d.rope_dim
    outs = dict(
        out_k=Guarded((d.T, H, Dn + R), torch.bfloat16, dev),
        out_v=Guarded((d.T, H, Dv), torch.bfloat16, dev),
        out_kpe=Guarded((d.T, R), torch.bfloat16, dev),
    )
    if d.q_lora_rank > 0:
        outs["out_q_int8"] = Guarded((d.T, H, Dn + R), torch.int8, dev)
        outs["out_scale"] = Guarded((d.T, d.num_heads) if d.quant_per_head else (d.T,), torch.float32, dev)
    return outs


def run_prolog(p, dins, outs):
    p.run(dins["x"], dins["gamma"], dins["W_a"], dins["W_b"], dins["positions"], dins["cos_sin"],
          outs["out_k"].t, outs["out_v"].t, outs["out_kpe"].t,
          outs["out_q_int8"].t if "out_q_int8" in outs else None,
          outs["out_scale"].t if "out_scale" in outs else None)


def bf16_within(got_bf16: torch.Tensor, want_bits: np.ndarray, name: str) -> None:
    """|d| <= 1e-2 + 1e-2 |ref| elementwise (the BF16 output bar)."""
    got = got_bf16.float().cpu().numpy().reshape(want_bits.shape)
    want = wl.bf16_bits_to_f32(want_bits)
    bad = ~(np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want))
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} outside 1e-2+1e-2|ref|; first at "
                           f"{np.argwhere(bad)[0].tolist()} got {got[bad][0]} want {want[bad][0]}")


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One unit in the last place of BF16 values (8 significand bits); 0 at 0."""
    a = np.abs(x.astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 0.0)


def rope_within(got_bf16: torch.Tensor, want_bits: np.ndarray, kpe_in_bits: np.ndarray, cos: np.ndarray,
                sin: np.ndarray, interleaved: bool, name: str) -> None:
    """Rotated k_pe rows (rotate-half layout [o1 | o2], last axis R; a head
    axis before it is broadcast) within the BF16 bar widened by what a
    one-ulp change of either BF16 input of the pair moves the output:
    ulp(x1)|cos| + ulp(x2)|sin| for o1, ulp(x2)|cos| + ulp(x1)|sin| for o2.
    The compression output is rounded to BF16 before the RoPE; where the
    exact sum lies within the FP32 accumulation's error of a rounding
    boundary, either neighbour is a correct rounding, and a pair whose
    products nearly cancel turns that one ulp into more than the bar.
    kpe_in_bits [n, R]: the oracle's BF16 k_pe; cos, sin [n, R/2]."""
    n, R = kpe_in_bits.shape
    half = R // 2
    kin = wl.bf16_bits_to_f32(kpe_in_bits).astype(np.float64)
    x1 = kin[:, 0::2] if interleaved else kin[:, :half]
    x2 = kin[:, 1::2] if interleaved else kin[:, half:]
    c, s = np.abs(cos.astype(np.float64)), np.abs(sin.astype(np.float64))
    slack = np.concatenate([_bf16_ulp(x1) * c + _bf16_ulp(x2) * s, _bf16_ulp(x2) * c + _bf16_ulp(x1) * s], axis=1)
    want = wl.bf16_bits_to_f32(want_bits).astype(np.float64)
    got = got_bf16.float().cpu().numpy().reshape(want_bits.shape).astype(np.float64)
    if want.ndim == 3:
        slack = slack[:, None, :]
    bad = ~(np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want) + slack)
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} outside the rope bar; first at "
                           f"{np.argwhere(bad)[0].tolist()} got {got[bad][0]} want {want[bad][0]}")


def quant_within(codes: torch.Tensor, scale: torch.Tensor, want_codes: np.ndarray, want_scale: np.ndarray) -> None:
    """Scales relative <= 1e-3; INT8 codes differ by <= 1 on <= 0.1% of elements."""
    s = scale.cpu().numpy().reshape(want_scale.shape)
    rel = np.abs(s - want_scale) / np.maximum(np.abs(want_scale), 1e-30)
    assert np.all((rel <= 1e-3) | ((s == 0) & (want_scale == 0))), f"scale rel err max {rel.max()}"
    c = codes.cpu().numpy().reshape(want_codes.shape).astype(np.int32)
    dq = np.abs(c - want_codes.astype(np.int32))
    assert dq.max() <= 1, f"int8 code differs by {dq.max()}"
    frac = float((dq > 0).mean())
    assert frac <= 1e-3, f"int8 codes differ on {frac:.2e} of elements"
