"""Workload registry and seeded synthetic inputs for the MLA attention prolog.

This module only draws and packs input bytes.  It holds none of the prolog's
arithmetic, so both the CUDA path and the CPU oracle can consume exactly the
same inputs.

Shapes follow the DeepSeek-V2-Lite MLA KV-prolog migration guide (section
"精度验证", case ``mla_prolog_001``: hidden 2048, kv_lora_rank 512, rope 64,
16 heads x (128 nope + 128 value)) and the DeepSeek-V3 full prolog with a
q path (q_lora_rank 1536, 128 heads, 128 nope + 64 rope).  No model weights
are used: every tensor is random with the distribution stated per workload.

Packing (a convention of this library, the pages are silent on it):
  * ``W_a``   = rows ``[W_q_a (Lq x D) ; W_kv_a ((Lkv + R) x D)]`` in ``[N, K]``
                layout; the kv rows are ``[c_kv (Lkv) ; k_pe (R)]``.
  * ``gamma`` = ``[gamma_q (Lq) ; gamma_kv (Lkv)]``.
  * ``W_b``   = ``W_q_b (H*(Dn+R) x Lq)`` followed by ``W_kv_b (H*(Dn+Dv) x Lkv)``,
                both ``[N, K]`` row-major, flattened back to back.
  * ``cos_sin`` = FP32 ``[max_pos, R]``; columns ``[0, R/2)`` hold
                ``cos(p * theta_i)`` and ``[R/2, R)`` hold ``sin(p * theta_i)`` with
                ``theta_i = base ** (-2 i / R)``, base 10000.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, Optional

import numpy as np
import torch

QUANT_Q = 1           # flag bits (the C header's MLA_PROLOG_*): INT8 quantisation of the q path
ROPE_INTERLEAVED = 2  # rope slices de-interleaved before the rotate-half RoPE
Q_HEAD_NORM = 4       # per-head RMSNorm (no gamma) of q before its RoPE
QUANT_PER_HEAD = 8    # one q scale per (token, head) instead of per token
W8A8 = 16             # INT8 weights and per-token INT8 activations in every projection

# Variant names (benchmark and tests) -> flag bits; "cache" is the latent
# KV-cache write of mla_prolog_run_cached, not a flag.
VARIANTS = {"interleaved": ROPE_INTERLEAVED, "head_norm": Q_HEAD_NORM, "per_head": QUANT_PER_HEAD, "cache": 0,
            "w8a8": W8A8}


@dataclasses.dataclass(frozen=True)
class Dims:
    T: int
    D: int
    q_lora_rank: int
    kv_lora_rank: int
    rope_dim: int
    num_heads: int
    nope_dim: int
    v_dim: int
    max_pos: int
    eps: float = 1e-6
    flags: int = 0

    # derived sizes -------------------------------------------------------
    @property
    def n_a(self) -> int:
        """Rows of the packed compression weight: Lq + Lkv + R."""
        return self.q_lora_rank + self.kv_lora_rank + self.rope_dim

    @property
    def n_q(self) -> int:
        """Columns of the expanded q row: H * (Dn + R)."""
        return self.num_heads * (self.nope_dim + self.rope_dim)

    @property
    def n_kv(self) -> int:
        """Columns of the expanded kv row: H * (Dn + Dv)."""
        return self.num_heads * (self.nope_dim + self.v_dim)

    @property
    def w_b_elems(self) -> int:
        return self.n_q * self.q_lora_rank + self.n_kv * self.kv_lora_rank

    @property
    def quant_q(self) -> bool:
        return bool(self.flags & QUANT_Q)

    @property
    def quant_per_head(self) -> bool:
        return bool(self.flags & QUANT_PER_HEAD)

    @property
    def w8a8(self) -> bool:
        return bool(self.flags & W8A8)

    @property
    def n_w_scales(self) -> int:
        """Weight rows with a W8A8 scale: W_a, W_q_b (none without a q path), W_kv_b."""
        return self.n_a + (self.n_q if self.q_lora_rank > 0 else 0) + self.n_kv

    @property
    def n_scales(self) -> int:
        """q scales per token."""
        return self.num_heads if self.quant_per_head else 1

    def with_T(self, T: int) -> "Dims":
        return dataclasses.replace(self, T=T)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    positions: str          # "arange" | "uniform"
    boost_frac: float = 0.0  # fraction of token rows of x scaled before rounding
    boost: float = 20.0
    bound: str = "latency"   # "hbm" | "tensor" | "latency"
    seed: int = 0


# The five workloads, in the order they are specified, plus a small q-path case.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload(
        "tiny", Dims(T=4, D=256, q_lora_rank=0, kv_lora_rank=64, rope_dim=16,
                     num_heads=2, nope_dim=32, v_dim=32, max_pos=4),
        positions="arange", bound="latency"),
    "v2lite_decode": Workload(
        "v2lite_decode", Dims(T=64, D=2048, q_lora_rank=0, kv_lora_rank=512, rope_dim=64,
                              num_heads=16, nope_dim=128, v_dim=128, max_pos=4096),
        positions="uniform", bound="hbm"),
    "v2lite_prefill": Workload(
        "v2lite_prefill", Dims(T=4096, D=2048, q_lora_rank=0, kv_lora_rank=512, rope_dim=64,
                               num_heads=16, nope_dim=128, v_dim=128, max_pos=4096),
        positions="arange", bound="tensor"),
    "v3_decode": Workload(
        "v3_decode", Dims(T=128, D=7168, q_lora_rank=1536, kv_lora_rank=512, rope_dim=64,
                          num_heads=128, nope_dim=128, v_dim=128, max_pos=32768, flags=QUANT_Q),
        positions="uniform", bound="hbm"),
    "v3_prefill": Workload(
        "v3_prefill", Dims(T=16384, D=7168, q_lora_rank=1536, kv_lora_rank=512, rope_dim=64,
                           num_heads=128, nope_dim=128, v_dim=128, max_pos=16384, flags=QUANT_Q),
        positions="arange", boost_frac=0.01, bound="tensor"),
    # Not one of the five: the smallest case that exercises the q path and quant.
    "tiny_q": Workload(
        "tiny_q", Dims(T=4, D=256, q_lora_rank=32, kv_lora_rank=64, rope_dim=16,
                       num_heads=2, nope_dim=32, v_dim=32, max_pos=4, flags=QUANT_Q),
        positions="arange", bound="latency"),
}

ORDERED = ["tiny", "v2lite_decode", "v2lite_prefill", "v3_decode", "v3_prefill"]


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    """FP32 tensor -> BF16 (round to nearest even) -> raw uint16 bits."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def cos_sin_table(max_pos: int, rope_dim: int, base: float = 10000.0) -> np.ndarray:
    """FP32 ``[max_pos, R]`` table: cos in the first half, sin in the second.

    Angles are formed and evaluated in float64, then rounded once to FP32.
    """
    half = rope_dim // 2
    i = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * i / rope_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * theta[None, :]
    tab = np.concatenate([np.cos(ang), np.sin(ang)], axis=1)
    return np.ascontiguousarray(tab.astype(np.float32))


@dataclasses.dataclass
class Inputs:
    dims: Dims
    x: np.ndarray          # uint16 (bf16 bits) [T, D]
    W_a: np.ndarray        # uint16 [Lq+Lkv+R, D]
    gamma: np.ndarray      # uint16 [Lq+Lkv]
    W_b: np.ndarray        # uint16 flat [H(Dn+R)Lq + H(Dn+Dv)Lkv]
    positions: np.ndarray  # int32 [T]
    cos_sin: np.ndarray    # float32 [max_pos, R]
    boosted_rows: np.ndarray  # int64 indices of rows of x scaled by `boost`

    def sha256(self) -> str:
        h = hashlib.sha256()
        for a in (self.x, self.W_a, self.gamma, self.W_b, self.positions, self.cos_sin):
            h.update(np.ascontiguousarray(a).tobytes())
        return h.hexdigest()


def make_inputs(wl: Workload, dims: Optional[Dims] = None, seed: Optional[int] = None) -> Inputs:
    """Seeded synthetic inputs for a workload.

    Draw order (fixed): x, W_a (q_a rows then kv_a rows), gamma, W_b (q_b then
    kv_b), positions, then the choice of boosted rows.  Values are drawn in
    FP32 and rounded to BF16 once, round-to-nearest-even.
      x ~ N(0, 1); W ~ N(0, 0.02); gamma ~ N(1, 0.1);
      positions: 0..T-1 ("arange") or uniform in [0, max_pos) ("uniform").
    """
    d = dims or wl.dims
    g = torch.Generator("cpu").manual_seed(wl.seed if seed is None else seed)
    Lq, Lkv, R, D, T = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.D, d.T
    x32 = torch.randn((T, D), generator=g, dtype=torch.float32)
    wqa = torch.randn((Lq, D), generator=g, dtype=torch.float32) * 0.02
    wkva = torch.randn((Lkv + R, D), generator=g, dtype=torch.float32) * 0.02
    gamma = 1.0 + 0.1 * torch.randn((Lq + Lkv,), generator=g, dtype=torch.float32)
    wqb = torch.randn((d.n_q * Lq,), generator=g, dtype=torch.float32) * 0.02
    wkvb = torch.randn((d.n_kv * Lkv,), generator=g, dtype=torch.float32) * 0.02
    if wl.positions == "arange":
        if T > d.max_pos:
            raise ValueError("arange positions need T <= max_pos")
        pos = torch.arange(T, dtype=torch.int32)
    else:
        pos = torch.randint(0, d.max_pos, (T,), generator=g, dtype=torch.int32)
    boosted = np.zeros(0, dtype=np.int64)
    if wl.boost_frac > 0:
        nb = int(round(wl.boost_frac * T))
        perm = torch.randperm(T, generator=g)[:nb]
        boosted = np.sort(perm.numpy().astype(np.int64))
        x32[perm] *= wl.boost
    return Inputs(
        dims=d,
        x=_bf16_bits(x32),
        W_a=_bf16_bits(torch.cat([wqa, wkva], 0)),
        gamma=_bf16_bits(gamma),
        W_b=_bf16_bits(torch.cat([wqb, wkvb], 0)),
        positions=pos.numpy().astype(np.int32).copy(),
        cos_sin=cos_sin_table(d.max_pos, R),
        boosted_rows=boosted,
    )


@dataclasses.dataclass
class W8A8Weights:
    W_a: np.ndarray      # int8 [Lq+Lkv+R, D] codes, the layout of the BF16 W_a
    W_b: np.ndarray      # int8 flat, the layout of the BF16 W_b
    w_scale: np.ndarray  # float32 [n_w_scales]: W_a rows, W_q_b rows, W_kv_b rows

    def sha256(self) -> str:
        h = hashlib.sha256()
        for a in (self.W_a, self.W_b, self.w_scale):
            h.update(np.ascontiguousarray(a).tobytes())
        return h.hexdigest()


def make_w8a8_weights(wl: Workload, dims: Optional[Dims] = None, seed: Optional[int] = None) -> W8A8Weights:
    """Seeded INT8 weights for the W8A8 projections, drawn on their own
    generator (the BF16 inputs of the same seed are unchanged).

    Codes are clamp(rint(N(0, 28)), -127, 127), the bell shape of a N(0, 0.02)
    weight matrix stored with one scale per row (its largest entry near 4.5
    standard deviations); each row's scale is 0.02 * 4.5 / 127 times U(0.8,
    1.2).  Draw order: W_a codes, W_b codes, scales.
    """
    d = dims or wl.dims
    g = torch.Generator("cpu").manual_seed((wl.seed if seed is None else seed) + 7919)
    def codes(n):
        return torch.clamp(torch.round(torch.randn((n,), generator=g, dtype=torch.float32) * 28.0), -127, 127)
    wa = codes(d.n_a * d.D).to(torch.int8).numpy().reshape(d.n_a, d.D).copy()
    wb = codes(d.w_b_elems).to(torch.int8).numpy().copy()
    sc = (0.02 * 4.5 / 127.0) * (0.8 + 0.4 * torch.rand((d.n_w_scales,), generator=g, dtype=torch.float32))
    return W8A8Weights(W_a=wa, W_b=wb, w_scale=sc.numpy().astype(np.float32).copy())


# ---------------------------------------------------------------------------
# Algorithmic work counts (inputs read once, outputs written once; GEMM flops).

def algorithmic_bytes(d: Dims, cache: bool = False) -> int:
    """Every input read once + every output written once; with ``cache`` also
    the slot indices read and the latent cache rows (Lkv + R BF16) written.
    W8A8 weights count one byte per code plus their FP32 row scales."""
    T = d.T
    wbytes = 1 if d.w8a8 else 2                            # INT8 or BF16 weights
    b = 2 * T * d.D + wbytes * d.n_a * d.D + 2 * (d.q_lora_rank + d.kv_lora_rank)
    b += wbytes * d.w_b_elems + 4 * T + 4 * T * d.rope_dim  # positions + gathered cos/sin rows
    if d.w8a8:
        b += 4 * d.n_w_scales                              # the weight rows' scales
    b += 2 * T * d.num_heads * (d.nope_dim + d.rope_dim)  # out_k
    b += 2 * T * d.num_heads * d.v_dim                    # out_v
    b += 2 * T * d.rope_dim                               # out_kpe
    if d.quant_q:
        b += T * d.n_q + 4 * T * d.n_scales               # int8 codes + scales
    if cache:
        b += 4 * T + 2 * T * (d.kv_lora_rank + d.rope_dim)  # slot_mapping + cache rows
    return b


def algorithmic_flops(d: Dims) -> int:
    return 2 * d.T * (d.n_a * d.D + d.n_q * d.q_lora_rank + d.n_kv * d.kv_lora_rank)


def output_shapes(d: Dims) -> Dict[str, tuple]:
    s = {
        "out_k": (d.T, d.num_heads, d.nope_dim + d.rope_dim),
        "out_v": (d.T, d.num_heads, d.v_dim),
        "out_kpe": (d.T, d.rope_dim),
    }
    if d.quant_q:
        s["out_q_int8"] = (d.T, d.num_heads, d.nope_dim + d.rope_dim)
        s["out_scale"] = (d.T, d.num_heads) if d.quant_per_head else (d.T,)
    return s


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen raw BF16 bits to FP32 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)
