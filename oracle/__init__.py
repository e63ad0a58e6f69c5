"""CPU oracle of the fused MLA attention prolog (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or runs anything here.

The oracle is plain C (``mla_prolog_oracle.c``), compiled with gcc into
``liboracle.so`` beside this file by :func:`build`, and driven through ctypes.
Every step it computes follows the pages' definitions (see the C file's header
for the precision of each step and the readings taken where the pages are
silent).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_prolog_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


QUANT_Q = 1            # dims flags, the same bits as the C oracle's
ROPE_INTERLEAVED = 2
Q_HEAD_NORM = 4
QUANT_PER_HEAD = 8
W8A8 = 16


class OracleDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "D", "q_lora_rank", "kv_lora_rank", "rope_dim", "num_heads",
        "nope_dim", "v_dim", "max_pos")] + [("eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            os.environ.get("CC", "gcc"), "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        L.oracle_mla_prolog.argtypes = [ctypes.POINTER(OracleDims)] + [P] * 6 + [P, ctypes.c_int32] + [P] * 8
        L.oracle_mla_prolog.restype = ctypes.c_int
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        L.oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.oracle_project_bf16.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P]
        L.oracle_project_f32.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P]
        L.oracle_rmsnorm_row.argtypes = [P, P, ctypes.c_int, ctypes.c_float, P, P]
        L.oracle_rope_f32.argtypes = [P, P, ctypes.c_int, P]
        L.oracle_quant_row.argtypes = [P, ctypes.c_int, P, P]
        L.oracle_deinterleave.argtypes = [P, ctypes.c_int, P]
        L.oracle_rmsnorm_f32_row.argtypes = [P, ctypes.c_int, ctypes.c_float, P]
        L.oracle_mla_prolog_w8a8.argtypes = [ctypes.POINTER(OracleDims)] + [P] * 7 + [P, ctypes.c_int32] + [P] * 14
        L.oracle_mla_prolog_w8a8.restype = ctypes.c_int
        L.oracle_dot_i8.argtypes = [P, P, ctypes.c_int]
        L.oracle_dot_i8.restype = ctypes.c_int64
        L.oracle_dequant.argtypes = [ctypes.c_int32, ctypes.c_float, ctypes.c_float]
        L.oracle_dequant.restype = ctypes.c_float
        L.oracle_project_w8a8.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_float, P, P]
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(d) -> OracleDims:
    return OracleDims(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads,
                      d.nope_dim, d.v_dim, d.max_pos, d.eps, d.flags)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def mla_prolog(d, x, gamma, W_a, W_b, positions, cos_sin,
               tokens: Optional[Sequence[int]] = None, taps: bool = False) -> Dict[str, np.ndarray]:
    """Whole prolog for all tokens (or the listed ones; rows then compact).

    Inputs are raw BF16 bits (uint16), int32 positions and the FP32 cos/sin
    table.  Returns BF16 outputs as uint16 bits, int8 codes and FP32 scales;
    with ``taps`` also the BF16 compression output ``c``, the BF16 ``normed``
    row and the FP32 post-RoPE ``q`` that the quant reads.  ``bad_positions``
    counts tokens whose position was outside ``[0, max_pos)``.
    """
    L = lib()
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = d.T if tok is None else len(tok)
    H, Dn, Dv, R = d.num_heads, d.nope_dim, d.v_dim, d.rope_dim
    out = {
        "out_k": np.zeros((n, H, Dn + R), np.uint16),
        "out_v": np.zeros((n, H, Dv), np.uint16),
        "out_kpe": np.zeros((n, R), np.uint16),
    }
    q8 = sc = None
    if d.q_lora_rank > 0:
        q8 = out["out_q_int8"] = np.zeros((n, H, Dn + R), np.int8)
        sc = out["out_scale"] = np.zeros((n, H) if d.flags & QUANT_PER_HEAD else (n,), np.float32)
    c = nrm = q = None
    if taps:
        c = out["c"] = np.zeros((n, d.q_lora_rank + d.kv_lora_rank + R), np.uint16)
        nrm = out["normed"] = np.zeros((n, d.q_lora_rank + d.kv_lora_rank), np.uint16)
        if d.q_lora_rank > 0:
            q = out["q"] = np.zeros((n, H * (Dn + R)), np.float32)
    arrs = [np.ascontiguousarray(a) for a in (x, gamma, W_a, W_b, positions, cos_sin)]
    dims = _dims(d)
    rc = L.oracle_mla_prolog(ctypes.byref(dims), *[_p(a) for a in arrs],
                             _p(tok), ctypes.c_int32(n),
                             _p(out["out_k"]), _p(out["out_v"]), _p(out["out_kpe"]), _p(q8), _p(sc),
                             _p(c), _p(nrm), _p(q))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    out["bad_positions"] = rc
    return out


def mla_prolog_w8a8(d, x, gamma, W_a, W_b, w_scale, positions, cos_sin,
                    tokens: Optional[Sequence[int]] = None, taps: bool = False,
                    given_codes: Optional[np.ndarray] = None,
                    given_scale: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The prolog with W8A8 projections (``d.flags`` has ``W8A8``).

    ``W_a`` and ``W_b`` are INT8 codes in the layouts of the BF16 weights,
    ``w_scale`` the FP32 scale of every weight row, [W_a rows; W_q_b rows
    (none when q_lora_rank is 0); W_kv_b rows].  Outputs as
    :func:`mla_prolog`; ``taps`` adds the x codes (``x_codes``, ``x_scale``)
    and the normed rows' codes (``n_codes``, ``n_scale`` [n, 2] = c_q, c_kv)
    to ``c``, ``normed`` (values before their quantisation) and ``q``.

    ``given_codes`` [n, Lq + Lkv] int8 and ``given_scale`` [n, 2] float32
    (rows compact like the outputs) replace the normed rows' codes and scales
    that the expansion projections take: every later step then runs on them.
    This checks a candidate whose normed codes legitimately differ from the
    oracle's own (their RMSNorm sums in another order) step for step from
    there on; the ``n_codes`` / ``n_scale`` taps still hold the oracle's own.
    """
    L = lib()
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = d.T if tok is None else len(tok)
    H, Dn, Dv, R = d.num_heads, d.nope_dim, d.v_dim, d.rope_dim
    Lq, Lkv = d.q_lora_rank, d.kv_lora_rank
    out = {
        "out_k": np.zeros((n, H, Dn + R), np.uint16),
        "out_v": np.zeros((n, H, Dv), np.uint16),
        "out_kpe": np.zeros((n, R), np.uint16),
    }
    q8 = sc = None
    if Lq > 0:
        q8 = out["out_q_int8"] = np.zeros((n, H, Dn + R), np.int8)
        sc = out["out_scale"] = np.zeros((n, H) if d.flags & QUANT_PER_HEAD else (n,), np.float32)
    c = nrm = q = xc = xs = nc = ns = None
    if taps:
        c = out["c"] = np.zeros((n, Lq + Lkv + R), np.uint16)
        nrm = out["normed"] = np.zeros((n, Lq + Lkv), np.uint16)
        if Lq > 0:
            q = out["q"] = np.zeros((n, H * (Dn + R)), np.float32)
        xc = out["x_codes"] = np.zeros((n, d.D), np.int8)
        xs = out["x_scale"] = np.zeros(n, np.float32)
        nc = out["n_codes"] = np.zeros((n, Lq + Lkv), np.int8)
        ns = out["n_scale"] = np.zeros((n, 2), np.float32)
    arrs = [np.ascontiguousarray(x, np.uint16), np.ascontiguousarray(gamma, np.uint16),
            np.ascontiguousarray(W_a, np.int8), np.ascontiguousarray(W_b, np.int8),
            np.ascontiguousarray(w_scale, np.float32), np.ascontiguousarray(positions, np.int32),
            np.ascontiguousarray(cos_sin, np.float32)]
    gc = gs = None
    if (given_codes is None) != (given_scale is None):
        raise ValueError("given_codes and given_scale go together")
    if given_codes is not None:
        gc = np.ascontiguousarray(given_codes, np.int8)
        gs = np.ascontiguousarray(given_scale, np.float32)
        if gc.shape != (n, Lq + Lkv) or gs.shape != (n, 2):
            raise ValueError(f"given codes {gc.shape} / scales {gs.shape} for {n} rows")
    dims = _dims(d)
    rc = L.oracle_mla_prolog_w8a8(ctypes.byref(dims), *[_p(a) for a in arrs], _p(tok), ctypes.c_int32(n),
                                  _p(out["out_k"]), _p(out["out_v"]), _p(out["out_kpe"]), _p(q8), _p(sc),
                                  _p(c), _p(nrm), _p(q), _p(xc), _p(xs), _p(nc), _p(ns), _p(gc), _p(gs))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    out["bad_positions"] = rc
    return out


def scatter_kv_cache(cache: np.ndarray, slot_mapping: np.ndarray, normed: np.ndarray, out_kpe: np.ndarray,
                     q_lora_rank: int) -> int:
    """Writes the latent KV cache rows of the listed tokens in place.

    The cache write of the pages (the DeepSeek-V3.2-Exp PyPTO article: results
    cached into the KV cache, written with ScatterUpdate into the KCache): row
    ``slot_mapping[j]`` of ``cache`` [num_slots, Lkv + R] receives token j's
    normed c_kv (BF16 bits) followed by its rotated k_pe.  A negative slot is
    skipped (a padding token); a slot >= num_slots is skipped and counted.
    Returns the number of out-of-range slots.
    """
    num_slots = cache.shape[0]
    bad = 0
    for j, slot in enumerate(np.asarray(slot_mapping, np.int64)):
        if slot < 0:
            continue
        if slot >= num_slots:
            bad += 1
            continue
        cache[slot] = np.concatenate([normed[j, q_lora_rank:], out_kpe[j]])
    return bad


# -- single steps, for the pins ------------------------------------------------

def f32_to_bf16(v: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(v)))


def f64_to_bf16(v: float) -> int:
    return int(lib().oracle_f64_to_bf16(float(v)))


def project_bf16(x_row: np.ndarray, W: np.ndarray) -> np.ndarray:
    x_row = np.ascontiguousarray(x_row, np.uint16)
    W = np.ascontiguousarray(W, np.uint16)
    N, K = W.shape
    out = np.zeros(N, np.uint16)
    lib().oracle_project_bf16(_p(x_row), _p(W), N, K, _p(out))
    return out


def project_f32(a_row: np.ndarray, W: np.ndarray) -> np.ndarray:
    a_row = np.ascontiguousarray(a_row, np.uint16)
    W = np.ascontiguousarray(W, np.uint16)
    N, K = W.shape
    out = np.zeros(N, np.float32)
    lib().oracle_project_f32(_p(a_row), _p(W), N, K, _p(out))
    return out


def rmsnorm_row(x_bits: np.ndarray, gamma_bits: Optional[np.ndarray], eps: float):
    x_bits = np.ascontiguousarray(x_bits, np.uint16)
    g = None if gamma_bits is None else np.ascontiguousarray(gamma_bits, np.uint16)
    L = len(x_bits)
    y32 = np.zeros(L, np.float32)
    y16 = np.zeros(L, np.uint16)
    lib().oracle_rmsnorm_row(_p(x_bits), _p(g), L, ctypes.c_float(eps), _p(y32), _p(y16))
    return y32, y16


def rope(x: np.ndarray, cs_row: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    cs_row = np.ascontiguousarray(cs_row, np.float32)
    out = np.zeros_like(x)
    lib().oracle_rope_f32(_p(x), _p(cs_row), len(x), _p(out))
    return out


def deinterleave(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros_like(x)
    lib().oracle_deinterleave(_p(x), len(x), _p(out))
    return out


def rmsnorm_f32_row(x: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros_like(x)
    lib().oracle_rmsnorm_f32_row(_p(x), len(x), ctypes.c_float(eps), _p(out))
    return out


def quant_row(y: np.ndarray):
    y = np.ascontiguousarray(y, np.float32)
    codes = np.zeros(len(y), np.int8)
    scale = np.zeros(1, np.float32)
    lib().oracle_quant_row(_p(y), len(y), _p(codes), _p(scale))
    return codes, float(scale[0])


def dot_i8(a: np.ndarray, w: np.ndarray) -> int:
    a = np.ascontiguousarray(a, np.int8)
    w = np.ascontiguousarray(w, np.int8)
    return int(lib().oracle_dot_i8(_p(a), _p(w), len(a)))


def dequant(y: int, a_scale: float, w_scale: float) -> float:
    return float(lib().oracle_dequant(ctypes.c_int32(y), ctypes.c_float(a_scale), ctypes.c_float(w_scale)))


def project_w8a8(a_codes: np.ndarray, W: np.ndarray, a_scale: float, w_scale: np.ndarray) -> np.ndarray:
    a_codes = np.ascontiguousarray(a_codes, np.int8)
    W = np.ascontiguousarray(W, np.int8)
    w_scale = np.ascontiguousarray(w_scale, np.float32)
    N, K = W.shape
    out = np.zeros(N, np.float32)
    lib().oracle_project_w8a8(_p(a_codes), _p(W), N, K, ctypes.c_float(a_scale), _p(w_scale), _p(out))
    return out
