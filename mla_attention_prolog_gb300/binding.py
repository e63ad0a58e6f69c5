"""Python binding of libmla_prolog.so: argument marshalling only.

Every step of the prolog runs in the library's CUDA kernels.  This module
checks tensor placement, dtype, shape and contiguity, turns tensors into raw
device pointers and calls the C ABI of ``include/mla_prolog.h`` through
ctypes.  There is no fallback: if the library is missing or the device is not
an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_prolog.so")

MLA_OK = 0
MLA_PROLOG_QUANT_Q = 1
MLA_PROLOG_ROPE_INTERLEAVED = 2
MLA_PROLOG_Q_HEAD_NORM = 4
MLA_PROLOG_QUANT_PER_HEAD = 8
MLA_PROLOG_W8A8 = 16
STATUS_POSITION_RANGE = 0x1
STATUS_WAIT_TIMEOUT = 0x2
STATUS_SLOT_RANGE = 0x4

EXPORTED = [
    "mla_prolog_create", "mla_prolog_run", "mla_prolog_destroy", "mla_prolog_device_status",
    "mla_prolog_strerror", "mla_prolog_last_cuda_error", "mla_prolog_quant_rows",
    "mla_prolog_set_wait_timeout", "mla_prolog_selftest_wait_timeout",
    "mla_prolog_set_timing_events", "mla_prolog_kernel_count", "mla_prolog_kernel_name",
    "mla_prolog_workspace_bytes", "mla_prolog_schedule", "mla_prolog_copy_tap", "mla_prolog_set_tuning",
    "mla_prolog_run_noalloc", "mla_prolog_run_cached", "mla_prolog_plan", "mla_prolog_lpt",
    "mla_prolog_load_w8a8",
]
TAP_NORMED, TAP_Q, TAP_AMAX = 1, 2, 3
TAP_X_CODES, TAP_X_SCALE, TAP_NORM_SCALE = 4, 5, 6
TUNE_COMPRESS_GROUP = 1
TUNE_COMPRESS_COMPENSATED = 2
TUNE_DECODE_FUSED = 3
TUNE_CLUSTER_NORM = 4
TUNE_PAIR_EXPAND = 6
TUNE_PAIR_COMPRESS = 7
TUNE_TMA_STORE = 8
TUNE_COMPRESS_TILE = 9
TUNE_L2_FETCH = 10
TUNE_Q_WIDE = 11
TUNE_KV_RESIDENT = 12
TUNE_QUANT_OVERLAP = 13
TUNE_KV_GROUP = 14
TUNE_L2_POLICY = 15
TUNE_KV_HALVES = 16


class MlaPrologDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "D", "q_lora_rank", "kv_lora_rank", "rope_dim", "num_heads",
        "nope_dim", "v_dim", "max_pos")] + [("eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class MlaPrologPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "decode", "bn_a", "splits_a", "group_a", "compress_jobs", "bn_kv", "kv_halves")] + \
        [("busiest_bytes", ctypes.c_int64)]


class MlaPrologError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().mla_prolog_strerror(code).decode()
        cuda = lib().mla_prolog_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (code {code}){' — ' + cuda if cuda and code == -3 else ''}")


_lib = None


def lib(path: Optional[str] = None):
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -m mla_attention_prolog_gb300.build)")
    L = ctypes.CDLL(p)
    V, I32, P = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER
    L.mla_prolog_create.argtypes = [P(MlaPrologDims), P(V)]
    L.mla_prolog_run.argtypes = [V] * 13
    L.mla_prolog_destroy.argtypes = [V]
    L.mla_prolog_device_status.argtypes = [V, V, P(I32)]
    L.mla_prolog_strerror.argtypes = [ctypes.c_int]
    L.mla_prolog_strerror.restype = ctypes.c_char_p
    L.mla_prolog_last_cuda_error.restype = ctypes.c_char_p
    L.mla_prolog_quant_rows.argtypes = [V, I32, I32, V, V, V]
    L.mla_prolog_set_wait_timeout.argtypes = [V, ctypes.c_uint64]
    L.mla_prolog_selftest_wait_timeout.argtypes = [V, ctypes.c_uint64, V]
    L.mla_prolog_set_timing_events.argtypes = [V, P(V), I32]
    L.mla_prolog_kernel_count.argtypes = [V]
    L.mla_prolog_kernel_count.restype = I32
    L.mla_prolog_kernel_name.argtypes = [V, I32]
    L.mla_prolog_kernel_name.restype = ctypes.c_char_p
    L.mla_prolog_workspace_bytes.argtypes = [V, P(ctypes.c_size_t)]
    L.mla_prolog_schedule.argtypes = [V, P(I32), P(I32), P(I32), P(I32)]
    L.mla_prolog_copy_tap.argtypes = [V, I32, V, ctypes.c_size_t, V]
    L.mla_prolog_set_tuning.argtypes = [V, I32, I32]
    L.mla_prolog_run_noalloc.argtypes = [P(MlaPrologDims)] + [V] * 13
    L.mla_prolog_run_cached.argtypes = [V] * 14 + [ctypes.c_int64, V]
    L.mla_prolog_plan.argtypes = [P(MlaPrologDims), I32, P(MlaPrologPlanInfo)]
    L.mla_prolog_lpt.argtypes = [P(ctypes.c_int64), I32, I32, P(I32), P(ctypes.c_int64)]
    L.mla_prolog_load_w8a8.argtypes = [V, V, V, V, V]
    for n in EXPORTED:
        if n not in ("mla_prolog_strerror", "mla_prolog_last_cuda_error", "mla_prolog_kernel_count",
                     "mla_prolog_kernel_name"):
            getattr(L, n).restype = ctypes.c_int
    _lib = L
    return L


def _check(rc: int, where: str) -> None:
    if rc != MLA_OK:
        raise MlaPrologError(rc, where)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> Optional[int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


def _ptr(t: Optional[torch.Tensor], name: str, dtype, shape: Sequence[int], device) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class MlaProlog:
    """One handle of the fused prolog for fixed dims on the current device."""

    def __init__(self, T, D, q_lora_rank, kv_lora_rank, rope_dim, num_heads, nope_dim, v_dim,
                 max_pos, eps: float = 1e-6, flags: Optional[int] = None):
        if flags is None:
            flags = MLA_PROLOG_QUANT_Q if q_lora_rank > 0 else 0
        self.dims = MlaPrologDims(T, D, q_lora_rank, kv_lora_rank, rope_dim, num_heads, nope_dim,
                                  v_dim, max_pos, eps, flags)
        self.device = torch.device("cuda", torch.cuda.current_device())
        h = ctypes.c_void_p()
        _check(lib().mla_prolog_create(ctypes.byref(self.dims), ctypes.byref(h)), "mla_prolog_create")
        self._h = h

    @classmethod
    def from_dims(cls, d) -> "MlaProlog":
        return cls(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim,
                   d.v_dim, d.max_pos, d.eps, d.flags)

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise RuntimeError("handle is closed")
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().mla_prolog_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _args(self, x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe, out_q_int8, out_scale):
        d = self.dims
        dev = self.device
        Lq, Lkv, R, H, Dn, Dv = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim, d.v_dim
        bf = torch.bfloat16
        wb = H * (Dn + R) * Lq + H * (Dn + Dv) * Lkv
        scale_shape = (d.T, H) if d.flags & MLA_PROLOG_QUANT_PER_HEAD else (d.T,)
        if d.flags & MLA_PROLOG_W8A8 and (W_a is not None or W_b is not None):
            raise ValueError("a W8A8 handle takes its weights from load_w8a8: pass W_a = W_b = None")
        return [
            _ptr(x, "x", bf, (d.T, d.D), dev),
            _ptr(gamma, "gamma", bf, (Lq + Lkv,), dev),
            _ptr(W_a, "W_a", bf, (Lq + Lkv + R, d.D), dev),
            _ptr(W_b, "W_b", bf, (wb,), dev),
            _ptr(positions, "positions", torch.int32, (d.T,), dev),
            _ptr(cos_sin, "cos_sin", torch.float32, (d.max_pos, R), dev),
            _ptr(out_k, "out_k", bf, (d.T, H, Dn + R), dev),
            _ptr(out_v, "out_v", bf, (d.T, H, Dv), dev),
            _ptr(out_kpe, "out_kpe", bf, (d.T, R), dev),
            _ptr(out_q_int8, "out_q_int8", torch.int8, (d.T, H, Dn + R), dev),
            _ptr(out_scale, "out_scale", torch.float32, scale_shape, dev),
        ]

    def run(self, x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe,
            out_q_int8=None, out_scale=None, stream=None) -> None:
        args = self._args(x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe, out_q_int8, out_scale)
        _check(lib().mla_prolog_run(self.handle, *args, _stream_ptr(stream)), "mla_prolog_run")

    def run_cached(self, x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe,
                   out_q_int8, out_scale, slot_mapping, kv_cache, stream=None) -> None:
        """``run`` plus the latent KV-cache write: row ``slot_mapping[t]`` of
        ``kv_cache`` (BF16 ``[num_slots, Lkv + R]``) gets ``[normed c_kv | k_pe_rot]``."""
        d = self.dims
        args = self._args(x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe, out_q_int8, out_scale)
        if kv_cache.dim() != 2:
            raise ValueError("kv_cache must be [num_slots, kv_lora_rank + rope_dim]")
        n = kv_cache.shape[0]
        cache = _ptr(kv_cache, "kv_cache", torch.bfloat16, (n, d.kv_lora_rank + d.rope_dim), self.device)
        slots = _ptr(slot_mapping, "slot_mapping", torch.int32, (d.T,), self.device)
        _check(lib().mla_prolog_run_cached(self.handle, *args, slots, cache, n, _stream_ptr(stream)),
               "mla_prolog_run_cached")

    def load_w8a8(self, W_a, W_b, w_scale, stream=None) -> None:
        """Loads INT8 weight codes (the layouts of the BF16 W_a and W_b) and
        their FP32 row scales ([W_a rows; W_q_b rows; W_kv_b rows]) into a
        W8A8 handle."""
        d = self.dims
        Lq, Lkv, R, H, Dn, Dv = d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim, d.v_dim
        NQw = H * (Dn + R) if Lq > 0 else 0
        wb = H * (Dn + R) * Lq + H * (Dn + Dv) * Lkv
        a = _ptr(W_a, "W_a", torch.int8, (Lq + Lkv + R, d.D), self.device)
        b = _ptr(W_b, "W_b", torch.int8, (wb,), self.device)
        s = _ptr(w_scale, "w_scale", torch.float32, (Lq + Lkv + R + NQw + H * (Dn + Dv),), self.device)
        _check(lib().mla_prolog_load_w8a8(self.handle, a, b, s, _stream_ptr(stream)), "mla_prolog_load_w8a8")

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int32(0)
        _check(lib().mla_prolog_device_status(self.handle, _stream_ptr(stream), ctypes.byref(v)),
               "mla_prolog_device_status")
        return int(v.value)

    def set_wait_timeout(self, ns: int) -> None:
        _check(lib().mla_prolog_set_wait_timeout(self.handle, int(ns)), "mla_prolog_set_wait_timeout")

    def selftest_wait_timeout(self, ns: int, stream=None) -> None:
        _check(lib().mla_prolog_selftest_wait_timeout(self.handle, int(ns), _stream_ptr(stream)),
               "mla_prolog_selftest_wait_timeout")

    def set_timing_events(self, events) -> None:
        if not events:
            _check(lib().mla_prolog_set_timing_events(self.handle, None, 0), "set_timing_events")
            return
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event on its first record
                e.record(torch.cuda.current_stream(self.device))
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        _check(lib().mla_prolog_set_timing_events(self.handle, arr, len(events)), "set_timing_events")

    def kernel_names(self):
        n = lib().mla_prolog_kernel_count(self.handle)
        return [lib().mla_prolog_kernel_name(self.handle, i).decode() for i in range(n)]

    def tap(self, which: int, stream=None) -> torch.Tensor:
        """Device copy of an intermediate of the last run (normed rows, FP32 q, amax)."""
        d = self.dims
        if which == TAP_NORMED:
            t = torch.empty((d.T, d.q_lora_rank + d.kv_lora_rank), dtype=torch.bfloat16, device=self.device)
        elif which == TAP_Q:
            t = torch.empty((d.T, d.num_heads * (d.nope_dim + d.rope_dim)), dtype=torch.float32, device=self.device)
        elif which == TAP_AMAX:
            t = torch.empty((d.T,), dtype=torch.float32, device=self.device)
        elif which == TAP_X_CODES:
            t = torch.empty((d.T, d.D), dtype=torch.bfloat16, device=self.device)
        elif which == TAP_X_SCALE:
            t = torch.empty((d.T,), dtype=torch.float32, device=self.device)
        elif which == TAP_NORM_SCALE:
            t = torch.empty((d.T, 2), dtype=torch.float32, device=self.device)
        else:
            raise ValueError(which)
        _check(lib().mla_prolog_copy_tap(self.handle, which, t.data_ptr(), t.numel() * t.element_size(),
                                         _stream_ptr(stream)), "mla_prolog_copy_tap")
        return t

    def set_tuning(self, key: int, value: int) -> None:
        _check(lib().mla_prolog_set_tuning(self.handle, key, value), "mla_prolog_set_tuning")

    def workspace_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _check(lib().mla_prolog_workspace_bytes(self.handle, ctypes.byref(v)), "workspace_bytes")
        return int(v.value)

    def schedule(self) -> dict:
        vals = [ctypes.c_int32(0) for _ in range(4)]
        _check(lib().mla_prolog_schedule(self.handle, *[ctypes.byref(v) for v in vals]), "schedule")
        return dict(zip(("bn_a", "splits_a", "bn_kv", "bn_q"), [v.value for v in vals]))


def quant_rows(y: torch.Tensor, codes: torch.Tensor, scale: torch.Tensor, stream=None) -> None:
    """Per-token INT8 quantisation of FP32 rows (the q path's last step)."""
    if y.dim() != 2:
        raise ValueError("y must be [rows, row_len]")
    rows, n = y.shape
    dev = y.device
    args = [_ptr(y, "y", torch.float32, (rows, n), dev), rows, n,
            _ptr(codes, "codes", torch.int8, (rows, n), dev),
            _ptr(scale, "scale", torch.float32, (rows,), dev), _stream_ptr(stream)]
    _check(lib().mla_prolog_quant_rows(*args), "mla_prolog_quant_rows")


def plan(d, sms: int) -> dict:
    """The schedule the library chooses for dims `d` on `sms` SMs (host only)."""
    dims = MlaPrologDims(d.T, d.D, d.q_lora_rank, d.kv_lora_rank, d.rope_dim, d.num_heads, d.nope_dim,
                         d.v_dim, d.max_pos, d.eps, d.flags)
    out = MlaPrologPlanInfo()
    _check(lib().mla_prolog_plan(ctypes.byref(dims), sms, ctypes.byref(out)), "mla_prolog_plan")
    return {n: getattr(out, n) for n, _ in MlaPrologPlanInfo._fields_}


def lpt(cost: Sequence[int], groups: int):
    """Longest-processing-time job assignment (host only): (per-worker job
    lists, largest worker load)."""
    n = len(cost)
    c = (ctypes.c_int64 * max(n, 1))(*cost)
    table = (ctypes.c_int32 * (groups + 1 + n))()
    busiest = ctypes.c_int64(0)
    _check(lib().mla_prolog_lpt(c, n, groups, table, ctypes.byref(busiest)), "mla_prolog_lpt")
    offs = list(table[:groups + 1])
    ids = list(table[groups + 1:])
    return [ids[offs[g]:offs[g + 1]] for g in range(groups)], busiest.value
