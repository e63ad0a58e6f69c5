"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and rejects bad arguments before any CUDA
call."""
import ctypes
import os
import re

import pytest

from mla_attention_prolog_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_prolog.h")


@pytest.fixture(scope="module")
def L():
    from mla_attention_prolog_gb300 import build
    build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_prolog_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_prolog_create", "mla_prolog_run", "mla_prolog_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    assert sorted(binding.EXPORTED) == sorted(declared_functions())


def test_strerror_covers_codes(L):
    for c in (0, -1, -2, -3, -4, -5):
        assert len(L.mla_prolog_strerror(c)) > 0
    assert L.mla_prolog_strerror(-99) == b"unknown error code"


def _dims(**kw):
    base = dict(T=4, D=256, q_lora_rank=0, kv_lora_rank=64, rope_dim=16, num_heads=2,
                nope_dim=32, v_dim=32, max_pos=4, eps=1e-6, flags=0)
    base.update(kw)
    return binding.MlaPrologDims(*[base[f] for f, _ in binding.MlaPrologDims._fields_])


@pytest.mark.parametrize("kw,code", [
    (dict(D=100), -2), (dict(kv_lora_rank=0), -2), (dict(rope_dim=24), -2), (dict(nope_dim=8), -2),
    (dict(rope_dim=144), -2), (dict(T=-1), -2), (dict(num_heads=0), -2), (dict(max_pos=0), -2),
    (dict(eps=float("nan")), -2), (dict(eps=-1.0), -2), (dict(q_lora_rank=24, flags=1), -2),
    (dict(q_lora_rank=64, flags=0), -1), (dict(flags=1), -1), (dict(flags=4), -1),
    (dict(q_lora_rank=64, flags=1, nope_dim=256, rope_dim=64), -2),
    (dict(flags=8), -1), (dict(flags=2 | 4), -1), (dict(flags=32), -1),   # q variants without a q path; unknown
    (dict(flags=16, kv_lora_rank=2064), -2), (dict(q_lora_rank=2064, flags=1 | 16), -2),  # W8A8: K <= 2048
    (dict(q_lora_rank=64, flags=1 | 32), -1), (dict(q_lora_rank=64, flags=8), -1),
    (dict(T=2**27), -2), (dict(T=2**24), -2),  # T * H * (Dn + R + Dv) > 4e9; T * D > 4e9
])
def test_create_rejects_bad_dims_without_touching_cuda(L, kw, code):
    h = ctypes.c_void_p()
    d = _dims(**kw)
    assert L.mla_prolog_create(ctypes.byref(d), ctypes.byref(h)) == code
    assert not h.value


def test_null_arguments(L):
    h = ctypes.c_void_p()
    assert L.mla_prolog_create(None, ctypes.byref(h)) == -1
    assert L.mla_prolog_run(None, *([None] * 12)) == -1
    assert L.mla_prolog_run_cached(None, *([None] * 13), 0, None) == -1
    assert L.mla_prolog_destroy(None) == 0
    st = ctypes.c_int32()
    assert L.mla_prolog_device_status(None, None, ctypes.byref(st)) == -1
    assert L.mla_prolog_set_wait_timeout(None, 5) == -1
    assert L.mla_prolog_kernel_count(None) == 0
    assert L.mla_prolog_kernel_name(None, 0) == b""


def test_quant_rows_validates_before_launch(L):
    assert L.mla_prolog_quant_rows(None, 4, 6, None, None, None) == -1   # row_len % 4
    assert L.mla_prolog_quant_rows(None, -1, 8, None, None, None) == -1
    assert L.mla_prolog_quant_rows(None, 0, 8, None, None, None) == 0     # empty: no-op
    assert L.mla_prolog_quant_rows(ctypes.c_void_p(8), 2, 8, None, None, None) == -1
    assert L.mla_prolog_quant_rows(ctypes.c_void_p(20), 2, 8, ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), None) == -1       # y not 16-B aligned


def test_flag_bits_agree_across_header_binding_and_inputs():
    """One set of flag bits: the header's, the binding's and the input module's."""
    src = open(HEADER).read()
    from mla_attention_prolog_gb300 import workloads as wl
    for name, py, w in (("QUANT_Q", binding.MLA_PROLOG_QUANT_Q, wl.QUANT_Q),
                        ("ROPE_INTERLEAVED", binding.MLA_PROLOG_ROPE_INTERLEAVED, wl.ROPE_INTERLEAVED),
                        ("Q_HEAD_NORM", binding.MLA_PROLOG_Q_HEAD_NORM, wl.Q_HEAD_NORM),
                        ("QUANT_PER_HEAD", binding.MLA_PROLOG_QUANT_PER_HEAD, wl.QUANT_PER_HEAD),
                        ("W8A8", binding.MLA_PROLOG_W8A8, wl.W8A8)):
        m = re.search(r"#define MLA_PROLOG_%s\s+(0x[0-9a-fA-F]+)u" % name, src)
        assert m and int(m.group(1), 16) == py == w, name
    m = re.search(r"#define MLA_STATUS_SLOT_RANGE\s+(0x[0-9a-fA-F]+)", src)
    assert m and int(m.group(1), 16) == binding.STATUS_SLOT_RANGE


def test_oracle_flag_bits_match():
    import oracle
    from mla_attention_prolog_gb300 import workloads as wl
    assert (oracle.QUANT_Q, oracle.ROPE_INTERLEAVED, oracle.Q_HEAD_NORM, oracle.QUANT_PER_HEAD, oracle.W8A8) == \
        (wl.QUANT_Q, wl.ROPE_INTERLEAVED, wl.Q_HEAD_NORM, wl.QUANT_PER_HEAD, wl.W8A8)


def test_w8a8_is_not_taken_by_the_noalloc_entry(L):
    d = _dims(flags=16)
    assert L.mla_prolog_run_noalloc(ctypes.byref(d), *([None] * 13)) == -1


def test_w8a8_load_needs_a_handle(L):
    assert L.mla_prolog_load_w8a8(None, None, None, None, None) == -1
