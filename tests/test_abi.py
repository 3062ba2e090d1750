"""The C ABI library builds, loads without a GPU and exports every entry point
the header declares; host-side argument checks answer without touching CUDA."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from llama2_decoder_forward_gb300 import binding, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.lib()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(llama_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(binding.exported_symbols())


def test_strerror(lib):
    assert lib.llama_strerror(0) == b"ok"
    assert b"argument" in lib.llama_strerror(1)
    assert lib.llama_strerror(999) == b"unknown status"


def _cfg(**kw):
    c = binding.make_config(synth.LLAMA2_7B, 32, 4096, 4096)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_workspace_bytes_and_config_checks(lib):
    n = ctypes.c_size_t()
    assert lib.llama_workspace_bytes(ctypes.byref(_cfg()), ctypes.byref(n)) == 0
    assert n.value > 0 and n.value % 256 == 0
    bad = [dict(n_kv_heads=5), dict(hidden=0), dict(dtype=7), dict(head_dim=64),  # bf16 wants d=128
           dict(max_batch=0), dict(rms_eps=0.0), dict(hidden=4100)]
    codes = [1, 1, 1, 2, 1, 1, 2]
    for kw, code in zip(bad, codes):
        assert lib.llama_workspace_bytes(ctypes.byref(_cfg(**kw)), ctypes.byref(n)) == code, kw
    assert lib.llama_workspace_bytes(None, ctypes.byref(n)) == 1
    tiny = binding.make_config(synth.TINY, 1, 16, 32)
    assert lib.llama_workspace_bytes(ctypes.byref(tiny), ctypes.byref(n)) == 0


def test_e4m3_weight_config_and_quantiser_argument_checks(lib):
    n = ctypes.c_size_t()
    w8 = _cfg(weight_dtype=binding.W_E4M3)
    assert lib.llama_workspace_bytes(ctypes.byref(w8), ctypes.byref(n)) == 0
    assert lib.llama_workspace_bytes(ctypes.byref(_cfg(weight_dtype=2)), ctypes.byref(n)) == 1
    # E4M3 projections need a bf16 model and 16-byte rows of bytes
    tiny = binding.make_config(synth.TINY, 1, 16, 32, weight_dtype=binding.W_E4M3)  # fp32
    assert lib.llama_workspace_bytes(ctypes.byref(tiny), ctypes.byref(n)) == 2
    assert lib.llama_workspace_bytes(ctypes.byref(_cfg(weight_dtype=1, intermediate=11000)),
                                     ctypes.byref(n)) == 2
    # the quantiser rejects bad arguments before touching the device
    buf = ctypes.create_string_buffer(4096 + 16)
    al = (ctypes.addressof(buf) + 15) // 16 * 16
    q = lib.llama_quantize_rows_e4m3
    assert q(None, 4, 64, al, al, None) == 1
    assert q(al, 0, 64, al, al, None) == 1
    assert q(al, 4, 40, al, al, None) == 1       # rows of 40 bytes
    assert q(al + 8, 4, 64, al, al, None) == 1   # misaligned source
    assert q(al, 4, 64, al, al + 2, None) == 1   # misaligned scales


def test_null_context_and_arguments_rejected(lib):
    kv = binding.KV()
    assert lib.llama_decode_step(None, None, None, 1, ctypes.byref(kv), None, None) == 1
    assert lib.llama_prefill(None, None, 1, 1, ctypes.byref(kv), None, None) == 1
    assert lib.llama_sync_status(None) == 1
    assert lib.llama_check_wait_timeout(None, 1000) == 1
    assert lib.llama_free(None) == 1
    assert lib.llama_launch_count(None) == 0
    sp = binding.Sampling(1.0, 0, 1.0, 1.0)
    assert lib.llama_sample(None, None, 1, 8, ctypes.byref(sp), None, None, 0, None, None) == 1
    out = ctypes.c_void_p()
    w = binding.Weights()
    assert lib.llama_init(ctypes.byref(_cfg()), ctypes.byref(w), None, 0, None, ctypes.byref(out)) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_bounds_check_build_exports_everything_and_reports_itself(lib):
    from llama2_decoder_forward_gb300 import build as b
    path = b.build_library(checked=True)
    checked = ctypes.CDLL(path)
    for n in sorted(_declared()):
        assert hasattr(checked, n), n
    checked.llama_bounds_checked.restype = ctypes.c_int32
    assert checked.llama_bounds_checked() == 1
    assert lib.llama_bounds_checked() == 0
