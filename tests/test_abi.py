"""The C-ABI library builds for sm_103a, loads, and exports every entry point the header
declares; the binding's signature table covers the same set. No GPU needed (no compute)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(qw_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    import decode_qwen3_decoder_gb300 as pkg
    path = pkg._build_lib()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for fn in ("qw_init_weights", "qw_prefill", "qw_decode_step", "qw_decode_steps", "qw_kv_alloc", "qw_kv_reset",
               "qw_kv_reserve", "qw_generate", "qw_sync_status", "qw_last_error"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header():
    from decode_qwen3_decoder_gb300 import qw
    assert set(qw.SIGNATURES) == _declared()


def test_binding_constants_match_header():
    """Every QW_OPT_* option, QW_PROF_* kind and QW_MAX_GRAPH_STEPS the binding defines has the
    header's value."""
    from decode_qwen3_decoder_gb300 import qw
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    vals = {k: int(v) for k, v in re.findall(r"\b(QW_(?:OPT|PROF)_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    vals.update({k: int(v) for k, v in re.findall(r"#define\s+(QW_[A-Z0-9_]+)\s+(\d+)", src)})
    names = [n for n in dir(qw) if n.startswith(("QW_OPT_", "QW_PROF_")) or n == "QW_MAX_GRAPH_STEPS"]
    assert "QW_MAX_GRAPH_STEPS" in names and "QW_OPT_BATCH1_CLUSTERS" in names
    for n in names:
        assert n in vals and getattr(qw, n) == vals[n], n


def test_host_only_calls_without_gpu(lib):
    """Entry points that touch no device: config validation and error strings."""
    from decode_qwen3_decoder_gb300 import qw
    import synth
    qw.load()
    cfg = qw.make_config(synth.QWEN3_0_6B, max_tokens=64, max_batch=8, max_context=2048)
    assert qw.qw_model_workspace_bytes(cfg) > 0
    bad = qw.make_config(synth.QWEN3_0_6B, max_tokens=64, max_batch=8, max_context=2048)
    bad.head_dim = 64
    assert qw.qw_model_workspace_bytes(bad) == 0
    bad2 = qw.make_config(synth.TINY, max_tokens=64, max_batch=8, max_context=64)
    assert qw.qw_model_workspace_bytes(bad2) == 0   # head_dim 16 is not built
    out = ctypes.c_void_p()
    st = qw.load().qw_init_weights(ctypes.byref(cfg), None, None, 0, None, ctypes.byref(out))
    assert st == -1 and out.value is None
    assert "weight pointers" in qw.qw_last_error() or "NULL" in qw.qw_last_error()
    assert qw.qw_kv_length(None, 0) == -1
    assert qw.qw_kv_free_pages(None) == -1


def test_decode_calls_refuse_bad_arguments_on_the_host(lib):
    """qw_decode_step / qw_decode_steps check their arguments before touching the device:
    NULL buffers, step counts outside [1, QW_MAX_GRAPH_STEPS] and a NULL model are refused
    with QW_ERR_INVALID_ARG and a message."""
    from decode_qwen3_decoder_gb300 import qw
    L = qw.load()
    seqs = (ctypes.c_int * 1)(0)
    buf = ctypes.c_void_p(16)   # never dereferenced: every call below is refused first
    assert L.qw_decode_step(None, None, 1, seqs, None, None, buf, None) == -1
    assert "NULL" in qw.qw_last_error()
    for n in (0, -3, qw.QW_MAX_GRAPH_STEPS + 1):
        assert L.qw_decode_steps(None, None, 1, seqs, n, buf, buf, None) == -1
        assert "n_steps" in qw.qw_last_error()
    assert L.qw_decode_steps(None, None, 1, seqs, 1, None, buf, None) == -1
    assert "NULL" in qw.qw_last_error()
    assert L.qw_decode_steps(None, None, 1, seqs, 4, buf, buf, None) == -1
    assert "NULL" in qw.qw_last_error()   # model or kv
