"""CPU-only checks of libtq.so: it loads, exports every declared symbol, builds the
same tables as the oracle, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from online_kv_cache_02_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    from online_kv_cache_02_gb300 import tq as mod
    return mod


def _declared():
    names = set()
    hdr_dir = os.path.join(ROOT, "include")
    for fn in os.listdir(hdr_dir):
        if fn.endswith(".h"):
            text = open(os.path.join(hdr_dir, fn)).read()
            names |= set(re.findall(r"^\s*(?:tq_status|const char\*)\s+(tq_\w+)\s*\(", text, re.M))
    return names


def test_every_declared_symbol_is_exported(tq):
    names = _declared()
    assert {"tq_create", "tq_quantize", "tq_decode_attention"} <= names
    lib = ctypes.CDLL(tq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert n in tq.EXPORTS, f"binding lacks {n}"


@pytest.mark.parametrize("seed", [0, 1, 123456789])
def test_rotation_matches_oracle(tq, seed):
    assert np.max(np.abs(tq.tq_host_rotation(128, seed) - oracle.rotation_matrix(128, seed))) < 1e-12


def test_qjl_matrix_matches_oracle(tq):
    assert np.max(np.abs(tq.tq_host_qjl(128, 128, 7) - oracle.qjl_matrix(128, 128, 7))) < 1e-14


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(tq, bits):
    c, t = tq.tq_host_codebook(bits)
    cb = oracle.lloyd_max_gaussian(bits)
    assert np.max(np.abs(c - cb.centroids)) < 1e-12
    assert np.max(np.abs(t - cb.boundaries)) < 1e-12
    assert t[(1 << bits) // 2 - 1] == 0.0


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_sphere_codebook_matches_oracle(tq, bits):
    """The library's rotated-coordinate codebook (incomplete beta by a continued fraction) against the
    oracle's (scipy's incomplete beta): equal to well inside the 1e-6 boundary band."""
    c, t = tq.tq_host_codebook_ex(bits, 128, tq.TQ_CODEBOOK_SPHERE)
    cb = oracle.lloyd_max_sphere(bits, 128)
    assert np.max(np.abs(c - cb.centroids)) < 1e-11
    assert np.max(np.abs(t - cb.boundaries)) < 1e-11
    g, _ = tq.tq_host_codebook_ex(bits, 128, tq.TQ_CODEBOOK_GAUSSIAN)
    assert np.array_equal(g, tq.tq_host_codebook(bits)[0])


def test_status_strings(tq):
    for s in range(7):
        assert tq.tq_status_string(s)
    assert "unknown" in tq.tq_status_string(99)


def test_config_validation_without_gpu(tq):
    st = tq.raw_status
    cfg = tq.TQConfig()
    assert st("tq_config_init", ctypes.byref(cfg), 128, 3, 128, 0) == tq.TQ_OK
    assert (cfg.k_bits_hi, cfg.k_split, cfg.page_size, cfg.k_qjl) == (3, 64, 16, 1)
    assert st("tq_config_init", ctypes.byref(cfg), 128, 5, 128, 0) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_config_init", ctypes.byref(cfg), 128, 3, 100, 0) == tq.TQ_ERR_INVALID_ARG
    for d in (48, 16, 288, 512):                      # head dims off the multiple-of-32 grid or above 256
        assert st("tq_config_init", ctypes.byref(cfg), d, 3, 128, 0) == tq.TQ_ERR_UNSUPPORTED
    for d, split in ((32, 0), (64, 32), (96, 32), (256, 128)):
        assert st("tq_config_init", ctypes.byref(cfg), d, 3, 128, 0) == tq.TQ_OK
        assert (cfg.d, cfg.k_split, cfg.v_split) == (d, split, split)
    out = ctypes.c_void_p()
    bad = tq.make_config(k_bits=(3, 3), v_bits=(3, 3), k_split=40)
    assert st("tq_create_ex", ctypes.byref(bad), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    bad = tq.make_config(k_bits=(0, 3))
    assert st("tq_create_ex", ctypes.byref(bad), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    bad = tq.make_config(codebook=2)                  # not a TQ_CODEBOOK_* density
    assert st("tq_create_ex", ctypes.byref(bad), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert cfg.codebook == tq.TQ_CODEBOOK_GAUSSIAN    # tq_config_init's default
    assert st("tq_create_ex", None, ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert out.value is None


def test_null_context_is_rejected(tq):
    st = tq.raw_status
    n = ctypes.c_size_t()
    assert st("tq_quantize", None, 1, 1, 0, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_workspace_size", None, 1, 1, 1, 16, ctypes.byref(n)) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_decode_attention", None, 1, 0, 1, 8, 1, 1, 16, 1, 1, 1, 1, 1, 16, ctypes.c_float(0.1), 1, 1,
              1024, None) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_destroy", None) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_check_device_status", None, None) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_cache_layout", None, 8, ctypes.byref(n), None) == tq.TQ_ERR_INVALID_ARG
    c = ctypes.c_int()
    assert st("tq_decode_chunk", None, 16, 32, 8, 16 * 1000, 1000, 0, ctypes.byref(c)) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_search_workspace_size", None, 4, 100, 10, ctypes.byref(n)) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_search_scores", None, 1, 0, 4, 1, 1, 8, 100, 10, 1, 1, 1 << 20, None) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_search", None, 1, 0, 4, 1, 1, 8, 100, 10, 1, 1, 1, 1 << 20, None) == tq.TQ_ERR_INVALID_ARG


def test_codebook_ex_arguments(tq):
    c, t = np.empty(16), np.empty(15)
    st = tq.raw_status
    assert st("tq_host_codebook_ex", 3, 128, 7, c.ctypes.data, t.ctypes.data) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_host_codebook_ex", 3, 3, tq.TQ_CODEBOOK_SPHERE, c.ctypes.data, t.ctypes.data) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_host_codebook_ex", 0, 128, tq.TQ_CODEBOOK_SPHERE, c.ctypes.data, t.ctypes.data) == tq.TQ_ERR_INVALID_ARG
    assert st("tq_host_codebook_ex", 3, 128, tq.TQ_CODEBOOK_SPHERE, None, t.ctypes.data) == tq.TQ_ERR_INVALID_ARG


@pytest.mark.parametrize("bits,d", [(3, 4), (4, 5), (3, 128)])
def test_sphere_codebook_small_d_matches_oracle(tq, bits, d):
    """The exact-density codebook at small d (support shorter than the Gaussian bulk) is finite and equals the
    oracle's."""
    c, t = tq.tq_host_codebook_ex(bits, d, tq.TQ_CODEBOOK_SPHERE)
    cb = oracle.lloyd_max_sphere(bits, d)
    assert np.all(np.isfinite(c)) and np.all(np.isfinite(t))
    assert np.max(np.abs(c - cb.centroids)) < 1e-10
    assert np.max(np.abs(t - cb.boundaries)) < 1e-10
