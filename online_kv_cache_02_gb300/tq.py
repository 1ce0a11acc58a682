"""ctypes binding of libtq.so: the C ABI in include/tq.h, same names.

Argument marshalling only.  Pointer arguments accept an int address, None
(NULL), or any object with ``data_ptr()`` (e.g. a torch tensor); stream
arguments accept an int handle or an object with ``cuda_stream``.  Every call
raises TQError on a non-OK status.  Importing this module loads the in-tree
library and fails loudly if it has not been built: there is no fallback.
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtq.so")

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_CUDA = 2
TQ_ERR_OOM = 3
TQ_ERR_UNSUPPORTED = 4
TQ_ERR_DEVICE_CHECK = 5
TQ_ERR_WORKSPACE = 6
TQ_BF16 = 0
TQ_F32 = 1


class TQError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        extra = f" [{tq_last_cuda_error()}]" if status == TQ_ERR_CUDA else ""
        super().__init__(f"{fn}: {tq_status_string(status)} (status {status}){extra}")


class TQConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("m", ctypes.c_int), ("page_size", ctypes.c_int),
                ("k_bits_hi", ctypes.c_int), ("k_bits_lo", ctypes.c_int), ("k_split", ctypes.c_int),
                ("v_bits_hi", ctypes.c_int), ("v_bits_lo", ctypes.c_int), ("v_split", ctypes.c_int),
                ("k_qjl", ctypes.c_int), ("seed", ctypes.c_uint64), ("codebook", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtq.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
    return ctypes.CDLL(LIB_PATH)


_lib = _load()
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64
_S = ctypes.c_int

EXPORTS = {
    "tq_config_init": ([ctypes.POINTER(TQConfig), _I, _I, _I, _U64], _S),
    "tq_create": ([_I, _I, _I, _U64, ctypes.POINTER(_P)], _S),
    "tq_create_ex": ([ctypes.POINTER(TQConfig), ctypes.POINTER(_P)], _S),
    "tq_destroy": ([_P], _S),
    "tq_get_config": ([_P, ctypes.POINTER(TQConfig)], _S),
    "tq_cache_layout": ([_P, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)], _S),
    "tq_host_rotation": ([_I, _U64, _P], _S),
    "tq_host_qjl": ([_I, _I, _U64, _P], _S),
    "tq_host_codebook": ([_I, _P, _P], _S),
    "tq_host_codebook_ex": ([_I, _I, _I, _P, _P], _S),
    "tq_search_workspace_size": ([_P, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)], _S),
    "tq_search": ([_P, _P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, ctypes.c_size_t, _P], _S),
    "tq_search_scores": ([_P, _P, _I, _I, _P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t, _P], _S),
    "tq_quantize": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P], _S),
    "tq_workspace_size": ([_P, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _S),
    "tq_decode_chunk": ([_P, _I, _I, _I, ctypes.c_longlong, _I, _I, ctypes.POINTER(_I)], _S),
    "tq_decode_attention": ([_P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float,
                             _P, _P, _SZ, _P], _S),
    "tq_decode_attention_ex": ([_P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float,
                                _P, _P, _SZ, _I, _P], _S),
    "tq_decode_attention_noalloc": ([_P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float,
                                     _P, _P], _S),
    "tq_append_decode": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float, _P,
                          _P, _SZ, _P], _S),
    "tq_append_decode_ex": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float, _P,
                             _P, _SZ, _P, _P, _P], _S),
    "tq_causal_workspace_size": ([_P, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _S),
    "tq_causal_attention": ([_P, _P, _I, _I, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _I, ctypes.c_float, _P, _P, _SZ,
                             _P], _S),
    "tq_check_device_status": ([_P, ctypes.POINTER(ctypes.c_uint32)], _S),
    "tq_refine_counters": ([_P, ctypes.POINTER(ctypes.c_ulonglong), _I], _S),
    "tq_status_string": ([_S], ctypes.c_char_p),
    "tq_last_cuda_error": ([], ctypes.c_char_p),
}
for _name, (_args, _res) in EXPORTS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)!r} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, st):
    if st != TQ_OK:
        raise TQError(fn, st)


def tq_status_string(status):
    return _lib.tq_status_string(status).decode()


def tq_last_cuda_error():
    return _lib.tq_last_cuda_error().decode()


def tq_config_init(d, b, m, seed):
    cfg = TQConfig()
    _check("tq_config_init", _lib.tq_config_init(ctypes.byref(cfg), d, b, m, seed))
    return cfg


TQ_CODEBOOK_GAUSSIAN, TQ_CODEBOOK_SPHERE = 0, 1


def make_config(k_bits=(3, 3), v_bits=(3, 3), m=128, seed=0, k_split=64, v_split=64, k_qjl=True, d=128,
                codebook=TQ_CODEBOOK_GAUSSIAN):
    return TQConfig(d, m, 16, k_bits[0], k_bits[1], k_split, v_bits[0], v_bits[1], v_split, int(k_qjl), seed,
                    codebook)


def tq_create(d, b, m, seed):
    out = _P()
    _check("tq_create", _lib.tq_create(d, b, m, seed, ctypes.byref(out)))
    return out.value


def tq_create_ex(cfg):
    out = _P()
    _check("tq_create_ex", _lib.tq_create_ex(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def tq_destroy(ctx):
    _check("tq_destroy", _lib.tq_destroy(ctx))


def tq_get_config(ctx):
    cfg = TQConfig()
    _check("tq_get_config", _lib.tq_get_config(ctx, ctypes.byref(cfg)))
    return cfg


def tq_cache_layout(ctx, num_kv_heads):
    k, v = _SZ(), _SZ()
    _check("tq_cache_layout", _lib.tq_cache_layout(ctx, num_kv_heads, ctypes.byref(k), ctypes.byref(v)))
    return k.value, v.value


def tq_host_rotation(d, seed):
    out = np.empty((d, d), dtype=np.float64)
    _check("tq_host_rotation", _lib.tq_host_rotation(d, seed, out.ctypes.data))
    return out


def tq_host_qjl(m, d, seed):
    out = np.empty((m, d), dtype=np.float64)
    _check("tq_host_qjl", _lib.tq_host_qjl(m, d, seed, out.ctypes.data))
    return out


def tq_host_codebook(bits):
    c = np.empty(1 << bits, dtype=np.float64)
    t = np.empty((1 << bits) - 1 if bits > 0 else 1, dtype=np.float64)
    _check("tq_host_codebook", _lib.tq_host_codebook(bits, c.ctypes.data, t.ctypes.data))
    return c, t


def tq_host_codebook_ex(bits, d, density):
    c = np.empty(1 << bits, dtype=np.float64)
    t = np.empty((1 << bits) - 1 if bits > 0 else 1, dtype=np.float64)
    _check("tq_host_codebook_ex", _lib.tq_host_codebook_ex(bits, d, density, c.ctypes.data, t.ctypes.data))
    return c, t


def tq_quantize(ctx, k, v, dtype, batch, n_new, num_kv_heads, start_pos, block_table,
                max_pages_per_seq, num_pages, k_cache, v_cache, stream=None):
    _check("tq_quantize", _lib.tq_quantize(ctx, _ptr(k), _ptr(v), dtype, batch, n_new, num_kv_heads,
                                           _ptr(start_pos), _ptr(block_table), max_pages_per_seq, num_pages,
                                           _ptr(k_cache), _ptr(v_cache), _stream(stream)))


def tq_decode_chunk(ctx, batch, num_q_heads, num_kv_heads, total_tokens, max_seq_len, fused_append=False):
    out = _I(0)
    _check("tq_decode_chunk", _lib.tq_decode_chunk(ctx, batch, num_q_heads, num_kv_heads, int(total_tokens),
                                                   max_seq_len, int(bool(fused_append)), ctypes.byref(out)))
    return out.value


def tq_workspace_size(ctx, batch, num_q_heads, max_seq_len, chunk_tokens=0):
    n = _SZ()
    _check("tq_workspace_size", _lib.tq_workspace_size(ctx, batch, num_q_heads, max_seq_len, chunk_tokens,
                                                       ctypes.byref(n)))
    return n.value


def tq_decode_attention(ctx, q, dtype, batch, num_q_heads, num_kv_heads, seq_lens, max_seq_len, block_table,
                        max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens, softmax_scale, out,
                        workspace, workspace_bytes, stream=None):
    _check("tq_decode_attention", _lib.tq_decode_attention(
        ctx, _ptr(q), dtype, batch, num_q_heads, num_kv_heads, _ptr(seq_lens), max_seq_len, _ptr(block_table),
        max_pages_per_seq, num_pages, _ptr(k_cache), _ptr(v_cache), chunk_tokens, softmax_scale, _ptr(out),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def tq_append_decode(ctx, k_new, v_new, q, dtype, batch, num_q_heads, num_kv_heads, seq_lens, max_seq_len,
                     block_table, max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens, softmax_scale, out,
                     workspace, workspace_bytes, stream=None, partials_events=None):
    """partials_events: optional (begin, end) CUDA event handles (ints) recorded around the partials kernel."""
    ev0, ev1 = partials_events if partials_events else (None, None)
    _check("tq_append_decode_ex", _lib.tq_append_decode_ex(
        ctx, _ptr(k_new), _ptr(v_new), _ptr(q), dtype, batch, num_q_heads, num_kv_heads, _ptr(seq_lens), max_seq_len,
        _ptr(block_table), max_pages_per_seq, num_pages, _ptr(k_cache), _ptr(v_cache), chunk_tokens, softmax_scale,
        _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream), ev0, ev1))


TQ_STAGE_QPREP, TQ_STAGE_PARTIALS, TQ_STAGE_MERGE, TQ_STAGE_ALL = 1, 2, 4, 7


def tq_decode_attention_ex(ctx, q, dtype, batch, num_q_heads, num_kv_heads, seq_lens, max_seq_len, block_table,
                           max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens, softmax_scale, out,
                           workspace, workspace_bytes, stages, stream=None):
    _check("tq_decode_attention_ex", _lib.tq_decode_attention_ex(
        ctx, _ptr(q), dtype, batch, num_q_heads, num_kv_heads, _ptr(seq_lens), max_seq_len, _ptr(block_table),
        max_pages_per_seq, num_pages, _ptr(k_cache), _ptr(v_cache), chunk_tokens, softmax_scale, _ptr(out),
        _ptr(workspace), workspace_bytes, stages, _stream(stream)))


def tq_decode_attention_noalloc(ctx, q, dtype, batch, num_q_heads, num_kv_heads, seq_lens, max_seq_len,
                                block_table, max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens,
                                softmax_scale, out, stream=None):
    """Decode attention with the library's fixed device scratch instead of a caller workspace."""
    _check("tq_decode_attention_noalloc", _lib.tq_decode_attention_noalloc(
        ctx, _ptr(q), dtype, batch, num_q_heads, num_kv_heads, _ptr(seq_lens), max_seq_len, _ptr(block_table),
        max_pages_per_seq, num_pages, _ptr(k_cache), _ptr(v_cache), chunk_tokens, softmax_scale, _ptr(out),
        _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20


def tq_check_device_status(ctx):
    """Returns the device error flags (0 when clean); raises only on CUDA errors."""
    flags = ctypes.c_uint32(0)
    st = _lib.tq_check_device_status(ctx, ctypes.byref(flags))
    if st not in (TQ_OK, TQ_ERR_DEVICE_CHECK):
        raise TQError("tq_check_device_status", st)
    return flags.value


def tq_refine_counters(ctx, reset=False):
    out = (ctypes.c_ulonglong * 2)()
    _check("tq_refine_counters", _lib.tq_refine_counters(ctx, out, int(reset)))
    return int(out[0]), int(out[1])


def raw_status(fn_name, *args):
    """Call an export with already-marshalled arguments and return its status (for argument-check tests)."""
    return getattr(_lib, fn_name)(*args)


def tq_causal_workspace_size(ctx, batch, n_new, num_q_heads, max_seq_len, chunk_tokens=0):
    n = ctypes.c_size_t()
    _check("tq_causal_workspace_size", _lib.tq_causal_workspace_size(ctx, batch, n_new, num_q_heads, max_seq_len,
                                                                     chunk_tokens, ctypes.byref(n)))
    return n.value


def tq_causal_attention(ctx, q, dtype, batch, n_new, num_q_heads, num_kv_heads, start_pos, max_seq_len, block_table,
                        max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens, softmax_scale, out, workspace,
                        workspace_bytes, stream=None):
    _check("tq_causal_attention", _lib.tq_causal_attention(
        ctx, _ptr(q), dtype, batch, n_new, num_q_heads, num_kv_heads, _ptr(start_pos), max_seq_len,
        _ptr(block_table), max_pages_per_seq, num_pages, _ptr(k_cache), _ptr(v_cache), chunk_tokens,
        ctypes.c_float(softmax_scale), _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def tq_search_workspace_size(ctx, nq, n_db, k_top):
    """Workspace bytes of tq_search with this k_top (0: of tq_search_scores)."""
    n = ctypes.c_size_t()
    _check("tq_search_workspace_size", _lib.tq_search_workspace_size(ctx, nq, n_db, k_top, ctypes.byref(n)))
    return n.value


def tq_search(ctx, q, dtype, nq, k_cache, block_table, num_pages, n_db, k_top, top_scores, top_index,
              workspace, workspace_bytes, stream=None):
    """Inner-product search: the k_top best database vectors per query (see tq.h)."""
    _check("tq_search", _lib.tq_search(ctx, _ptr(q), dtype, nq, _ptr(k_cache), _ptr(block_table), num_pages, n_db,
                                       k_top, _ptr(top_scores), _ptr(top_index), _ptr(workspace), workspace_bytes,
                                       _stream(stream)))


def tq_search_scores(ctx, q, dtype, nq, k_cache, block_table, num_pages, n_db, k_top, scores, workspace,
                     workspace_bytes, stream=None):
    """Every score [nq][n_db] of the search, by the arithmetic tq_search uses for this k_top (see tq.h)."""
    _check("tq_search_scores", _lib.tq_search_scores(ctx, _ptr(q), dtype, nq, _ptr(k_cache), _ptr(block_table),
                                                     num_pages, n_db, k_top, _ptr(scores), _ptr(workspace),
                                                     workspace_bytes, _stream(stream)))
