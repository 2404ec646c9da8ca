"""fp64 CPU oracle for batch decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The product path (``paged_kv_decode_23_gb300``)
never imports it, and this package never imports the product path: the two share no code.

The arithmetic lives in ``pkd_oracle.c`` (plain loops in double precision); this module only
compiles it with gcc and marshals numpy arrays through ctypes.  See the C file's header for
the definition it follows (FlashInfer attention API page, BatchDecodeWithPagedKVCacheWrapper
plan()/run()) and the readings it takes where that page is silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkd_oracle.so")
_lock = threading.Lock()
_lib = None

# dtype codes understood by the C oracle
F16, BF16, E4M3, F32, F64 = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile ``pkd_oracle.c`` into ``oracle/_build/libpkd_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            vp = ctypes.c_void_p
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_array.restype = ctypes.c_int
            lib.oracle_decode_array.argtypes = [vp, ctypes.c_int, ctypes.c_int64, vp]
            lib.oracle_kv_len.restype = ctypes.c_int
            lib.oracle_kv_len.argtypes = [i32p, i32p, ctypes.c_int, ctypes.c_int, vp]
            lib.oracle_merge_states.restype = ctypes.c_int
            lib.oracle_merge_states.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_batch_decode.restype = ctypes.c_int
            lib.oracle_batch_decode.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                i32p, i32p, i32p,
                vp, ctypes.c_int, vp, vp, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                vp, vp, ctypes.c_int]
            lib.oracle_batch_decode_q.restype = ctypes.c_int
            lib.oracle_batch_decode_q.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, i32p, i32p, i32p,
                vp, ctypes.c_int, vp, vp, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                vp, vp, ctypes.c_int]
            lib.oracle_batch_decode_pos.restype = ctypes.c_int
            lib.oracle_batch_decode_pos.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, i32p, i32p, i32p,
                vp, ctypes.c_int, vp, vp, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double,
                ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                vp, vp, ctypes.c_int]
            lib.oracle_mla_decode.restype = ctypes.c_int
            lib.oracle_mla_decode.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                i32p, i32p, i32p, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int,
                ctypes.c_double, vp, vp, ctypes.c_int]
            _lib = lib
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def decode_array(raw: np.ndarray, dtype_code: int) -> np.ndarray:
    """Decode raw element bit patterns (uint16 for fp16/bf16, uint8 for e4m3) to float64."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, dtype=np.float64)
    rc = _load().oracle_decode_array(raw.ctypes.data, dtype_code, raw.size, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode_array failed ({rc})")
    return out.reshape(raw.shape)


def kv_len(indptr, last_page_len, page_size: int) -> np.ndarray:
    indptr = _i32(indptr)
    lpl = _i32(last_page_len)
    out = np.empty(len(lpl), dtype=np.int64)
    _load().oracle_kv_len(_ptr_i32(indptr), _ptr_i32(lpl), len(lpl), page_size, out.ctypes.data)
    return out


def merge_states(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Combine partials ``o_parts [n, D]`` / ``lse_parts [n]`` (natural log) into (o, lse)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.empty(d, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    _load().oracle_merge_states(n, d, o_parts.ctypes.data, lse_parts.ctypes.data,
                                o.ctypes.data, lse.ctypes.data)
    return o, float(lse[0])


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def batch_decode(indptr, indices, last_page_len, q_raw: np.ndarray, q_dtype: int,
                 k_raw: np.ndarray, v_raw: np.ndarray, kv_dtype: int,
                 strides, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                 page_size: int, sm_scale: float | None = None,
                 logits_soft_cap: float = 0.0, window_left: int = -1,
                 q_scale: float = 1.0, k_scale: float = 1.0, v_scale: float = 1.0,
                 chunk_tokens: int = 0, num_threads: int = 0, q_len: int = 1,
                 pos_encoding_mode: str = "NONE", rope_scale: float = 1.0,
                 rope_theta: float = 1e4):
    """Batch decode attention in fp64.

    ``q_raw``: element bits of q ``[batch * q_len, num_qo_heads, head_dim]`` (contiguous,
    request-major; ``q_len`` query tokens per request, the last ``q_len`` positions, each
    masked causally).  ``pos_encoding_mode``: "NONE", "ROPE_LLAMA" (q rotated at its position,
    each key at its token index, pairs (i, i + D/2), angle pos / rope_scale *
    rope_theta^(-2i/D)) or "ALIBI" (slope_g * (t - pos) added to the scaled logit).
    ``k_raw`` / ``v_raw``: element bits of the key and value pools; ``strides`` =
    ``(page, slot, head)`` strides in elements, the head_dim axis contiguous.  For a 5-D pool,
    pass the same array twice with ``v_raw`` offset by the K/V stride (see ``tests``).
    Returns ``(o [batch * q_len, num_qo_heads, head_dim] float64, lse [batch * q_len,
    num_qo_heads] float64)``.
    """
    indptr = _i32(indptr)
    indices = _i32(indices) if len(indices) else np.zeros(1, dtype=np.int32)
    lpl = _i32(last_page_len)
    batch = len(lpl)
    assert len(indptr) == batch + 1
    q_raw = np.ascontiguousarray(q_raw)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(head_dim)
    rows = batch * int(q_len)
    o = np.zeros((rows, num_qo_heads, head_dim), dtype=np.float64)
    lse = np.zeros((rows, num_qo_heads), dtype=np.float64)
    ps, ss, hs = (int(s) for s in strides)
    k_ptr = k_raw.ctypes.data if isinstance(k_raw, np.ndarray) else int(k_raw)
    v_ptr = v_raw.ctypes.data if isinstance(v_raw, np.ndarray) else int(v_raw)
    mode = {"NONE": 0, "ROPE_LLAMA": 1, "ALIBI": 2}[pos_encoding_mode]
    rc = _load().oracle_batch_decode_pos(
        batch, int(q_len), num_qo_heads, num_kv_heads, head_dim, page_size,
        _ptr_i32(indptr), _ptr_i32(indices), _ptr_i32(lpl),
        q_raw.ctypes.data, q_dtype, k_ptr, v_ptr, kv_dtype, ps, ss, hs,
        float(sm_scale), float(logits_soft_cap or 0.0), int(window_left),
        float(q_scale), float(k_scale), float(v_scale), mode,
        float(1.0 if rope_scale is None else rope_scale),
        float(1e4 if rope_theta is None else rope_theta), int(chunk_tokens),
        o.ctypes.data, lse.ctypes.data, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_batch_decode rejected the problem (code {rc})")
    return o, lse


def batch_decode_pool(indptr, indices, last_page_len, q_raw, q_dtype, pool_raw: np.ndarray,
                      kv_dtype: int, layout: str, **kw):
    """Convenience form for a 5-D pool ``[pages, 2, ...]`` in NHD or HND layout.

    Element strides are read off the array's shape; K is ``pool[:, 0]`` and V ``pool[:, 1]``.
    ``num_qo_heads`` defaults to ``q_raw.shape[1]``.
    """
    pool_raw = np.ascontiguousarray(pool_raw)
    _, two, a, b, head_dim = pool_raw.shape
    assert two == 2
    if layout == "NHD":
        page_size, num_kv_heads = a, b
        strides = (2 * a * b * head_dim, b * head_dim, head_dim)
    elif layout == "HND":
        num_kv_heads, page_size = a, b
        strides = (2 * a * b * head_dim, head_dim, b * head_dim)
    else:
        raise ValueError(layout)
    base = pool_raw.ctypes.data
    v_base = base + a * b * head_dim * pool_raw.itemsize
    num_qo_heads = kw.pop("num_qo_heads", q_raw.shape[1])
    return batch_decode(indptr, indices, last_page_len, q_raw, q_dtype, base, v_base, kv_dtype,
                        strides, num_qo_heads, num_kv_heads, head_dim, page_size, **kw)


def mla_decode(kv_indptr, kv_indices, kv_len, q_nope_raw: np.ndarray, q_pe_raw: np.ndarray,
               q_dtype: int, ckv_raw: np.ndarray, kpe_raw: np.ndarray, kv_dtype: int,
               page_size: int, sm_scale: float, num_threads: int = 0):
    """MLA paged decode in fp64 (BatchMLAPagedAttentionWrapper): key = [ckv, kpe], value = ckv.

    ``q_nope_raw`` ``[batch, H, Dc]`` and ``q_pe_raw`` ``[batch, H, Dp]``, ``ckv_raw``
    ``[pages, page_size, Dc]`` and ``kpe_raw`` ``[pages, page_size, Dp]``: element bits.
    Returns ``(o [batch, H, Dc] float64, lse [batch, H] float64, natural log)``.
    """
    kv_indptr = _i32(kv_indptr)
    kv_indices = _i32(kv_indices) if len(kv_indices) else np.zeros(1, dtype=np.int32)
    kv_len = _i32(kv_len)
    q_nope_raw = np.ascontiguousarray(q_nope_raw)
    q_pe_raw = np.ascontiguousarray(q_pe_raw)
    ckv_raw = np.ascontiguousarray(ckv_raw)
    kpe_raw = np.ascontiguousarray(kpe_raw)
    batch, heads, dc = q_nope_raw.shape
    dp = q_pe_raw.shape[2]
    o = np.zeros((batch, heads, dc), dtype=np.float64)
    lse = np.zeros((batch, heads), dtype=np.float64)
    rc = _load().oracle_mla_decode(batch, heads, dc, dp, int(page_size), _ptr_i32(kv_indptr),
                                   _ptr_i32(kv_indices), _ptr_i32(kv_len), q_nope_raw.ctypes.data,
                                   q_pe_raw.ctypes.data, q_dtype, ckv_raw.ctypes.data,
                                   kpe_raw.ctypes.data, kv_dtype, float(sm_scale),
                                   o.ctypes.data, lse.ctypes.data, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode rejected the problem (code {rc})")
    return o, lse
