"""pkd_decode_noalloc: the entry point for callers that cannot allocate device memory.

A runtime that owns every device allocation (its own pool or memory budget) cannot let a
plug-in call cudaMalloc, and may have no workspace to lend either.  pkd_decode_noalloc plans
and runs in one call with scratch built into the library.  These tests call it through the C
ABI: twice in a row on two different batches (the second reuses scratch the first left
behind), checking each result against the fp64 oracle and against the handle-based plan/run
path within the same tolerances as the other parity tests; on e4m3 KV with head_dim 256, a
soft cap and a window; and on a batch whose work list cannot fit the built-in scratch.  They
live in a file of their own, collected last, and pass alone in a fresh process as well as
after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from helpers import LSE_ATOL, TOL, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

_CODE = {"f16": 0, "bf16": 1, "e4m3": 2}


def _noalloc(w, q, pool, disable_split_kv=None):
    from paged_kv_decode_23_gb300 import _lib as L
    dev = torch.device("cuda")
    q = q.to(dev).contiguous()
    pool = pool.to(dev).contiguous()
    indices = torch.from_numpy(w.indices).to(dev)
    o = torch.empty(q.shape, dtype=W.TORCH_DTYPES[w.o_dtype], device=dev)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    if w.layout == "NHD":
        strides = (pool.stride(0), pool.stride(2), pool.stride(3))
    else:
        strides = (pool.stride(0), pool.stride(3), pool.stride(2))
    ip = np.ascontiguousarray(w.indptr, dtype=np.int32)
    lpl = np.ascontiguousarray(w.last_page_len, dtype=np.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    sm = float("nan") if w.sm_scale is None else float(w.sm_scale)
    rc = L.lib().pkd_decode_noalloc(
        ip.ctypes.data_as(i32p), lpl.ctypes.data_as(i32p), w.batch, indices.data_ptr(),
        indices.numel(), w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, sm,
        float(w.logits_soft_cap or 0.0), w.window_left, w.fixed_split_size,
        int(w.disable_split_kv if disable_split_kv is None else disable_split_kv),
        _CODE[w.q_dtype], _CODE[w.kv_dtype], _CODE[w.o_dtype], -1,
        0 if w.layout == "NHD" else 1, q.data_ptr(), pool.data_ptr(),
        pool.data_ptr() + pool.stride(1) * pool.element_size(), pool.shape[0],
        (ctypes.c_int64 * 3)(*strides), 1.0, float(w.k_scale), float(w.v_scale),
        o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    L.check(rc)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def _compare(w, got, ref):
    atol, rtol = TOL[w.kv_dtype]
    o, lse = got
    ro, rl = ref
    assert np.all(np.abs(o - ro) <= atol + rtol * np.abs(ro)), \
        f"o differs by up to {np.abs(o - ro).max():.3e}"
    neg = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - rl[~neg]) <= LSE_ATOL)


def test_noalloc_matches_oracle_and_handle_path_on_two_calls_in_a_row():
    from paged_kv_decode_23_gb300 import noalloc_check_status
    # first call: split requests (partials in the built-in scratch), bf16, NHD
    w1 = W.custom([3000, 17, 0, 1200, 4096, 64, 1], 16, 2, 128, 16, layout="NHD",
                  q_dtype="bf16", seed=21, fixed_split_size=16)
    q1, p1 = W.make_q(w1), W.make_pool(w1)
    # second call: other shapes and dtypes, heuristic split, soft cap and window, HND
    w2 = W.custom([700, 5, 2500, 33, 1800], 32, 4, 64, 32, layout="HND", q_dtype="f16",
                  seed=22, logits_soft_cap=20.0, window_left=900)
    q2, p2 = W.make_q(w2), W.make_pool(w2)

    got1 = _noalloc(w1, q1, p1)
    assert noalloc_check_status() == 0
    got2 = _noalloc(w2, q2, p2)
    assert noalloc_check_status() == 0
    _compare(w1, got1, run_oracle(w1, q1, p1))
    _compare(w2, got2, run_oracle(w2, q2, p2))
    _compare(w1, got1, run_gpu(w1, q1, p1))
    _compare(w2, got2, run_gpu(w2, q2, p2))


def test_noalloc_e4m3_head_dim_256_cap_window():
    from paged_kv_decode_23_gb300 import noalloc_check_status
    w = W.custom([1, 300, 5000, 64, 2049, 0, 8000], 16, 2, 256, 32, layout="NHD",
                 q_dtype="bf16", kv_dtype="e4m3", seed=23, logits_soft_cap=30.0,
                 window_left=4096, kv_store_scale=0.5, k_scale=0.5, v_scale=0.5)
    q, p = W.make_q(w), W.make_pool(w)
    got = _noalloc(w, q, p)
    assert noalloc_check_status() == 0
    _compare(w, got, run_oracle(w, q, p))
    _compare(w, got, run_gpu(w, q, p))


def test_noalloc_rejects_a_work_list_beyond_the_scratch():
    """One chunk per request (disable_split_kv) for more requests than the built-in work list
    holds: PKD_ERR_WORKSPACE_TOO_SMALL, naming the limit, and nothing launched."""
    from paged_kv_decode_23_gb300 import PkdError
    n = 24577  # PKD_NOALLOC_MAX_ITEMS + 1
    w = W.custom([3] * n, 8, 1, 64, 8, layout="NHD", q_dtype="f16", seed=24)
    q, p = W.make_q(w), W.make_pool(w)
    with pytest.raises(PkdError) as e:
        _noalloc(w, q, p, disable_split_kv=1)
    assert e.value.code == -3
    assert "PKD_NOALLOC_MAX_ITEMS" in str(e.value)


def test_noalloc_mix_configuration_matches_the_handle_path_bit_for_bit():
    """The full-size e4m3 head_dim-256 batch (128 requests, window 4096, soft cap 30): the
    planner cuts its long rows once and merges 176 split units inside the launch.  Both entry
    points share the planner and the kernels, so their outputs agree bit for bit; both match
    the fp64 oracle."""
    w = W.workload("mix")
    q, p = W.make_q(w), W.make_pool(w)
    got = _noalloc(w, q, p)
    from paged_kv_decode_23_gb300 import noalloc_check_status
    assert noalloc_check_status() == 0
    ref = run_gpu(w, q, p)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    _compare(w, got, run_oracle(w, q, p))
