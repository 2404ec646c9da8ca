"""Shared test helpers: run the CUDA path and the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

ORACLE_CODE = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3}

# |gpu - ref| <= ATOL + RTOL * |ref| elementwise (fp16/bf16 KV, then e4m3 KV); lse absolute.
TOL = {"f16": (2e-3, 1e-2), "bf16": (2e-3, 1e-2), "e4m3": (3e-2, 3e-2)}
LSE_ATOL = 1e-3


def plan_kwargs(w: W.Workload, **over):
    kw = dict(q_data_type=W.TORCH_DTYPES[w.q_dtype], kv_data_type=W.TORCH_DTYPES[w.kv_dtype],
              o_data_type=W.TORCH_DTYPES[w.o_dtype], sm_scale=w.sm_scale,
              logits_soft_cap=w.logits_soft_cap or None, window_left=w.window_left,
              fixed_split_size=w.fixed_split_size or None, disable_split_kv=w.disable_split_kv)
    kw.update(over)
    return kw


def gpu_decoder(w: W.Workload, ws_bytes: int = 256 << 20, **plan_over):
    from paged_kv_decode_23_gb300 import BatchDecodePagedKV
    dev = torch.device("cuda")
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    dec = BatchDecodePagedKV(ws, w.layout, int_workspace_buffer=torch.zeros(
        32 << 20, dtype=torch.uint8, device=dev))
    indices = torch.from_numpy(w.indices).to(dev) if len(w.indices) else torch.zeros(
        1, dtype=torch.int32, device=dev)
    dec.plan(torch.from_numpy(w.indptr), indices, torch.from_numpy(w.last_page_len),
             w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, **plan_kwargs(w, **plan_over))
    dec._keep = (ws, indices)
    return dec


def run_gpu(w: W.Workload, q: torch.Tensor, pool, dec=None, q_scale: float = 1.0, **plan_over):
    """o (float64) and lse (float64) from the CUDA path; q / pool may live on either device.
    ``q_scale`` is run()'s; k_scale and v_scale come from the workload."""
    dec = dec or gpu_decoder(w, **plan_over)
    dev = torch.device("cuda")
    if isinstance(pool, (tuple, list)):
        kv = tuple(t.to(dev) for t in pool)
    else:
        kv = pool.to(dev)
    o, lse = dec.run(q.to(dev), kv, q_scale=q_scale, k_scale=w.k_scale, v_scale=w.v_scale,
                     return_lse=True)
    torch.cuda.synchronize()
    assert dec.check_status() == 0, "device status word reports a failure"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def run_oracle(w: W.Workload, q: torch.Tensor, pool: torch.Tensor, chunk_tokens: int = 0,
               q_len: int = 1, q_scale: float = 1.0, **pos):
    """``pos``: pos_encoding_mode / rope_scale / rope_theta, passed to the oracle."""
    return oracle.batch_decode_pool(
        w.indptr, w.indices, w.last_page_len, W.raw_bits(q.cpu()), ORACLE_CODE[w.q_dtype],
        W.raw_bits(pool.cpu()), ORACLE_CODE[w.kv_dtype], w.layout, sm_scale=w.sm_scale,
        logits_soft_cap=w.logits_soft_cap, window_left=w.window_left, q_scale=q_scale,
        k_scale=w.k_scale, v_scale=w.v_scale, chunk_tokens=chunk_tokens, q_len=q_len, **pos)


def assert_close(w: W.Workload, got, ref, what=""):
    o, lse = got
    ro, rl = ref
    atol, rtol = TOL[w.kv_dtype]
    assert o.shape == ro.shape and lse.shape == rl.shape
    bad = np.abs(o - ro) > atol + rtol * np.abs(ro)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} o elements out of tolerance, first at "
                             f"{tuple(idx)}: gpu {o[tuple(idx)]} ref {ro[tuple(idx)]}; "
                             f"max |d| {np.abs(o - ro).max():.3e}")
    neg = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), neg), f"{what}: -inf lse pattern differs"
    d = np.abs(lse[~neg] - rl[~neg])
    assert d.size == 0 or d.max() <= LSE_ATOL, f"{what}: lse max |d| {d.max():.3e}"


def sub_problem(w: W.Workload, reqs, q: torch.Tensor, pool: torch.Tensor):
    """The workload restricted to requests `reqs`, with only their pages copied to the host
    (pages keep their contents; ids are renumbered).  Used to check full-size runs, and
    single requests of a batch, against the oracle."""
    reqs = list(reqs)
    pages = [w.indices[w.indptr[i]:w.indptr[i + 1]] for i in reqs]
    flat = np.concatenate(pages) if pages else np.zeros(0, np.int32)
    uniq = np.unique(flat)
    indptr = np.zeros(len(reqs) + 1, dtype=np.int32)
    indptr[1:] = np.cumsum([len(pg) for pg in pages])
    indices = np.searchsorted(uniq, flat).astype(np.int32)  # ids renumbered into sub_pool
    idx_t = torch.from_numpy(uniq.astype(np.int64)).to(pool.device)
    sub_pool = pool.index_select(0, idx_t).cpu()
    sub = W.Workload(w.name + "-sub", len(reqs), w.num_qo_heads, w.num_kv_heads, w.head_dim,
                     w.page_size, w.layout, w.q_dtype, w.kv_dtype, w.o_dtype,
                     w.kv_lens[reqs], indptr, indices,
                     w.last_page_len[reqs], len(uniq), sm_scale=w.sm_scale,
                     logits_soft_cap=w.logits_soft_cap, window_left=w.window_left,
                     kv_store_scale=w.kv_store_scale, k_scale=w.k_scale, v_scale=w.v_scale)
    return sub, q[reqs].cpu(), sub_pool
