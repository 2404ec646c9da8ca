"""CUDA-graph mode (the pages' use_cuda_graph=True wrapper and CUDAGraphBatchDecode wrapper):
run() captured once in a CUDA graph must replay correctly after later plans of the same batch
size -- different lengths, different splits, zero-length padding -- checked against the oracle
through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


def _table(lens, page_size, pool_pages, rng):
    """A page table over an existing pool: each request's pages drawn without replacement."""
    lens = np.asarray(lens, dtype=np.int64)
    pages = np.where(lens > 0, (lens + page_size - 1) // page_size, 0)
    lpl = np.where(lens > 0, lens - (pages - 1) * page_size, 0).astype(np.int32)
    indptr = np.zeros(len(lens) + 1, dtype=np.int32)
    np.cumsum(pages, out=indptr[1:])
    indices = rng.permutation(pool_pages)[:indptr[-1]].astype(np.int32)
    return indptr, indices, lpl


def _workload(base, lens, indptr, indices, lpl):
    return W.Workload("graph", len(lens), base.num_qo_heads, base.num_kv_heads, base.head_dim,
                      base.page_size, base.layout, base.q_dtype, base.kv_dtype, base.o_dtype,
                      np.asarray(lens, dtype=np.int64), indptr, indices, lpl, base.num_pages,
                      sm_scale=base.sm_scale, logits_soft_cap=base.logits_soft_cap,
                      window_left=base.window_left, kv_store_scale=base.kv_store_scale,
                      k_scale=base.k_scale, v_scale=base.v_scale)


@pytest.mark.parametrize("kv,tc", [("bf16", True), ("bf16", False), ("e4m3", True), ("e4m3", False)])
def test_captured_run_replays_across_plans(kv, tc):
    from paged_kv_decode_23_gb300 import CUDAGraphBatchDecodePagedKV
    dev = torch.device("cuda")
    ps, batch = 16, 6
    # the pool every plan draws its pages from
    base = W.custom([4000] * batch, 16, 2, 128, ps, layout="NHD", q_dtype="bf16", kv_dtype=kv,
                    seed=21, pool_factor=1.0, logits_soft_cap=30.0 if kv == "e4m3" else 0.0)
    if kv == "e4m3":
        base.kv_store_scale, base.k_scale, base.v_scale = 0.5, 0.5, 0.5
    pool = W.make_pool(base, device=dev)
    max_pages = base.num_pages
    rng = np.random.default_rng(5)
    indptr_buf = torch.zeros(batch + 1, dtype=torch.int32, device=dev)
    indices_buf = torch.zeros(max_pages, dtype=torch.int32, device=dev)
    lpl_buf = torch.zeros(batch, dtype=torch.int32, device=dev)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    iws = torch.zeros(4 << 20, dtype=torch.uint8, device=dev)
    dec = CUDAGraphBatchDecodePagedKV(ws, indptr_buf, indices_buf, lpl_buf, "NHD",
                                      use_tensor_cores=tc, int_workspace_buffer=iws)
    q_static = torch.zeros(batch, 16, 128, dtype=torch.bfloat16, device=dev)
    o_static = torch.zeros_like(q_static)
    lse_static = torch.zeros(batch, 16, dtype=torch.float32, device=dev)

    # length mixes of the same batch size: long (many split chunks), short, zero-length padding
    plans = [[3900, 17, 250, 1, 3000, 640],
             [100, 2500, 0, 0, 33, 3999],       # two padded (empty) requests
             [1, 1, 1, 1, 1, 1],
             [3999, 3998, 3997, 3996, 3995, 3994]]
    graph = None
    for k, lens in enumerate(plans):
        indptr, indices, lpl = _table(lens, ps, max_pages, rng)
        w = _workload(base, lens, indptr, indices, lpl)
        idx_dev = torch.from_numpy(indices if len(indices) else np.zeros(1, np.int32)).to(dev)
        dec.plan(torch.from_numpy(indptr), idx_dev, torch.from_numpy(lpl), 16, 2, 128, ps,
                 q_data_type=torch.bfloat16, kv_data_type=W.TORCH_DTYPES[kv],
                 logits_soft_cap=base.logits_soft_cap or None)
        q = W.make_q(w, layer=k)
        q_static.copy_(q.to(dev))
        if graph is None:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # warm-up outside the capture
                dec.run(q_static, pool, k_scale=base.k_scale, v_scale=base.v_scale,
                        out=o_static, lse=lse_static)
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                dec.run(q_static, pool, k_scale=base.k_scale, v_scale=base.v_scale,
                        out=o_static, lse=lse_static)
        o_static.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert dec.check_status() == 0
        # the page table landed in the caller's buffers
        assert torch.equal(indptr_buf.cpu(), torch.from_numpy(indptr))
        assert torch.equal(lpl_buf.cpu(), torch.from_numpy(lpl))
        if indptr[-1]:
            assert torch.equal(indices_buf[:indptr[-1]].cpu(), torch.from_numpy(indices))
        got = (o_static.double().cpu().numpy(), lse_static.double().cpu().numpy())
        assert_close(w, got, run_oracle(w, q, pool.cpu()), f"plan {k} kv={kv} tc={tc}")


def test_graph_mode_fixes_the_batch_size():
    from paged_kv_decode_23_gb300 import BatchDecodePagedKV, PkdError
    dev = torch.device("cuda")
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device=dev)
    bufs = dict(paged_kv_indptr_buffer=torch.zeros(9, dtype=torch.int32, device=dev),
                paged_kv_indices_buffer=torch.zeros(64, dtype=torch.int32, device=dev),
                paged_kv_last_page_len_buffer=torch.zeros(8, dtype=torch.int32, device=dev))
    dec = BatchDecodePagedKV(ws, "NHD", use_cuda_graph=True, **bufs)
    idx = torch.arange(64, dtype=torch.int32, device=dev)
    dec.plan(torch.tensor([0, 2, 5], dtype=torch.int32), idx, torch.tensor([3, 16], dtype=torch.int32),
             8, 2, 128, 16)
    with pytest.raises(PkdError):  # a different batch size
        dec.plan(torch.tensor([0, 2, 5, 6], dtype=torch.int32), idx,
                 torch.tensor([3, 16, 1], dtype=torch.int32), 8, 2, 128, 16)
    with pytest.raises(PkdError):  # more pages than the indices buffer holds
        dec.plan(torch.tensor([0, 2, 65], dtype=torch.int32), torch.arange(70, dtype=torch.int32, device=dev),
                 torch.tensor([3, 16], dtype=torch.int32), 8, 2, 128, 16)
    with pytest.raises(ValueError):  # graph mode without its buffers
        BatchDecodePagedKV(ws, "NHD", use_cuda_graph=True)


def test_captured_run_replays_head_cut_plans():
    """A batch whose whole rows fill most of one wave of CTA slots (128 requests x 2 kv heads,
    half of them long): the planner cuts the long rows once (a second, partial wave of
    remainders, merged in the launch).  One captured run replays correctly across three such
    plans of the same batch size and an evenly split one."""
    from paged_kv_decode_23_gb300 import CUDAGraphBatchDecodePagedKV
    dev = torch.device("cuda")
    ps, batch = 16, 128
    base = W.custom([4000] * batch, 16, 2, 128, ps, layout="NHD", q_dtype="bf16",
                    kv_dtype="bf16", seed=23, pool_factor=1.0)
    pool = W.make_pool(base, device=dev)
    pool_cpu = pool.cpu()
    rng = np.random.default_rng(9)
    indptr_buf = torch.zeros(batch + 1, dtype=torch.int32, device=dev)
    indices_buf = torch.zeros(base.num_pages, dtype=torch.int32, device=dev)
    lpl_buf = torch.zeros(batch, dtype=torch.int32, device=dev)
    ws = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
    iws = torch.zeros(8 << 20, dtype=torch.uint8, device=dev)
    dec = CUDAGraphBatchDecodePagedKV(ws, indptr_buf, indices_buf, lpl_buf, "NHD",
                                      int_workspace_buffer=iws)
    q_static = torch.zeros(batch, 16, 128, dtype=torch.bfloat16, device=dev)
    o_static = torch.zeros_like(q_static)
    lse_static = torch.zeros(batch, 16, dtype=torch.float32, device=dev)
    plans = []
    for _ in range(3):
        lens = rng.integers(1, 2500, size=batch)
        lens[rng.permutation(batch)[:batch // 2]] = rng.integers(3600, 4001, size=batch // 2)
        plans.append(lens.tolist())
    plans.append([1500] * batch)
    graph = None
    for k, lens in enumerate(plans):
        indptr, indices, lpl = _table(lens, ps, base.num_pages, rng)
        w = _workload(base, lens, indptr, indices, lpl)
        dec.plan(torch.from_numpy(indptr), torch.from_numpy(indices).to(dev),
                 torch.from_numpy(lpl), 16, 2, 128, ps, q_data_type=torch.bfloat16)
        info = dec.plan_info()
        if k < 3:  # the head cut: more tasks than the 256 whole-row units, split rows merged
            assert info["tasks"] > batch * 2 and info["merges"] > 0, info
        q = W.make_q(w, layer=k)
        q_static.copy_(q.to(dev))
        if graph is None:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                dec.run(q_static, pool, out=o_static, lse=lse_static)
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                dec.run(q_static, pool, out=o_static, lse=lse_static)
        o_static.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert dec.check_status() == 0
        got = (o_static.double().cpu().numpy(), lse_static.double().cpu().numpy())
        assert_close(w, got, run_oracle(w, q, pool_cpu), f"head-cut plan {k}")
