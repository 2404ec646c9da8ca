"""MLA paged decode (the pages' BatchMLAPagedAttentionWrapper, decode): the CUDA path through
the C ABI against the fp64 oracle, element by element.  Tolerances as for fp16 / bf16 decode:
|o - ref| <= 2e-3 + 1e-2 |ref|, lse within 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

CODE = {"bf16": oracle.BF16, "f16": oracle.F16}


BACKENDS = ["fa2", "tcgen05"]


def _run(w, qn, qp, ckv, kpe, base_e=True, ws_mb=256, backend="auto"):
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention
    dev = torch.device("cuda")
    mla = BatchMLAPagedAttention(torch.zeros(ws_mb << 20, dtype=torch.uint8, device=dev),
                                 backend=backend)
    idx = torch.from_numpy(w.kv_indices if len(w.kv_indices) else np.zeros(1, np.int32)).to(dev)
    mla.plan(torch.arange(w.batch + 1, dtype=torch.int32), torch.from_numpy(w.kv_indptr), idx,
             torch.from_numpy(w.kv_lens), w.num_heads, 512, 64, w.page_size, False, w.sm_scale,
             W.TORCH_DTYPES[w.dtype], W.TORCH_DTYPES[w.dtype])
    o, lse = mla.run(qn.to(dev), qp.to(dev), ckv.to(dev), kpe.to(dev), return_lse=True,
                     return_lse_base_on_e=base_e)
    torch.cuda.synchronize()
    assert mla.check_status() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def _oracle(w, qn, qp, ckv, kpe):
    return oracle.mla_decode(w.kv_indptr, w.kv_indices, w.kv_lens, W.raw_bits(qn.cpu()),
                             W.raw_bits(qp.cpu()), CODE[w.dtype], W.raw_bits(ckv.cpu()),
                             W.raw_bits(kpe.cpu()), CODE[w.dtype], w.page_size, w.sm_scale)


def _close(got, ref, what, lse_base_e=True):
    o, lse = got
    ro, rl = ref
    if not lse_base_e:
        rl = rl / np.log(2.0)
    bad = np.abs(o - ro) > 2e-3 + 1e-2 * np.abs(ro)
    assert not bad.any(), (f"{what}: {bad.sum()} o out of tolerance, max |d| "
                           f"{np.abs(o - ro).max():.3e}")
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl)), f"{what}: -inf pattern"
    fin = np.isfinite(rl)
    assert fin.sum() == 0 or np.abs(lse[fin] - rl[fin]).max() <= 1e-3, f"{what}: lse"


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("ps", [1, 16, 64])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_mla_lengths_pages_dtypes(ps, dt, backend):
    lens = [1, 31, 32, 33, 0, 100, 777, 64]
    # 40 heads: a partial head slice (fa2) or a head tile of 128 with 88 empty rows (tcgen05)
    w = W.mla_custom(lens, 40, ps, dt, seed=ps, extra_pages=1)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    ref = _oracle(w, qn, qp, ckv, kpe)
    _close(_run(w, qn, qp, ckv, kpe, backend=backend), ref, f"mla ps={ps} {dt} {backend}")
    _close(_run(w, qn, qp, ckv, kpe, base_e=False, backend=backend), ref,
           f"mla ps={ps} {dt} {backend} base 2", lse_base_e=False)


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("heads", [16, 32, 128, 192])
def test_mla_split_requests(heads, backend):
    """A small batch of long requests is split into chunks (one wave of CTAs) and merged
    inside the launch; 192 heads take two head tiles on the tcgen05 kernel."""
    w = W.mla_custom([3000, 4500, 20], heads, 1, "bf16", seed=heads)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    _close(_run(w, qn, qp, ckv, kpe, backend=backend), _oracle(w, qn, qp, ckv, kpe),
           f"mla split H={heads} {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
def test_mla_many_chunks_one_request(backend):
    """One request long enough that the one-wave plan cuts it into one chunk per CTA slot
    (76 chunks on the tcgen05 kernel's CTA pairs): the fused merge folds them all."""
    w = W.mla_custom([40000, 300], 16, 1, "bf16", seed=21)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    _close(_run(w, qn, qp, ckv, kpe, backend=backend), _oracle(w, qn, qp, ckv, kpe),
           f"mla many chunks {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
def test_mla_split_run_to_run_determinism(backend):
    """Split requests: the merge folds the chunks in slot order whichever CTA finishes last,
    so repeated launches agree bit for bit."""
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention
    w = W.mla_custom([3000, 4500, 20, 999], 128, 1, "bf16", seed=22)
    dev = torch.device("cuda")
    qn, qp = W.make_mla_q(w, device=dev)
    ckv, kpe = W.make_mla_cache(w, device=dev)
    mla = BatchMLAPagedAttention(torch.zeros(256 << 20, dtype=torch.uint8, device=dev),
                                 backend=backend)
    mla.plan(torch.arange(w.batch + 1, dtype=torch.int32), torch.from_numpy(w.kv_indptr),
             torch.from_numpy(w.kv_indices).to(dev), torch.from_numpy(w.kv_lens), w.num_heads,
             512, 64, w.page_size, False, w.sm_scale, torch.bfloat16, torch.bfloat16)
    outs = [mla.run(qn, qp, ckv, kpe, return_lse=True) for _ in range(6)]
    torch.cuda.synchronize()
    assert mla.check_status() == 0
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("backend", BACKENDS)
def test_mla_logits_far_apart(backend):
    """Latent rows shifted by a ramp over the page pool spread the logits over tens of units,
    so the running maximum of a head jumps by more than 8 (log2) several times along a
    request and the lazily kept output must be rescaled; the softmax is nearly one-hot."""
    w = W.mla_custom([700, 64, 2000], 128, 1, "bf16", seed=5)
    w.sm_scale = 0.5
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    ramp = torch.linspace(0.0, 3.0, ckv.shape[0]).to(ckv.dtype).view(-1, 1, 1)
    ckv = (ckv.float() + ramp.float() * qn.float().mean(dim=(0, 1)).sign()).to(ckv.dtype)
    _close(_run(w, qn, qp, ckv, kpe, backend=backend), _oracle(w, qn, qp, ckv, kpe),
           f"mla far-apart logits {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
def test_mla_full_example_sampled(backend):
    """The pages' example at full size (batch 114, 128 heads, kv_len 999, page_size 1),
    sampled requests against the oracle."""
    w = W.mla_workload()
    dev = torch.device("cuda")
    qn, qp = W.make_mla_q(w, device=dev)
    ckv, kpe = W.make_mla_cache(w, device=dev)
    got = _run(w, qn, qp, ckv, kpe, backend=backend)
    for i in (0, 57, 113):
        sub = W.mla_custom([int(w.kv_lens[i])], w.num_heads, 1, "bf16")
        pages = w.kv_indices[w.kv_indptr[i]:w.kv_indptr[i + 1]]
        sub.kv_indices = np.arange(len(pages), dtype=np.int32)
        sub.kv_indptr = np.array([0, len(pages)], dtype=np.int32)
        sel = torch.from_numpy(pages.astype(np.int64)).to(dev)
        ref = _oracle(sub, qn[i:i + 1], qp[i:i + 1], ckv.index_select(0, sel),
                      kpe.index_select(0, sel))
        _close((got[0][i:i + 1], got[1][i:i + 1]), ref, f"mla example request {i}")


def test_mla_rejects_other_shapes():
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention, PkdError
    dev = torch.device("cuda")
    mla = BatchMLAPagedAttention(torch.zeros(1 << 20, dtype=torch.uint8, device=dev))
    idx = torch.zeros(4, dtype=torch.int32, device=dev)
    args = (torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0, 4], dtype=torch.int32), idx,
            torch.tensor([4], dtype=torch.int32), 16)
    with pytest.raises(PkdError):  # head_dim_ckv other than 512
        mla.plan(*args, 256, 64, 1, False, 0.1, torch.bfloat16, torch.bfloat16)
    with pytest.raises(PkdError):  # kv_len beyond the pages
        mla.plan(torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0, 4], dtype=torch.int32),
                 idx, torch.tensor([5], dtype=torch.int32), 16, 512, 64, 1, False, 0.1,
                 torch.bfloat16, torch.bfloat16)
    with pytest.raises(ValueError):
        BatchMLAPagedAttention(torch.zeros(1 << 20, dtype=torch.uint8, device=dev), backend="fa3")
    with pytest.raises(NotImplementedError):  # two queries in a request
        mla.plan(torch.tensor([0, 2], dtype=torch.int32), *args[1:], 512, 64, 1, False, 0.1,
                 torch.bfloat16, torch.bfloat16)


@pytest.mark.parametrize("backend", BACKENDS)
def test_mla_page_ids_outside_the_caches_read_as_zero_rows(backend):
    """A page id outside [0, num_pages) reads as a zero row (logit 0, value 0), as a read past
    the end of the caches does; checked against the oracle on caches with an appended zero page
    that those ids point to."""
    w = W.mla_custom([40, 300, 77], 128, 4, "bf16", seed=11)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    npg = ckv.shape[0]
    bad = w.kv_indices.copy()
    bad[[0, 5, 13, 40, 41, len(bad) - 1]] = [npg, -1, npg + 7, -5, npg, 2 ** 30]
    w_bad = W.mla_custom([40, 300, 77], 128, 4, "bf16", seed=11)
    w_bad.kv_indices = bad
    got = _run(w_bad, qn, qp, ckv, kpe, backend=backend)
    ref_idx = np.where((bad < 0) | (bad >= npg), npg, bad).astype(np.int32)
    w_ref = W.mla_custom([40, 300, 77], 128, 4, "bf16", seed=11)
    w_ref.kv_indices = ref_idx
    zc = torch.cat([ckv, torch.zeros_like(ckv[:1])])
    zk = torch.cat([kpe, torch.zeros_like(kpe[:1])])
    _close(got, _oracle(w_ref, qn, qp, zc, zk), f"mla bad page ids {backend}")


@pytest.mark.parametrize("backend,heads", [("fa2", 32), ("tcgen05", 128)])
def test_mla_cuda_graph_replays_across_plans(backend, heads):
    """The wrapper's use_cuda_graph=True: run() captured once replays correctly after later
    plans of the same batch size (different lengths, splits and zero-length padding), each
    checked against the oracle."""
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention, mla_graph_workspace_bytes
    dev = torch.device("cuda")
    ps, batch = 16, 4
    base = W.mla_custom([3000] * batch, heads, ps, "bf16", seed=31, pool_factor=1.0)
    ckv, kpe = W.make_mla_cache(base)
    ckv_d, kpe_d = ckv.to(dev), kpe.to(dev)
    max_pages = base.num_pages
    fb, ib = mla_graph_workspace_bytes(batch + 152, heads, backend)
    ws = torch.zeros(fb, dtype=torch.uint8, device=dev)
    iws = torch.zeros(ib, dtype=torch.uint8, device=dev)
    bufs = dict(qo_indptr=torch.zeros(batch + 1, dtype=torch.int32, device=dev),
                kv_indptr=torch.zeros(batch + 1, dtype=torch.int32, device=dev),
                kv_indices=torch.zeros(max_pages, dtype=torch.int32, device=dev),
                kv_len_arr=torch.zeros(batch, dtype=torch.int32, device=dev))
    mla = BatchMLAPagedAttention(ws, use_cuda_graph=True, backend=backend,
                                 int_workspace_buffer=iws, max_items=batch + 152, **bufs)
    qn_s = torch.zeros(batch, heads, 512, dtype=torch.bfloat16, device=dev)
    qp_s = torch.zeros(batch, heads, 64, dtype=torch.bfloat16, device=dev)
    o_s = torch.zeros_like(qn_s)
    lse_s = torch.zeros(batch, heads, dtype=torch.float32, device=dev)
    rng = np.random.default_rng(6)
    plans = [[3000, 17, 250, 999], [100, 2900, 0, 0], [1, 1, 1, 1], [2990, 2980, 2970, 2960]]
    graph = None
    for k, lens in enumerate(plans):
        lens = np.asarray(lens, dtype=np.int64)
        pages = np.where(lens > 0, (lens + ps - 1) // ps, 0)
        indptr = np.zeros(batch + 1, dtype=np.int32)
        np.cumsum(pages, out=indptr[1:])
        indices = rng.permutation(max_pages)[:indptr[-1]].astype(np.int32)
        w = W.MlaWorkload("graph", batch, heads, ps, "bf16", lens.astype(np.int32), indptr,
                          indices, max_pages, sm_scale=base.sm_scale, seed=31 + k)
        idx_dev = torch.from_numpy(indices if len(indices) else np.zeros(1, np.int32)).to(dev)
        mla.plan(torch.arange(batch + 1, dtype=torch.int32), torch.from_numpy(indptr), idx_dev,
                 torch.from_numpy(w.kv_lens), heads, 512, 64, ps, False, w.sm_scale,
                 torch.bfloat16, torch.bfloat16)
        qn, qp = W.make_mla_q(w, layer=k)
        qn_s.copy_(qn.to(dev))
        qp_s.copy_(qp.to(dev))
        if graph is None:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # warm-up outside the capture
                mla.run(qn_s, qp_s, ckv_d, kpe_d, out=o_s, lse=lse_s, return_lse=True,
                        return_lse_base_on_e=True)
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                mla.run(qn_s, qp_s, ckv_d, kpe_d, out=o_s, lse=lse_s, return_lse=True,
                        return_lse_base_on_e=True)
        o_s.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert mla.check_status() == 0
        assert torch.equal(bufs["kv_len_arr"].cpu(), torch.from_numpy(w.kv_lens))
        _close((o_s.double().cpu().numpy(), lse_s.double().cpu().numpy()),
               _oracle(w, qn, qp, ckv, kpe), f"mla graph plan {k} {backend}")


def test_mla_cuda_graph_rejects_changed_shapes():
    """In CUDA-graph mode the first plan fixes the batch size and what a captured run holds."""
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention, PkdError
    dev = torch.device("cuda")
    bufs = dict(kv_indptr=torch.zeros(5, dtype=torch.int32, device=dev),
                kv_indices=torch.zeros(64, dtype=torch.int32, device=dev),
                kv_len_arr=torch.zeros(4, dtype=torch.int32, device=dev))
    mla = BatchMLAPagedAttention(torch.zeros(64 << 20, dtype=torch.uint8, device=dev),
                                 use_cuda_graph=True, **bufs)
    idx = torch.arange(8, dtype=torch.int32, device=dev)

    def plan(batch, heads=32, ps=1, scale=0.1):
        lens = np.full(batch, 2, dtype=np.int32)
        ip = np.arange(0, 2 * batch + 1, 2, dtype=np.int32)
        mla.plan(torch.arange(batch + 1, dtype=torch.int32), torch.from_numpy(ip), idx,
                 torch.from_numpy(lens), heads, 512, 64, ps, False, scale, torch.bfloat16,
                 torch.bfloat16)

    plan(4)
    with pytest.raises(PkdError):
        plan(3)          # batch changed
    with pytest.raises(PkdError):
        plan(4, heads=16)
    with pytest.raises(PkdError):
        plan(4, ps=2)
    with pytest.raises(PkdError):
        plan(4, scale=0.2)
    with pytest.raises(ValueError):
        BatchMLAPagedAttention(torch.zeros(1 << 20, dtype=torch.uint8, device=dev),
                               use_cuda_graph=True)
    plan(4)  # the same shapes plan again


def test_run_accepts_the_page_keywords_and_refuses_unbuilt_ones():
    """run() takes the page's keyword set: profiler_buffer, kv_len and page_table left as None
    run normally; given, they name parts that are not built (the profiler, the cutlass
    backend's run-time page table) and are refused."""
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention
    dev = torch.device("cuda")
    w = W.mla_custom([5, 40], 16, 16, "bf16", seed=4)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    mla = BatchMLAPagedAttention(torch.zeros(64 << 20, dtype=torch.uint8, device=dev))
    mla.plan(torch.arange(w.batch + 1, dtype=torch.int32), torch.from_numpy(w.kv_indptr),
             torch.from_numpy(w.kv_indices).to(dev), torch.from_numpy(w.kv_lens), w.num_heads,
             512, 64, w.page_size, False, w.sm_scale, torch.bfloat16, torch.bfloat16)
    args = (qn.to(dev), qp.to(dev), ckv.to(dev), kpe.to(dev))
    o = mla.run(*args, profiler_buffer=None, kv_len=None, page_table=None)
    torch.cuda.synchronize()
    ref, _ = _oracle(w, qn, qp, ckv, kpe)
    got = o.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))
    with pytest.raises(NotImplementedError):
        mla.run(*args, profiler_buffer=torch.zeros(16, device=dev))
    with pytest.raises(NotImplementedError):
        mla.run(*args, kv_len=torch.from_numpy(w.kv_lens).to(dev))
