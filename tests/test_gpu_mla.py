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


def _run(w, qn, qp, ckv, kpe, base_e=True, ws_mb=256):
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention
    dev = torch.device("cuda")
    mla = BatchMLAPagedAttention(torch.zeros(ws_mb << 20, dtype=torch.uint8, device=dev))
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


@pytest.mark.parametrize("ps", [1, 16, 64])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_mla_lengths_pages_dtypes(ps, dt):
    lens = [1, 31, 32, 33, 0, 100, 777, 64]
    w = W.mla_custom(lens, 40, ps, dt, seed=ps, extra_pages=1)  # 40 heads: a partial slice
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    ref = _oracle(w, qn, qp, ckv, kpe)
    _close(_run(w, qn, qp, ckv, kpe), ref, f"mla ps={ps} {dt}")
    _close(_run(w, qn, qp, ckv, kpe, base_e=False), ref, f"mla ps={ps} {dt} base 2",
           lse_base_e=False)


@pytest.mark.parametrize("heads", [16, 32, 128])
def test_mla_split_requests(heads):
    """A small batch of long requests is split into chunks (one wave of CTAs) and merged
    inside the launch."""
    w = W.mla_custom([3000, 4500, 20], heads, 1, "bf16", seed=heads)
    qn, qp = W.make_mla_q(w)
    ckv, kpe = W.make_mla_cache(w)
    _close(_run(w, qn, qp, ckv, kpe), _oracle(w, qn, qp, ckv, kpe), f"mla split H={heads}")


def test_mla_full_example_sampled():
    """The pages' example at full size (batch 114, 128 heads, kv_len 999, page_size 1),
    sampled requests against the oracle."""
    w = W.mla_workload()
    dev = torch.device("cuda")
    qn, qp = W.make_mla_q(w, device=dev)
    ckv, kpe = W.make_mla_cache(w, device=dev)
    got = _run(w, qn, qp, ckv, kpe)
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
    with pytest.raises(NotImplementedError):  # two queries in a request
        mla.plan(torch.tensor([0, 2], dtype=torch.int32), *args[1:], 512, 64, 1, False, 0.1,
                 torch.bfloat16, torch.bfloat16)
