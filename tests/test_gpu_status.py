"""The device status word (failure detection without faulting the GPU).

Every pipeline wait of the decode kernel is bounded.  With the wait limit set to 0, each wait
that is not already complete gives up at once: the CTA sets PKD_STATUS_TIMEOUT, lets the copies
it has issued land, and exits without writing its outputs; later launches on the same status
word return at once until pkd_check_status clears it.  A page id outside the pool is read as
zeros and reported with PKD_STATUS_BAD_PAGE, without stopping later launches.
"""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import LSE_ATOL, TOL, assert_close, gpu_decoder, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

SENTINEL = 123.0
L2_FLUSH = torch.Size([2 * 129 * 1024 * 1024 // 4])


def _flush(dev):
    torch.empty(L2_FLUSH, dtype=torch.float32, device=dev).fill_(1.0)


def _run_into(dec, w, q, pool, dev):
    o = torch.full(q.shape, SENTINEL, dtype=W.TORCH_DTYPES[w.o_dtype], device=dev)
    lse = torch.full(q.shape[:2], SENTINEL, dtype=torch.float32, device=dev)
    dec.run(q, pool, k_scale=w.k_scale, v_scale=w.v_scale, out=o, lse=lse)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("tc", [True, False])
def test_wait_limit_zero_gives_up_reports_and_recovers(tc):
    from paged_kv_decode_23_gb300 import _lib as L
    dev = torch.device("cuda")
    lens = [3000, 17, 2000, 4000, 1000, 700, 0, 2500] * 4
    w = W.custom(lens, 16, 2, 128, 16, layout="NHD", q_dtype="bf16", seed=61)
    q, pool = W.make_q(w).to(dev), W.make_pool(w).to(dev)
    ref_o, ref_lse = run_oracle(w, q, pool)
    # split requests: merges inside the launch too
    dec = gpu_decoder(w, fixed_split_size=8, use_tensor_cores=tc)
    atol, rtol = TOL[w.kv_dtype]

    # 1. every wait that is not already complete gives up
    dec.set_wait_limit(0)
    _flush(dev)
    o, lse = _run_into(dec, w, q, pool, dev)
    written = ~np.all(o == SENTINEL, axis=2)          # per (row, qo head)
    assert not written.all(), "a timed-out launch wrote every output"
    # what was written is complete and right; what was not is untouched
    ok = np.abs(o - ref_o) <= atol + rtol * np.abs(ref_o)
    assert ok[written].all(), "a written output row is wrong"
    assert np.all(o[~written] == SENTINEL)
    fin = np.isfinite(ref_lse)
    lw = lse != SENTINEL
    assert np.all(np.abs(lse[lw & fin] - ref_lse[lw & fin]) <= LSE_ATOL)
    assert np.array_equal(lw, written), "o and lse written for different rows"

    # 2. with the word still set, a later launch (default limit) returns at once
    dec.set_wait_limit(2_000_000_000)
    o2, lse2 = _run_into(dec, w, q, pool, dev)
    assert np.all(o2 == SENTINEL) and np.all(lse2 == SENTINEL)

    # 3. the host reads and clears the word
    st = dec.check_status()
    assert st & L.STATUS_TIMEOUT, f"status {st}: the timeout was not reported"
    assert dec.check_status() == 0

    # 4. the next run of the same plan is complete and right (merge counters were reset)
    got = run_gpu(w, q, pool, dec=dec)
    assert_close(w, got, (ref_o, ref_lse), "after recovery")


def test_wait_limit_is_bounded():
    from paged_kv_decode_23_gb300 import PkdError
    w = W.custom([40], 8, 2, 128, 16, seed=62)
    dec = gpu_decoder(w)
    with pytest.raises(PkdError) as e:
        dec.set_wait_limit(2_000_000_001)
    assert e.value.code == -1


@pytest.mark.parametrize("tc", [True, False])
def test_page_id_outside_the_pool_reads_zeros_and_is_reported(tc):
    from paged_kv_decode_23_gb300 import _lib as L
    dev = torch.device("cuda")
    lens = [100, 300, 50, 700]
    w = W.custom(lens, 8, 2, 128, 16, layout="HND", q_dtype="f16", seed=63)
    q, pool = W.make_q(w), W.make_pool(w)
    bad = w.indices.copy()
    bad[w.indptr[1] + 3] = w.num_pages          # one past the last page
    bad[w.indptr[3] + 10] = -1                  # negative
    wb = W.custom(lens, 8, 2, 128, 16, layout="HND", q_dtype="f16", seed=63)
    wb.indices = bad
    # the oracle sees the same table over a pool with one extra all-zero page standing in for
    # both out-of-range ids
    zpool = torch.cat([pool, torch.zeros_like(pool[:1])])
    wz = W.custom(lens, 8, 2, 128, 16, layout="HND", q_dtype="f16", seed=63)
    wz.indices = np.where((bad < 0) | (bad >= w.num_pages), w.num_pages, bad).astype(np.int32)
    ref = run_oracle(wz, q, zpool)
    dec = gpu_decoder(wb, use_tensor_cores=tc)
    qd, pd = q.to(dev), pool.to(dev)
    for k in range(2):
        # the second run starts with the bit already set: it still runs (only a timeout stops
        # later launches)
        o, lse = dec.run(qd, pd, return_lse=True)
        torch.cuda.synchronize()
        got = (o.double().cpu().numpy(), lse.double().cpu().numpy())
        assert_close(wb, got, ref, f"bad page ids tc={tc} run {k}")
    st = dec.check_status()
    assert st == L.STATUS_BAD_PAGE, f"status {st}"
    assert dec.check_status() == 0
    # a clean table on the same handle reports nothing
    got = run_gpu(w, q, pool, use_tensor_cores=tc)
    assert_close(w, got, run_oracle(w, q, pool), "clean table")
