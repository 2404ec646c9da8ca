"""Host-side tests (no GPU): the C ABI loads and exports what include/pkd.h declares, and the
planner's work list is a correct partition of every request's attended keys."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkd():
    import __graft_entry__ as g
    from paged_kv_decode_23_gb300 import build
    build.build()
    import paged_kv_decode_23_gb300 as p
    return p


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "pkd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkd_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(pkd):
    from paged_kv_decode_23_gb300 import _lib as L
    lib = L.lib()
    declared = _declared_symbols()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in pkd.h but not exported"
        assert name in L.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_create_without_device_fails_cleanly(pkd):
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    from paged_kv_decode_23_gb300 import _lib as L
    h = ctypes.c_void_p()
    rc = L.lib().pkd_create(ctypes.byref(h), 0, 0, 0, 0, L.LAYOUT_NHD)
    assert rc == -4 and not h.value
    assert L.lib().pkd_last_error().decode()


def _units(plan):
    """Tasks grouped by (row, kv head, slice), each group sorted by its first attended token."""
    by_unit = {}
    for t in plan["tasks"]:
        by_unit.setdefault((int(t[0]), int(t[8]), int(t[9])), []).append(t)
    return {k: sorted(v, key=lambda x: int(x[3])) for k, v in by_unit.items()}


def _check_partition(w, plan, C, q_len=1):
    """Every (row, kv head, slice) unit's attended tokens are covered exactly once by its
    tasks; chunks start at page boundaries (at multiples of C from token 0 with a fixed split);
    a unit of one task writes its final output, a split unit has consecutive partial slots and
    one merge entry; the tasks are grouped by CTA."""
    tasks, merges = plan["tasks"], plan["merges"]
    G = w.num_qo_heads // w.num_kv_heads
    hpc = 8 if plan["kernel"] == 1 else max(2, min(8, 1 << (G - 1).bit_length()))
    gsl = (G + hpc - 1) // hpc
    units = _units(plan)
    rows = w.batch * q_len
    assert sorted(units) == [(r, h, g) for r in range(rows) for h in range(w.num_kv_heads)
                             for g in range(gsl)]
    slots = []
    for (row, kvh, gs), ts in units.items():
        i, j = divmod(row, q_len)
        n = max(0, int(w.kv_lens[i]) - (q_len - 1 - j))
        lo = 0 if w.window_left < 0 else max(0, n - 1 - w.window_left)
        assert all(int(t[1]) == int(w.indptr[i]) for t in ts)
        if n == 0:
            assert len(ts) == 1 and ts[0][3] == ts[0][4] == 0 and ts[0][5] == -1
            continue
        assert all(int(t[7]) == n - 1 for t in ts)
        assert int(ts[0][3]) == lo and int(ts[-1][4]) == n
        for a, b in zip(ts, ts[1:]):
            assert int(a[4]) == int(b[3])
        for t in ts:
            c0, b0, e0 = int(t[2]), int(t[3]), int(t[4])
            assert c0 % w.page_size == 0 and c0 <= b0 < e0
            if C:
                assert c0 % C == 0 and e0 - c0 <= C
        if len(ts) == 1:
            assert ts[0][5] == -1 and ts[0][6] == -1
        else:
            m = merges[int(ts[0][6])]
            assert all(int(t[6]) == int(ts[0][6]) for t in ts)
            assert int(m[0]) == row and int(m[2]) == len(ts) and int(m[3]) == kvh * gsl + gs
            assert [int(t[5]) for t in ts] == list(range(int(m[1]), int(m[1]) + len(ts)))
            slots += [int(t[5]) for t in ts]
    assert sorted(slots) == list(range(plan["num_slots"]))
    # one CTA per task, launched longest first
    assert plan["num_ctas"] == len(tasks) and np.array_equal(tasks[:, 10], np.arange(len(tasks)))
    lens = tasks[:, 4] - tasks[:, 3]
    assert np.all(np.diff(lens) <= 0)


@pytest.mark.parametrize("name", ["worked", "uniform", "lognormal", "long", "mix"])
def test_plan_partitions_every_workload(pkd, name):
    w = W.workload(name)
    plan = pkd.plan_host(w.indptr, w.last_page_len, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                         w.page_size, window_left=w.window_left,
                         fixed_split_size=w.fixed_split_size,
                         kv_dtype={"f16": 0, "bf16": 1, "e4m3": 2}[w.kv_dtype])
    C = w.fixed_split_size * w.page_size
    _check_partition(w, plan, C)
    if name == "long":  # 4 requests x 8 chunks of 256 pages, per kv head
        assert len(plan["tasks"]) == 4 * 8 * 8 and len(plan["merges"]) == 4 * 8
    elif w.batch * w.num_kv_heads <= 304:
        # the unsplit rows fit one wave of CTA slots: either a split that keeps one wave, or
        # every long row cut once (a partial second wave of remainders)
        assert len(plan["tasks"]) <= 304 or all(len(ts) <= 2 for ts in _units(plan).values())


def test_one_wave_batch_of_similar_rows_cuts_its_long_rows_once(pkd):
    """mix: 128 rows x 2 kv heads fit one wave of 304 CTA slots unsplit, but half the rows
    attend the whole 4097-token window.  The list-scheduling score prefers cutting every row
    longer than some C once, after its first C tokens (page-aligned), so the remainders run in
    the slots the short rows free; rows of at most C stay whole."""
    w = W.workload("mix")
    ps = w.page_size
    plan = pkd.plan_host(w.indptr, w.last_page_len, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                         w.page_size, window_left=w.window_left, kv_dtype=2)
    _check_partition(w, plan, 0)
    units = _units(plan)
    cut = [ts for ts in units.values() if len(ts) == 2]
    assert cut and all(len(ts) <= 2 for ts in units.values())
    assert len(plan["tasks"]) > 304
    first = [int(ts[0][4]) - int(ts[0][3]) for ts in cut]
    C = max(first)
    assert all(C - ps < f <= C for f in first)
    assert all(int(ts[0][4]) % ps == 0 for ts in cut)
    assert all(int(ts[1][4]) - int(ts[1][3]) <= C for ts in cut)
    whole = [int(ts[0][4]) - int(ts[0][3]) for ts in units.values() if len(ts) == 1]
    assert max(whole) <= C and 2 * C >= max(int(ts[1][4]) - int(ts[0][3]) for ts in cut)


@pytest.mark.parametrize("fixed", [0, 1, 2, 7, 64])
@pytest.mark.parametrize("window", [-1, 0, 10, 1000])
def test_plan_modes(pkd, fixed, window):
    lens = [0, 1, 7, 8, 9, 100, 1000, 5000]
    w = W.custom(lens, 8, 2, 128, 8, window_left=window)
    plan = pkd.plan_host(w.indptr, w.last_page_len, 8, 2, 128, 8, window_left=window,
                         fixed_split_size=fixed)
    _check_partition(w, plan, fixed * 8)
    nosplit = pkd.plan_host(w.indptr, w.last_page_len, 8, 2, 128, 8, window_left=window,
                            fixed_split_size=fixed, disable_split_kv=True)
    _check_partition(w, nosplit, 0)
    assert len(nosplit["tasks"]) == len(lens) * 2 and len(nosplit["merges"]) == 0


def test_fixed_split_is_batch_invariant(pkd):
    lens = [5000, 33, 1200]
    w = W.custom(lens, 8, 2, 128, 16)
    full = pkd.plan_host(w.indptr, w.last_page_len, 8, 2, 128, 16, fixed_split_size=16)
    for i in range(3):
        wi = W.custom([lens[i]], 8, 2, 128, 16)
        alone = pkd.plan_host(wi.indptr, wi.last_page_len, 8, 2, 128, 16, fixed_split_size=16)
        mine = sorted((int(x[8]), int(x[2]), int(x[3]), int(x[4])) for x in full["tasks"]
                      if x[0] == i)
        theirs = sorted((int(x[8]), int(x[2]), int(x[3]), int(x[4])) for x in alone["tasks"])
        assert mine == theirs


def test_one_wave_plan_cuts_a_long_row_into_equal_chunks(pkd):
    """Rows that fit one wave of CTA slots unsplit: the longest is cut into equal page-aligned
    chunks, as many as keep every CTA in that one wave."""
    lens = [200000, 50, 3000, 7]
    w = W.custom(lens, 8, 1, 128, 16)
    plan = pkd.plan_host(w.indptr, w.last_page_len, 8, 1, 128, 16)
    _check_partition(w, plan, 0)
    assert 250 <= len(plan["tasks"]) <= 304
    ts = plan["tasks"][plan["tasks"][:, 0] == 0]
    lens0 = ts[:, 4] - ts[:, 3]
    assert lens0.max() - lens0.min() <= 16


def test_kernel_choice_and_tiles(pkd):
    w = W.workload("worked")
    auto = pkd.plan_host(w.indptr, w.last_page_len, 64, 8, 128, 16)
    cc = pkd.plan_host(w.indptr, w.last_page_len, 64, 8, 128, 16, use_tensor_cores=0)
    assert auto["kernel"] == 1 and cc["kernel"] == 0
    assert auto["tile_tokens"] == 64
    assert pkd.plan_host(w.indptr, w.last_page_len, 64, 8, 256, 16)["tile_tokens"] == 32
    assert pkd.plan_host(w.indptr, w.last_page_len, 64, 8, 256, 16, kv_dtype=2)["tile_tokens"] == 64


@pytest.mark.parametrize("bad", [
    dict(num_qo_heads=12, num_kv_heads=8),           # not a multiple
    dict(head_dim=96),                               # unsupported head_dim
    dict(page_size=24),                              # not a power of two
    dict(page_size=4),                               # below 8
    dict(lpl_fix=0),                                 # last_page_len 0 on a request with pages
    dict(lpl_fix=17),                                # last_page_len > page_size
    dict(indptr_fix=True),                           # decreasing indptr
    dict(head_dim=64, kv_dtype=2),                   # e4m3 needs head_dim >= 128
])
def test_plan_rejects_bad_input(pkd, bad):
    from paged_kv_decode_23_gb300 import PkdError
    ip = np.array([0, 3, 5, 9], dtype=np.int32)
    lpl = np.array([4, 16, 1], dtype=np.int32)
    if "lpl_fix" in bad:
        lpl[1] = bad.pop("lpl_fix")
    if bad.pop("indptr_fix", False):
        ip[2] = 2
    args = dict(num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16)
    args.update(bad)
    with pytest.raises(PkdError) as e:
        pkd.plan_host(ip, lpl, **args)
    assert e.value.code in (-1, -5)


def test_check_page_table_names_the_first_bad_id(pkd):
    """The optional host validation of a page table (pkd_check_page_table): ids must lie in
    [0, num_pages); the message names the request and the position of the first bad id."""
    from paged_kv_decode_23_gb300 import PkdError
    ip = np.array([0, 3, 3, 6], dtype=np.int32)
    ix = np.array([4, 0, 9, 1, 2, 3, 77], dtype=np.int32)  # the tail past indptr[-1] is ignored
    pkd.check_page_table(ip, ix, 10)
    pkd.check_page_table(ip, ix[:6], 10)
    for pos, val, req in ((2, 10, 0), (4, -1, 2), (0, 2 ** 31 - 1, 0)):
        bad = ix.copy()
        bad[pos] = val
        with pytest.raises(PkdError) as e:
            pkd.check_page_table(ip, bad, 10)
        assert e.value.code == -1
        assert f"request {req}" in str(e.value) and f"indices[{pos}]" in str(e.value)
    with pytest.raises(PkdError):
        pkd.check_page_table(ip, ix[:5], 10)  # fewer ids than indptr[-1]
    with pytest.raises(PkdError):
        pkd.check_page_table(np.array([0, 3, 2, 6], dtype=np.int32), ix, 10)  # decreasing
    pkd.check_page_table(np.array([0], dtype=np.int32), np.zeros(0, np.int32), 1)  # empty batch


def test_workspace_bytes_covers_partials(pkd):
    w = W.workload("long")
    fb, ib = pkd.workspace_bytes(w.indptr, w.last_page_len, 32, 8, 128, 64,
                                 fixed_split_size=256, kv_dtype=1)
    assert fb >= 32 * 32 * 128 * 4 + 32 * 32 * 4
    assert ib >= 256 + 32 * 32 + 4 * 16


@pytest.mark.parametrize("name", ["uniform", "lognormal", "mix", "worked"])
def test_work_capacity_bounds_the_plan(pkd, name):
    """CUDA-graph mode bounds the work list: the heuristic grows its chunks until the items fit,
    and the result is still a valid partition of every request."""
    w = W.workload(name)
    kv = {"f16": 0, "bf16": 1, "e4m3": 2}[w.kv_dtype]
    for cap in (w.batch, w.batch + 1, w.batch + 7, w.batch + 100, 10 * w.batch):
        plan = pkd.plan_host(w.indptr, w.last_page_len, w.num_qo_heads, w.num_kv_heads,
                             w.head_dim, w.page_size, window_left=w.window_left, kv_dtype=kv,
                             work_capacity=cap)
        assert len(plan["tasks"]) <= cap * w.num_kv_heads
        _check_partition(w, plan, 0)


def test_work_capacity_rejects_what_cannot_fit(pkd):
    from paged_kv_decode_23_gb300 import PkdError
    w = W.workload("long")  # fixed split of 256 pages: 8 chunks per request, 32 in all
    with pytest.raises(PkdError) as e:
        pkd.plan_host(w.indptr, w.last_page_len, 32, 8, 128, 64, fixed_split_size=256,
                      kv_dtype=1, work_capacity=31)
    assert e.value.code == -3
    ok = pkd.plan_host(w.indptr, w.last_page_len, 32, 8, 128, 64, fixed_split_size=256,
                       kv_dtype=1, work_capacity=32)
    assert len(ok["tasks"]) == 32 * 8
    with pytest.raises(PkdError):  # more requests than items
        pkd.plan_host(w.indptr, w.last_page_len, 32, 8, 128, 64, work_capacity=3)


def test_graph_workspace_bytes(pkd):
    fb, ib = pkd.graph_workspace_bytes(100, 32, 8, 128)
    # 100 chunks per row in all, per kv head: 800 tasks and slots of 8 heads x 128 floats (and
    # their lses), 400 merge entries with their counters
    assert fb >= 800 * 8 * 128 * 4 + 800 * 8 * 4
    assert ib >= 256 + 400 * 4 + 800 * 48 + 400 * 16


@pytest.mark.parametrize("q_len", [1, 2, 5])
@pytest.mark.parametrize("mode", [dict(), dict(fixed_split_size=3), dict(disable_split_kv=True)])
def test_multi_token_rows_partition_their_causal_keys(pkd, q_len, mode):
    """q_len_per_req > 1: output row i*q_len + j covers exactly the keys its query token sees,
    t <= n - q_len + j within its window, read through request i's pages."""
    lens = [0, 1, 3, 16, 17, 300, 2000]
    window = 40 if "fixed_split_size" in mode else -1
    w = W.custom(lens, 8, 2, 128, 16, window_left=window)
    plan = pkd.plan_host(w.indptr, w.last_page_len, 8, 2, 128, 16, window_left=window,
                         q_len_per_req=q_len, **mode)
    C = mode.get("fixed_split_size", 0) * 16
    _check_partition(w, plan, C, q_len=q_len)


def _mla_partition_ok(plan, kv_indptr, kv_lens):
    """Every request's [0, kv_len) is covered exactly once by its items, in chunk order, and the
    merge entries list exactly the split requests with their consecutive slots."""
    items, merges = plan["items"], plan["merges"]
    by_req = {}
    for it in items:
        by_req.setdefault(int(it[0]), []).append(it)
    assert sorted(by_req) == list(range(len(kv_lens)))
    split = {}
    for r, its in by_req.items():
        n = int(kv_lens[r])
        assert all(int(it[1]) == int(kv_indptr[r]) for it in its)  # the request's first page id
        if n == 0:
            assert len(its) == 1 and its[0][3] == its[0][4] == 0 and its[0][5] == -1
            continue
        spans = sorted((int(it[3]), int(it[4])) for it in its)
        assert spans[0][0] == 0 and spans[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        assert all(it[2] <= it[3] and it[3] < it[4] for it in its)
        if len(its) > 1:
            slots = sorted(int(it[5]) for it in its)
            assert slots == list(range(slots[0], slots[0] + len(its)))
            assert len({int(it[6]) for it in its}) == 1
            split[r] = (slots[0], len(its))
        else:
            assert its[0][5] == -1 and its[0][6] == -1
    assert {int(m[0]): (int(m[1]), int(m[2])) for m in merges} == split
    return split


@pytest.mark.parametrize("backend,heads,ctas", [("fa2", 40, 2), ("fa2", 128, 4),
                                                ("tcgen05", 40, 2), ("tcgen05", 128, 2),
                                                ("tcgen05", 192, 4), ("auto", 64, 2),
                                                ("auto", 128, 2), ("auto", 32, 1),
                                                ("auto", 96, 2)])
def test_mla_plan_partitions_requests(pkd, backend, heads, ctas):
    """MLA work lists (host-only planner): a partition of every request for each kernel, with
    the kernel's CTAs per item (32-head slices for fa2, 128-head CTA pairs for tcgen05; auto
    takes the pair kernel above 32 heads: 96 heads are one pair, not three slices)."""
    w = W.mla_custom([1, 31, 32, 33, 0, 100, 777, 64, 5000, 12000], heads, 16, "bf16", seed=3)
    plan = pkd.mla_plan_host(w.kv_indptr, w.kv_lens, heads, 16, backend=backend)
    assert plan["ctas_per_item"] == ctas
    _mla_partition_ok(plan, w.kv_indptr, w.kv_lens)
    assert plan["float_ws_bytes"] > 0 and plan["int_ws_bytes"] > 0


def test_mla_plan_splits_the_example_into_full_waves(pkd):
    """The wrapper's example (114 x 999 tokens, 128 heads) on 152 SMs (76 CTA pairs): 76 whole
    requests, then 38 requests in two halves -- two full waves of one CTA per SM.  One chunk size
    for every request would give 1.5 waves unsplit or three waves of halves, each wave paying
    the per-item overhead once more."""
    w = W.mla_workload()
    plan = pkd.mla_plan_host(w.kv_indptr, w.kv_lens, 128, 1, backend="auto")
    split = _mla_partition_ok(plan, w.kv_indptr, w.kv_lens)
    assert plan["ctas_per_item"] == 2
    assert len(plan["items"]) == 152 and len(plan["merges"]) == 38
    assert len(split) == 38 and all(n == 2 for _, n in split.values())
    lens = plan["items"][:, 4] - plan["items"][:, 3]
    # longest first: the whole requests fill the first wave, the halves the second
    assert (lens[:76] == 999).all()
    assert lens[76:].min() >= 499 and lens[76:].max() <= 500


def test_mla_plan_fills_whole_waves_on_mixed_lengths(pkd):
    """A batch more than one wave deep: whatever the split, the work items cover every request
    exactly once, and no item is shorter than the minimum chunk unless its request is."""
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 6000, size=300).astype(np.int32)
    w = W.mla_custom(lens.tolist(), 128, 1, "bf16", seed=11)
    plan = pkd.mla_plan_host(w.kv_indptr, w.kv_lens, 128, 1, backend="tcgen05")
    split = _mla_partition_ok(plan, w.kv_indptr, w.kv_lens)
    items = plan["items"]
    ilen = items[:, 4] - items[:, 3]
    assert (np.diff(ilen) <= 0).all()  # longest first
    for r, (_, k) in split.items():
        assert k * 128 <= int(lens[r])  # halves of at least 128 tokens


def test_mla_plan_one_long_request_fills_the_gpu(pkd):
    """One long request alone: the one-wave rule cuts it into one chunk per CTA slot (76 CTA
    pairs of the tcgen05 kernel on 152 SMs), and on a larger GPU into more."""
    w = W.mla_custom([300000], 16, 1, "bf16", seed=2)
    plan = pkd.mla_plan_host(w.kv_indptr, w.kv_lens, 16, 1, backend="tcgen05")
    assert _mla_partition_ok(plan, w.kv_indptr, w.kv_lens)[0][1] == 76
    plan = pkd.mla_plan_host(w.kv_indptr, w.kv_lens, 16, 1, backend="tcgen05", num_sms=400)
    assert _mla_partition_ok(plan, w.kv_indptr, w.kv_lens)[0][1] == 200


def test_mla_graph_workspace_bytes(pkd):
    """CUDA-graph mode sizes the workspaces for the capacity: partials for every item slot of
    every head slice, growing with the capacity and the head count."""
    f1, i1 = pkd.mla_graph_workspace_bytes(100, 128, "tcgen05")
    f2, i2 = pkd.mla_graph_workspace_bytes(200, 128, "tcgen05")
    assert f2 > f1 > 100 * 128 * 512 * 4 and i2 > i1 > 100 * 32
    f3, _ = pkd.mla_graph_workspace_bytes(100, 256, "fa2")
    assert f3 > 100 * 256 * 512 * 4
    with pytest.raises(pkd.PkdError):
        pkd.mla_graph_workspace_bytes(0, 128)
    with pytest.raises(ValueError):
        pkd.mla_graph_workspace_bytes(10, 128, "fa3")


def test_mla_plan_rejects_bad_input(pkd):
    with pytest.raises(pkd.PkdError):  # kv_len beyond the pages
        pkd.mla_plan_host(np.array([0, 1], np.int32), np.array([5], np.int32), 16, 4)
    with pytest.raises(ValueError):
        pkd.mla_plan_host(np.array([0, 1], np.int32), np.array([1], np.int32), 16, 4,
                          backend="fa3")


def _lpt_span(chunk_lens, per_row, slots=304, overhead=352):
    """Makespan of launching per_row tasks per chunk, longest first, each on the CTA slot that
    frees first (brute force with a heap)."""
    import heapq
    tasks = sorted((c + overhead for c in chunk_lens for _ in range(per_row)), reverse=True)
    h = [0] * slots
    for t in tasks:
        heapq.heapreplace(h, h[0] + t)
    return max(h)


@pytest.mark.parametrize("seed", range(6))
def test_one_wave_plans_score_no_worse_than_whole_rows(pkd, seed):
    """For batches whose whole rows fit one wave of CTA slots, the planner's choice (equal
    split or head cut) never has a larger list-scheduling makespan than keeping every row
    whole, counted independently here by brute force (one page of slack: cuts end on page
    boundaries)."""
    rng = np.random.default_rng(seed)
    rows = int(rng.integers(40, 150))
    lens = rng.integers(1, 9000, size=rows).tolist()
    if seed % 2:
        lens[: rows // 2] = [8000] * (rows // 2)  # many long rows, the head cut's case
    w = W.custom(lens, 16, 2, 256, 32, window_left=4096 if seed % 3 == 0 else -1)
    plan = pkd.plan_host(w.indptr, w.last_page_len, 16, 2, 256, 32, window_left=w.window_left,
                         kv_dtype=2)
    _check_partition(w, plan, 0)
    units = _units(plan)
    chunks = [int(t[4]) - int(t[3]) for (r, h, g), ts in units.items() if h == 0 for t in ts]
    whole = [int(ts[-1][4]) - int(ts[0][3]) for (r, h, g), ts in units.items() if h == 0]
    assert _lpt_span(chunks, 2) <= _lpt_span(whole, 2) + 32
