"""CUDA path vs the fp64 oracle, element by element, through the C ABI (libpkd).

Small cases span several tiles and a ragged tail and run every variant (tensor-core and
CUDA-core kernels, NHD/HND, 5-D pool and (k, v) pair, fp16/bf16/e4m3, head_dim 64/128/256,
GQA groups 1..16, page sizes 8..128, soft cap, window, split modes).  Edge cases: empty
requests, single tokens, window 0, an empty batch, NaN/Inf in every slot no request owns.
Properties the pages fix: batch invariance under fixed_split_size, run-to-run determinism.
Full-size workloads are checked on every request in the same launch configuration the
benchmark times.  run()'s calibration scales are checked on every KV dtype and both kernels.
"""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_close, gpu_decoder, run_gpu, run_oracle, sub_problem

pytestmark = pytest.mark.gpu


def _case(lens, hq, hkv, d, ps, layout="NHD", dt="f16", kv=None, seed=0, **kw):
    w = W.custom(lens, hq, hkv, d, ps, layout=layout, q_dtype=dt, kv_dtype=kv or dt, seed=seed, **kw)
    if w.kv_dtype == "e4m3":
        w.kv_store_scale, w.k_scale, w.v_scale = 0.5, 0.5, 0.5
    return w, W.make_q(w), W.make_pool(w)


LENS = [1, 15, 16, 17, 64, 65, 300, 777, 0, 129]


def test_worked_example_both_kernels():
    w = W.workload("worked")
    q, pool = W.make_q(w), W.make_pool(w)
    ref = run_oracle(w, q, pool)
    for tc in (True, False):
        assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), ref, f"worked tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_dtypes_layouts_head_dims(tc, layout, dt, d):
    w, q, pool = _case(LENS, 8, 2, d, 16, layout, dt, seed=d)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"{layout} {dt} D{d} tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (12, 3), (16, 2), (16, 1), (32, 2), (6, 1)])
def test_gqa_groups(tc, hq, hkv):
    w, q, pool = _case([33, 250, 1, 96], hq, hkv, 128, 16, seed=hq * 7 + hkv)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"G{hq // hkv} tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("ps", [8, 32, 64, 128])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_page_sizes(tc, ps, layout):
    w, q, pool = _case([5, ps, ps + 1, 3 * ps - 1, 700], 8, 1, 128, ps, layout, "bf16", seed=ps)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"ps{ps} {layout} tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("cap,window", [(0.0, 0), (0.0, 37), (30.0, -1), (5.0, 100), (1.0, 5000)])
def test_soft_cap_and_window(tc, cap, window):
    w, q, pool = _case(LENS, 8, 2, 128, 16, "NHD", "f16", seed=3, logits_soft_cap=cap,
                       window_left=window)
    q = q * 4  # larger logits so the cap matters
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"cap{cap} win{window} tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("mode", [dict(fixed_split_size=1), dict(fixed_split_size=3),
                                  dict(fixed_split_size=50), dict(disable_split_kv=True), {}])
def test_split_modes(tc, mode):
    w, q, pool = _case([1, 16, 130, 1000, 2047, 0], 8, 2, 128, 16, "HND", "bf16", seed=4,
                       window_left=900 if mode.get("fixed_split_size") == 3 else -1)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc, **mode), run_oracle(w, q, pool),
                 f"{mode} tc={tc}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("qdt", ["f16", "bf16"])
@pytest.mark.parametrize("d", [128, 256])
def test_e4m3_kv(tc, qdt, d):
    w, q, pool = _case(LENS, 16, 2, d, 32, "NHD", qdt, kv="e4m3", seed=d + 1,
                       logits_soft_cap=30.0, window_left=200)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"e4m3 {qdt} D{d} tc={tc}")


@pytest.mark.parametrize("kv,d", [("bf16", 64), ("f16", 128), ("bf16", 256), ("e4m3", 128),
                                  ("e4m3", 256)])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (8, 2), (16, 2), (6, 1)])
@pytest.mark.parametrize("pos", ["NONE", "ALIBI"])
def test_cuda_core_lane_splits(kv, d, hq, hkv, pos):
    """The CUDA-core kernel splits a K/V row over 2..32 lanes depending on head_dim, KV dtype
    and the head group (1, 2, 4, 8 qo heads per CTA, with dead heads in a partial group):
    every split, with 16- and 8-byte lane loads, against the oracle, with a window and a cap
    so rows at slice edges are masked, and with ALiBi (each lane's finished scores take their
    own head's slope)."""
    w, q, pool = _case([1, 9, 64, 300, 1031], hq, hkv, d, 16, "HND",
                       "bf16" if kv == "e4m3" else kv, kv=kv, seed=d + 7 * hq + hkv,
                       logits_soft_cap=20.0, window_left=700)
    got = run_gpu(w, q, pool, use_tensor_cores=False, fixed_split_size=16, pos_encoding_mode=pos)
    assert_close(w, got, run_oracle(w, q, pool, pos_encoding_mode=pos),
                 f"cc {kv} D{d} {hq}/{hkv} {pos}")


def test_e4m3_large_query_values():
    """bf16 q far outside fp16 range still works with e4m3 KV (the tensor-core kernel rescales q)."""
    w, q, pool = _case([40, 300], 8, 1, 128, 16, "NHD", "bf16", kv="e4m3", seed=9,
                       logits_soft_cap=50.0)
    q = (q.float() * 1e5).to(torch.bfloat16)
    for tc in (True, False):
        assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                     f"large q tc={tc}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_kv_tuple_matches_5d(layout):
    w, q, pool = _case(LENS, 8, 4, 128, 16, layout, "f16", seed=5)
    k, v = pool[:, 0].contiguous(), pool[:, 1].contiguous()
    got = run_gpu(w, q, (k, v))
    assert_close(w, got, run_oracle(w, q, pool), f"tuple {layout}")
    five = run_gpu(w, q, pool)
    assert np.array_equal(got[0], five[0]) and np.array_equal(got[1], five[1])


@pytest.mark.parametrize("tc", [True, False])
def test_garbage_in_unowned_slots_is_ignored(tc):
    """Slots past last_page_len and pages no request owns hold NaN/Inf (FlashInfer users have
    met this hazard: a masked-but-read tail poisons the output)."""
    w, q, pool = _case([1, 17, 250, 33, 0], 8, 2, 128, 16, "NHD", "bf16", seed=6,
                       window_left=40)
    clean = run_gpu(w, q, pool, use_tensor_cores=tc)
    dirty = pool.clone()
    owned = np.zeros(w.num_pages, dtype=bool)
    owned[w.indices] = True
    dirty[torch.from_numpy(~owned)] = float("nan")
    for i in range(w.batch):
        if w.indptr[i + 1] > w.indptr[i]:
            last = int(w.indices[w.indptr[i + 1] - 1])
            lp = int(w.last_page_len[i])
            dirty[last, :, lp:] = float("inf") if i % 2 else float("nan")
    got = run_gpu(w, q, dirty, use_tensor_cores=tc)
    assert np.array_equal(got[0], clean[0]) and np.array_equal(got[1], clean[1])
    assert_close(w, got, run_oracle(w, q, pool), f"garbage tc={tc}")


def test_empty_requests_and_empty_batch():
    w, q, pool = _case([0, 0, 5, 0], 4, 2, 64, 8, seed=7)
    o, lse = run_gpu(w, q, pool)
    assert np.all(o[[0, 1, 3]] == 0) and np.all(np.isneginf(lse[[0, 1, 3]]))
    assert_close(w, (o, lse), run_oracle(w, q, pool), "empty requests")
    w0, q0, pool0 = _case([], 4, 2, 64, 8, seed=7)
    o0, lse0 = run_gpu(w0, q0, pool0)
    assert o0.shape == (0, 4, 64) and lse0.shape == (0, 4)


@pytest.mark.parametrize("tc", [True, False])
def test_batch_invariance_with_fixed_split(tc):
    """With fixed_split_size a request's output is bitwise the same alone or in any batch."""
    lens = [3000, 17, 1200, 4096, 64]
    w, q, pool = _case(lens, 16, 2, 128, 16, "HND", "bf16", seed=8)
    full = run_gpu(w, q, pool, use_tensor_cores=tc, fixed_split_size=32)
    for i in (0, 2, 3):
        sub, qs, ps_ = sub_problem(w, [i], q, pool)
        alone = run_gpu(sub, qs, ps_, use_tensor_cores=tc, fixed_split_size=32)
        assert np.array_equal(alone[0][0], full[0][i]), f"request {i} o differs"
        assert np.array_equal(alone[1][0], full[1][i]), f"request {i} lse differs"


@pytest.mark.parametrize("tc", [True, False])
def test_run_to_run_determinism(tc):
    w, q, pool = _case([2500, 100, 7000], 8, 2, 128, 16, "NHD", "f16", seed=10)
    dec = gpu_decoder(w, use_tensor_cores=tc)
    a = run_gpu(w, q, pool, dec=dec)
    b = run_gpu(w, q, pool, dec=dec)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_pdl_on_and_off_agree():
    """Programmatic dependent launch changes only when the kernel is scheduled, not results."""
    w, q, pool = _case([900, 40, 2500], 8, 2, 128, 16, "NHD", "bf16", seed=12)
    dec = gpu_decoder(w)
    dev = torch.device("cuda")
    qd, pd = q.to(dev), pool.to(dev)
    outs = []
    for pdl in (False, True, True, False):
        o, lse = dec.run(qd, pd, return_lse=True, enable_pdl=pdl)
        outs.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert dec.check_status() == 0
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_plan_reused_across_layers():
    w, q, pool = _case([300, 45, 1000], 8, 2, 128, 16, "NHD", "f16", seed=11)
    dec = gpu_decoder(w)
    for layer in range(3):
        ql, pl = W.make_q(w, layer=layer), W.make_pool(w, layer=layer)
        assert_close(w, run_gpu(w, ql, pl, dec=dec), run_oracle(w, ql, pl), f"layer {layer}")


# ----------------------------------------------------------------- full-size workloads
def _full(name, layers=(0,), tc=None):
    """The named workload at full size, planned and launched as the benchmark does, with
    every request's output compared against the oracle (the oracle reads only the pages the
    batch uses, copied to the host)."""
    w = W.workload(name)
    dev = torch.device("cuda")
    dec = gpu_decoder(w, **({} if tc is None else dict(use_tensor_cores=tc)))
    every = list(range(w.batch))
    for layer in layers:
        q = W.make_q(w, device=dev, layer=layer)
        pool = W.make_pool(w, device=dev, layer=layer)
        got = run_gpu(w, q, pool, dec=dec)
        sub, qs, ps_ = sub_problem(w, every, q, pool)
        del pool
        torch.cuda.empty_cache()
        assert_close(sub, got, run_oracle(sub, qs, ps_), f"{name} layer {layer}")


def test_full_uniform_bf16_nhd():
    _full("uniform", layers=(0, 31))


def test_full_lognormal_f16_split():
    _full("lognormal")


def test_full_long_hnd_fixed_split():
    _full("long")


def test_full_mix_e4m3_cap_window():
    _full("mix")


def test_full_worked_example():
    _full("worked")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("kv", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("mode", [dict(fixed_split_size=8), {}])
@pytest.mark.parametrize("scales", [(0.37, 1.0, 1.0), (3.0, 1.0, 1.0), (1.0, 1.7, 0.6),
                                    (0.37, 2.5, 1.9), (3.0, 0.45, 2.2)])
def test_calibration_scales(tc, kv, mode, scales):
    """run()'s q_scale, k_scale and v_scale (the page's calibration scales) on every KV dtype:
    q_scale and k_scale multiply the logit ahead of the soft cap, v_scale the output, through
    split requests merged inside the launch."""
    q_scale, k_scale, v_scale = scales
    w, q, pool = _case([1, 40, 700, 2100, 0, 3000], 16, 2, 128, 16, "NHD",
                       "bf16" if kv == "e4m3" else kv, kv=kv, seed=51, logits_soft_cap=12.0)
    w.k_scale *= k_scale
    w.v_scale *= v_scale
    q = q * 4  # logits of a few units, so the cap bends them and a dropped scale shows
    got = run_gpu(w, q, pool, q_scale=q_scale, use_tensor_cores=tc, **mode)
    assert_close(w, got, run_oracle(w, q, pool, q_scale=q_scale),
                 f"scales {scales} {kv} tc={tc} {mode}")


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("order", ["rising", "falling"])
@pytest.mark.parametrize("tc", [True, False])
def test_scores_drifting_along_the_sequence(kv, order, tc):
    """K rows are constant along head_dim and grow (or shrink) with the token index, so the
    logits sweep ~30 natural-log units along each request: the online softmax's reference
    max has to move many times (rising) or never after the first tile (falling)."""
    lens = [1500, 700, 33, 2100]
    w, q, pool = _case(lens, 16, 2, 128, 16, "NHD", "bf16", kv=kv, seed=13)
    q = torch.ones_like(q)
    vals = pool.float()
    for i, n in enumerate(lens):
        t = np.arange(n)
        ramp = (t if order == "rising" else n - 1 - t) * (2.6 / 2100)
        pages = w.indices[w.indptr[i] + t // w.page_size]
        vals[torch.from_numpy(pages).long(), 0, torch.from_numpy(t % w.page_size).long()] = (
            torch.from_numpy(ramp).float()[:, None, None] / (w.k_scale if kv == "e4m3" else 1.0))
    pool = vals.to(pool.dtype)
    assert_close(w, run_gpu(w, q, pool, use_tensor_cores=tc), run_oracle(w, q, pool),
                 f"{order} {kv} tc={tc}")


@pytest.mark.parametrize("q_len", [2, 3, 5])
@pytest.mark.parametrize("kv,tc", [("bf16", True), ("bf16", False), ("e4m3", True), ("e4m3", False)])
def test_several_query_tokens_per_request(q_len, kv, tc):
    """run's q_len_per_req > 1: each request's last q_len positions attend causally (and
    through their own windows); rows are request-major.  Lengths include requests shorter
    than q_len, whose first query tokens see no key."""
    lens = [1, 2, 16, 17, 300, 1500, 0, 777]
    for mode in (dict(), dict(fixed_split_size=4, window_left=120)):
        w = W.custom(lens, 16, 2, 128, 16, layout="NHD", q_dtype="bf16", kv_dtype=kv,
                     seed=30 + q_len, logits_soft_cap=30.0 if kv == "e4m3" else 0.0,
                     window_left=mode.get("window_left", -1))
        if kv == "e4m3":
            w.kv_store_scale, w.k_scale, w.v_scale = 0.5, 0.5, 0.5
        gen = torch.Generator().manual_seed(77 + q_len)
        q = torch.randn(len(lens) * q_len, 16, 128, generator=gen).to(torch.bfloat16)
        pool = W.make_pool(w)
        got = run_gpu(w, q, pool, use_tensor_cores=tc, q_len_per_req=q_len,
                      fixed_split_size=mode.get("fixed_split_size"))
        assert_close(w, got, run_oracle(w, q, pool, q_len=q_len),
                     f"q_len {q_len} {kv} tc={tc} {mode}")


@pytest.mark.parametrize("kv", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("tc", [True, False])
def test_alibi(kv, tc):
    """pos_encoding_mode ALIBI: slope_g * (t - pos) added to every logit (qo heads 12: slopes
    beyond the largest power of two), with a split, a window and several query tokens."""
    lens = [1, 40, 300, 1200, 0, 2600]
    w, q, pool = _case(lens, 12, 3, 128, 16, "NHD", "bf16" if kv == "e4m3" else kv, kv=kv,
                       seed=41, window_left=700, logits_soft_cap=20.0 if kv == "e4m3" else 0.0)
    for q_len in (1, 2):
        qq = q if q_len == 1 else torch.cat([q, q * 0.5]).reshape(2, -1, 12, 128).transpose(0, 1) \
            .reshape(-1, 12, 128).contiguous()
        got = run_gpu(w, qq, pool, use_tensor_cores=tc, pos_encoding_mode="ALIBI",
                      q_len_per_req=q_len, fixed_split_size=8 if q_len == 2 else None)
        assert_close(w, got, run_oracle(w, qq, pool, q_len=q_len, pos_encoding_mode="ALIBI"),
                     f"alibi {kv} tc={tc} q_len={q_len}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("kv,d", [("f16", 64), ("bf16", 128), ("bf16", 256), ("f16", 256),
                                  ("e4m3", 128), ("e4m3", 256)])
def test_rope_llama(kv, d, tc):
    """pos_encoding_mode ROPE_LLAMA on both kernels: q rotated at its position, every key at
    its index; non-default theta and scale; a split, a window, a soft cap and two query tokens
    per request on the second pass."""
    lens = [1, 17, 333, 1500, 0, 4100]
    qdt = "bf16" if kv == "e4m3" else kv
    w, q, pool = _case(lens, 16, 2, d, 32, "NHD", qdt, kv=kv, seed=d + 5, window_left=2000,
                       logits_soft_cap=30.0)
    for q_len, theta, scale in ((1, 1e4, 1.0), (2, 5e5, 4.0)):
        qq = q.repeat_interleave(q_len, dim=0).contiguous()
        pos = dict(pos_encoding_mode="ROPE_LLAMA", rope_theta=theta, rope_scale=scale)
        got = run_gpu(w, qq, pool, use_tensor_cores=tc, q_len_per_req=q_len, **pos)
        assert_close(w, got, run_oracle(w, qq, pool, q_len=q_len, **pos),
                     f"rope {kv} D{d} tc={tc} q_len={q_len} theta={theta}")


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (12, 2), (6, 1), (32, 2)])
def test_rope_llama_cuda_core_head_groups(kv, d, hq, hkv):
    """ROPE_LLAMA on the CUDA-core kernel at every head-group width it is built for (1, 2, 4,
    8 qo heads per CTA, with dead heads in a partial group; at head_dim 256 the two-stage
    instances too), keys straddling every slice offset of a tile, HND pages of 16 tokens."""
    lens = [1, 8, 9, 16, 250, 1031]
    w, q, pool = _case(lens, hq, hkv, d, 16, "HND", "f16" if kv == "e4m3" else kv, kv=kv,
                       seed=hq * 13 + hkv + d)
    pos = dict(pos_encoding_mode="ROPE_LLAMA", rope_theta=1e4, rope_scale=2.0)
    got = run_gpu(w, q, pool, use_tensor_cores=False, fixed_split_size=256, **pos)
    assert_close(w, got, run_oracle(w, q, pool, **pos), f"rope cuda-core {kv} G{hq // hkv}")


@pytest.mark.parametrize("tc", [True, False])
@pytest.mark.parametrize("kv,d,layout,lens", [
    ("bf16", 128, "HND", [20000, 9000]),
    ("bf16", 128, "HND", [131072, 65553]),
    ("e4m3", 256, "NHD", [131072, 4097]),
])
def test_rope_long_positions_keep_precision(kv, d, layout, lens, tc):
    """Positions up to 131072 (the long-context configuration's length): the kernel's reduced
    angles must track the fp64 oracle (an fp32 angle t * rate alone would drift by ~1e-3 rad
    at 20k and ~1e-2 rad at 131k)."""
    w, q, pool = _case(lens, 16 if kv == "e4m3" else 8, 2 if kv == "e4m3" else 1, d,
                       32 if kv == "e4m3" else 64, layout, "bf16", kv=kv, seed=77 + lens[0] % 97)
    pos = dict(pos_encoding_mode="ROPE_LLAMA", rope_theta=1e4, rope_scale=1.0)
    got = run_gpu(w, q, pool, use_tensor_cores=tc, **pos)
    assert_close(w, got, run_oracle(w, q, pool, **pos),
                 f"rope long positions {kv} D{d} {lens} tc={tc}")


def test_wrapper_keywords_of_the_page():
    """The decode wrapper takes the page's keyword set: run_return_lse is run(return_lse=True);
    backend 'auto' / 'fa2' run this library's kernels, the others (other libraries' kernels),
    jit_args, and plan's block_tables / seq_lens (the trtllm-gen page-table form) are refused."""
    from paged_kv_decode_23_gb300 import BatchDecodePagedKV
    dev = torch.device("cuda")
    w, q, pool = _case([33, 250, 1], 8, 2, 128, 16, seed=12)
    dec = gpu_decoder(w)
    o1, l1 = dec.run(q.to(dev), pool.to(dev), return_lse=True)
    o2, l2 = dec.run_return_lse(q.to(dev), pool.to(dev))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    BatchDecodePagedKV(ws, "NHD", backend="fa2")
    for bad in ("fa3", "trtllm-gen", "cudnn"):
        with pytest.raises(NotImplementedError):
            BatchDecodePagedKV(ws, "NHD", backend=bad)
    with pytest.raises(NotImplementedError):
        BatchDecodePagedKV(ws, "NHD", jit_args=[1])
    with pytest.raises(NotImplementedError):
        gpu_decoder(w, block_tables=torch.zeros(3, 4, dtype=torch.int32, device=dev))
