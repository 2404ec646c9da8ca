"""Pins for the fp64 oracle: checks against facts fixed outside the oracle itself.

Each test ties the oracle to something it cannot agree with by construction: values the
FlashInfer attention API page prints for its worked example, library casts of every
fp16 / bf16 / e4m3 bit pattern, dense brute-force attention written a different way (numpy
einsum + scipy softmax over K/V that are scattered into random pages), closed forms
(single key, two keys, constant V, zero query, window 0) and invariants (page permutation,
GQA as MHA with repeated kv heads, split-and-merge, garbage in unused slots).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- element decoders

def test_f16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(codes, oracle.F16)
    ref = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(codes, oracle.BF16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_array(codes, oracle.E4M3)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    ref = ref.astype(np.float64)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0


# ---------------------------------------------------------------- worked example

def test_worked_example_kv_len_and_shape():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    kv = oracle.kv_len(g["kv_page_indptr"], g["kv_last_page_len"], g["page_size"])
    assert kv.tolist() == g["kv_len_expected"]
    w = W.workload("worked")
    assert list(W.pool_shape(w)) == g["kv_cache_shape_nhd"]
    q = W.make_q(w)
    pool = W.make_pool(w)
    o, lse = oracle.batch_decode_pool(w.indptr, w.indices, w.last_page_len, W.raw_bits(q),
                                      oracle.F16, W.raw_bits(pool), oracle.F16, "NHD",
                                      sm_scale=w.sm_scale)
    assert list(o.shape) == g["output_shape"]
    assert list(lse.shape) == g["output_shape"][:2]
    assert np.isfinite(o).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------- brute force

def _brute(kv_lens, Hq, Hkv, D, q, K, V, sm_scale, cap=0.0, window_left=-1):
    """Dense attention on per-request K/V [n, Hkv, D] (float64), no page table involved."""
    G = Hq // Hkv
    B = len(kv_lens)
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for i in range(B):
        n = kv_lens[i]
        if n == 0:
            continue
        lo = 0 if window_left < 0 else max(0, n - 1 - window_left)
        Kr = np.repeat(K[i][lo:n], G, axis=1)   # [a, Hq, D]
        Vr = np.repeat(V[i][lo:n], G, axis=1)
        x = sm_scale * np.einsum("hd,thd->ht", q[i], Kr)
        s = cap * np.tanh(x / cap) if cap > 0 else x
        o[i] = np.einsum("ht,thd->hd", scipy.special.softmax(s, axis=1), Vr)
        lse[i] = scipy.special.logsumexp(s, axis=1)
    return o, lse


def _scatter(kv_lens, K, V, page_size, layout, rng, extra_pages=3, fill=0.0):
    """Scatter dense per-request K/V into a float64 5-D pool at random pages."""
    Hkv, D = K[0].shape[1], K[0].shape[2]
    npages = [(n + page_size - 1) // page_size for n in kv_lens]
    total = sum(npages)
    P = total + extra_pages
    perm = rng.permutation(P)
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    indices = perm[:total].astype(np.int32)
    lpl = np.array([n - (p - 1) * page_size if p else 0 for n, p in zip(kv_lens, npages)],
                   dtype=np.int32)
    shape = (P, 2, page_size, Hkv, D) if layout == "NHD" else (P, 2, Hkv, page_size, D)
    pool = np.full(shape, fill, dtype=np.float64)
    for i, n in enumerate(kv_lens):
        for t in range(n):
            page = indices[indptr[i] + t // page_size]
            slot = t % page_size
            if layout == "NHD":
                pool[page, 0, slot] = K[i][t]
                pool[page, 1, slot] = V[i][t]
            else:
                pool[page, 0, :, slot] = K[i][t]
                pool[page, 1, :, slot] = V[i][t]
    return indptr, indices, lpl, pool


def _run_f64(indptr, indices, lpl, q, pool, layout, **kw):
    return oracle.batch_decode_pool(indptr, indices, lpl, np.ascontiguousarray(q), oracle.F64,
                                    pool, oracle.F64, layout, **kw)


def _rand_problem(rng, kv_lens, Hq, Hkv, D):
    q = rng.standard_normal((len(kv_lens), Hq, D))
    K = [rng.standard_normal((n, Hkv, D)) for n in kv_lens]
    V = [rng.standard_normal((n, Hkv, D)) for n in kv_lens]
    return q, K, V


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("case", [
    dict(kv_lens=[5, 17, 40], Hq=4, Hkv=2, D=8, ps=4),
    dict(kv_lens=[1, 16, 33], Hq=6, Hkv=3, D=16, ps=8, cap=2.5),
    dict(kv_lens=[9, 31, 2], Hq=4, Hkv=1, D=4, ps=3, window_left=5),
    dict(kv_lens=[0, 12, 7], Hq=2, Hkv=2, D=8, ps=4, cap=1.0, window_left=0),
])
def test_brute_force_agreement(layout, case):
    rng = np.random.default_rng(1234)
    kv_lens, Hq, Hkv, D, ps = case["kv_lens"], case["Hq"], case["Hkv"], case["D"], case["ps"]
    cap, wl = case.get("cap", 0.0), case.get("window_left", -1)
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    sm = 0.37
    ref_o, ref_lse = _brute(kv_lens, Hq, Hkv, D, q, K, V, sm, cap, wl)
    indptr, indices, lpl, pool = _scatter(kv_lens, K, V, ps, layout, rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, layout, sm_scale=sm, logits_soft_cap=cap,
                      window_left=wl)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)


def _brute_multi(kv_lens, q_len, Hq, Hkv, D, q, K, V, sm_scale, cap=0.0, window_left=-1):
    """Dense attention of q_len query tokens per request under the causal mask of the batch
    prefill example, tril(ones(qo_len, kv_len), diagonal=kv_len - qo_len), narrowed by a
    left window band of window_left + 1 keys per row.  q: [B, q_len, Hq, D]."""
    G = Hq // Hkv
    B = len(kv_lens)
    o = np.zeros((B, q_len, Hq, D))
    lse = np.full((B, q_len, Hq), -np.inf)
    for i in range(B):
        n = kv_lens[i]
        if n == 0:
            continue
        mask = np.tril(np.ones((q_len, n), dtype=bool), k=n - q_len)
        if window_left >= 0:
            mask &= ~np.tril(np.ones((q_len, n), dtype=bool), k=n - q_len - window_left - 1)
        Kr = np.repeat(K[i], G, axis=1)  # [n, Hq, D]
        Vr = np.repeat(V[i], G, axis=1)
        for j in range(q_len):
            if not mask[j].any():
                continue
            x = sm_scale * np.einsum("hd,thd->ht", q[i, j], Kr[mask[j]])
            s = cap * np.tanh(x / cap) if cap > 0 else x
            o[i, j] = np.einsum("ht,thd->hd", scipy.special.softmax(s, axis=1), Vr[mask[j]])
            lse[i, j] = scipy.special.logsumexp(s, axis=1)
    return o.reshape(B * q_len, Hq, D), lse.reshape(B * q_len, Hq)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("case", [
    dict(kv_lens=[5, 17, 40], q_len=3, Hq=4, Hkv=2, D=8, ps=4),
    dict(kv_lens=[1, 2, 33], q_len=4, Hq=6, Hkv=3, D=16, ps=8, cap=2.5),
    dict(kv_lens=[9, 31, 0], q_len=2, Hq=4, Hkv=1, D=4, ps=3, window_left=5),
    dict(kv_lens=[12, 7], q_len=5, Hq=2, Hkv=2, D=8, ps=4, window_left=0),
])
def test_multi_token_queries_brute_force(layout, case):
    """q_len_per_req > 1 (run's q_len_per_req): each request's last q_len positions attend
    causally; requests shorter than q_len leave their first query tokens with no key."""
    rng = np.random.default_rng(4321)
    kv_lens, ql = case["kv_lens"], case["q_len"]
    Hq, Hkv, D, ps = case["Hq"], case["Hkv"], case["D"], case["ps"]
    cap, wl = case.get("cap", 0.0), case.get("window_left", -1)
    q = rng.standard_normal((len(kv_lens), ql, Hq, D))
    K = [rng.standard_normal((n, Hkv, D)) for n in kv_lens]
    V = [rng.standard_normal((n, Hkv, D)) for n in kv_lens]
    sm = 0.41
    ref_o, ref_lse = _brute_multi(kv_lens, ql, Hq, Hkv, D, q, K, V, sm, cap, wl)
    indptr, indices, lpl, pool = _scatter(kv_lens, K, V, ps, layout, rng)
    o, lse = _run_f64(indptr, indices, lpl, q.reshape(-1, Hq, D), pool, layout, sm_scale=sm,
                      logits_soft_cap=cap, window_left=wl, q_len=ql)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    # the last query token of every request is plain decode
    o1, lse1 = _run_f64(indptr, indices, lpl, np.ascontiguousarray(q[:, -1]), pool, layout,
                        sm_scale=sm, logits_soft_cap=cap, window_left=wl)
    np.testing.assert_array_equal(o.reshape(len(kv_lens), ql, Hq, D)[:, -1], o1)


# ------------------------------------------------- positional encoding (pos_encoding_mode)

def _rope_complex(x, pos, theta, scale):
    """ROPE_LLAMA written with complex numbers: pair (x_i, x_{i+D/2}) is z = x_i + i*x_{i+D/2},
    rotated by multiplying with exp(i * (pos / scale) * theta^(-2i/D))."""
    D = x.shape[-1]
    half = D // 2
    z = x[..., :half] + 1j * x[..., half:]
    ang = (pos / scale) * theta ** (-2.0 * np.arange(half) / D)
    z = z * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


def _alibi_slopes(H):
    """ALiBi slopes: the geometric sequence starting at 2^(-8/m) with ratio 2^(-8/m) for the
    largest power of two m <= H, completed by every other slope of the 2m-head sequence."""
    m = 2 ** int(np.floor(np.log2(H)))
    first = [(2.0 ** (-8.0 / m)) ** (k + 1) for k in range(m)]
    rest = [(2.0 ** (-8.0 / (2 * m))) ** (k + 1) for k in range(0, 2 * (H - m), 2)]
    return np.array(first + rest)


def _brute_pos(kv_lens, Hq, Hkv, D, q, K, V, sm, mode, theta=1e4, scale=1.0, window_left=-1,
               cap=0.0):
    """Dense decode attention with the positional encoding applied to dense q / K."""
    G = Hq // Hkv
    o = np.zeros((len(kv_lens), Hq, D))
    lse = np.full((len(kv_lens), Hq), -np.inf)
    slopes = _alibi_slopes(Hq)
    for i, n in enumerate(kv_lens):
        if n == 0:
            continue
        lo = 0 if window_left < 0 else max(0, n - 1 - window_left)
        t = np.arange(lo, n)
        Kr = np.repeat(K[i][lo:n], G, axis=1)
        Vr = np.repeat(V[i][lo:n], G, axis=1)
        qi = q[i]
        if mode == "ROPE_LLAMA":
            qi = _rope_complex(qi, n - 1, theta, scale)
            Kr = np.stack([_rope_complex(Kr[k], t[k], theta, scale) for k in range(len(t))])
        x = sm * np.einsum("hd,thd->ht", qi, Kr)
        if mode == "ALIBI":
            x = x + slopes[:, None] * (t[None, :] - (n - 1))
        s = cap * np.tanh(x / cap) if cap > 0 else x
        o[i] = np.einsum("ht,thd->hd", scipy.special.softmax(s, axis=1), Vr)
        lse[i] = scipy.special.logsumexp(s, axis=1)
    return o, lse


@pytest.mark.parametrize("case", [
    dict(mode="ROPE_LLAMA", kv_lens=[5, 40, 0, 17], Hq=4, Hkv=2, D=8),
    dict(mode="ROPE_LLAMA", kv_lens=[300, 33], Hq=2, Hkv=1, D=16, theta=500.0, scale=2.5,
         window_left=50),
    dict(mode="ALIBI", kv_lens=[5, 40, 17], Hq=8, Hkv=2, D=8),
    dict(mode="ALIBI", kv_lens=[60, 3], Hq=6, Hkv=3, D=8, cap=3.0),
])
def test_positional_encoding_brute_force(case):
    rng = np.random.default_rng(99)
    kv_lens, Hq, Hkv, D = case["kv_lens"], case["Hq"], case["Hkv"], case["D"]
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    kw = dict(theta=case.get("theta", 1e4), scale=case.get("scale", 1.0),
              window_left=case.get("window_left", -1), cap=case.get("cap", 0.0))
    ref_o, ref_lse = _brute_pos(kv_lens, Hq, Hkv, D, q, K, V, 0.3, case["mode"], **kw)
    indptr, indices, lpl, pool = _scatter(kv_lens, K, V, 4, "NHD", rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=0.3,
                      pos_encoding_mode=case["mode"], rope_theta=kw["theta"],
                      rope_scale=kw["scale"], window_left=kw["window_left"],
                      logits_soft_cap=kw["cap"])
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-11)
    fin = np.isfinite(ref_lse)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-11)


def test_alibi_slopes_of_eight_heads_are_powers_of_one_half():
    """The ALiBi paper's example: 8 heads take 1/2, 1/4, ..., 1/256.  One key at distance d
    behind the query, with q = 0, gets logit -slope*d: lse over {d, 0} = log(1 + 2^(-d*k))."""
    np.testing.assert_allclose(_alibi_slopes(8), [2.0 ** -(k + 1) for k in range(8)], rtol=1e-15)
    D, H = 4, 8
    q = np.zeros((1, H, D))
    K = [np.zeros((2, 1, D))]
    V = [np.ones((2, 1, D))]
    rng = np.random.default_rng(3)
    indptr, indices, lpl, pool = _scatter([2], K, V, 4, "NHD", rng)
    _, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=1.0,
                      pos_encoding_mode="ALIBI")
    np.testing.assert_allclose(lse[0], np.log1p(np.exp(-2.0 ** -(np.arange(H) + 1.0))),
                               rtol=0, atol=1e-14)


def _oracle_alibi_slopes(H):
    """The slopes the oracle applies, read back from its output: per head, two keys at
    distances 1 and 0 behind the query with q = 0, V = 1 for the first key and 0 for the
    second, so o = e^-s / (1 + e^-s) and s = ln((1 - o) / o)."""
    D = 4
    q = np.zeros((1, H, D))
    K = [np.zeros((2, 1, D))]
    V = [np.stack([np.ones((1, D)), np.zeros((1, D))])]
    rng = np.random.default_rng(5)
    indptr, indices, lpl, pool = _scatter([2], K, V, 4, "NHD", rng)
    o, _ = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=1.0,
                    pos_encoding_mode="ALIBI")
    p = o[0, :, 0]
    return np.log((1.0 - p) / p)


@pytest.mark.parametrize("heads", [8, 16, 12])
def test_alibi_slopes_match_the_published_sets(heads):
    """The oracle's ALiBi slopes against the values the ALiBi paper prints (tests/golden/
    alibi_slopes.json): its 8- and 16-head sets, and for 12 heads (not a power of two, as in
    the GPU ALiBi test) the 8-head set followed by alternate entries of the 16-head set."""
    g = json.load(open(os.path.join(GOLDEN, "alibi_slopes.json")))
    want = 2.0 ** -np.asarray(g[f"heads_{heads}"], dtype=np.float64)
    np.testing.assert_allclose(_oracle_alibi_slopes(heads), want, rtol=1e-12, atol=0)


def test_rope_depends_only_on_relative_position():
    """Rotating q at p and k at t gives a logit that depends only on t - p: a request whose
    keys are preceded by s unattended tokens (window) returns the same output as the bare
    request (ALiBi's bias depends on t - p as well)."""
    rng = np.random.default_rng(11)
    D, m, s_pad = 16, 9, 23
    q = rng.standard_normal((1, 2, D))
    Kc = rng.standard_normal((m, 1, D))
    Vc = rng.standard_normal((m, 1, D))
    junk = rng.standard_normal((s_pad, 1, D))
    i1, x1, l1, p1 = _scatter([m], [Kc], [Vc], 4, "NHD", rng)
    i2, x2, l2, p2 = _scatter([m + s_pad], [np.concatenate([junk, Kc])],
                              [np.concatenate([junk, Vc])], 4, "NHD", rng)
    for mode in ("ROPE_LLAMA", "ALIBI"):
        o1, lse1 = _run_f64(i1, x1, l1, q, p1, "NHD", sm_scale=0.5, pos_encoding_mode=mode)
        o2, lse2 = _run_f64(i2, x2, l2, q, p2, "NHD", sm_scale=0.5, pos_encoding_mode=mode,
                            window_left=m - 1)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse1, rtol=0, atol=1e-12)
    # a key equal to q at the query's own position: both get the same rotation, so the logit
    # is |q|^2 (a rotation preserves dot products)
    K1 = [np.repeat(q[:, :1, :], 1, axis=0).reshape(1, 1, D)]
    i3, x3, l3, p3 = _scatter([1], K1, [np.ones((1, 1, D))], 4, "NHD", rng)
    _, lse3 = _run_f64(i3, x3, l3, q[:, :1, :].copy(), p3, "NHD", sm_scale=1.0,
                       num_qo_heads=1, pos_encoding_mode="ROPE_LLAMA")
    np.testing.assert_allclose(lse3[0, 0], np.sum(q[0, 0] ** 2), rtol=1e-13)


def test_scales_multiply_inputs():
    rng = np.random.default_rng(7)
    kv_lens, Hq, Hkv, D = [6, 11], 4, 2, 8
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    qs, ks, vs = 0.5, 3.0, 0.25
    ref_o, ref_lse = _brute(kv_lens, Hq, Hkv, D, qs * q, [ks * k for k in K],
                            [vs * v for v in V], 0.3)
    indptr, indices, lpl, pool = _scatter(kv_lens, K, V, 4, "NHD", rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=0.3, q_scale=qs,
                      k_scale=ks, v_scale=vs)
    np.testing.assert_allclose(o, ref_o, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_default_sm_scale_is_inverse_sqrt_head_dim():
    rng = np.random.default_rng(8)
    kv_lens, Hq, Hkv, D = [7, 3], 2, 1, 16
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    ref_o, ref_lse = _brute(kv_lens, Hq, Hkv, D, q, K, V, 0.25)
    indptr, indices, lpl, pool = _scatter(kv_lens, K, V, 4, "NHD", rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD")
    np.testing.assert_allclose(o, ref_o, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def _single_request(rng, n, D=8, Hkv=1, Hq=1, ps=4):
    q, K, V = _rand_problem(rng, [n], Hq, Hkv, D)
    indptr, indices, lpl, pool = _scatter([n], K, V, ps, "NHD", rng)
    return q, K, V, indptr, indices, lpl, pool


def test_single_key_returns_v0_and_its_logit():
    rng = np.random.default_rng(3)
    q, K, V, indptr, indices, lpl, pool = _single_request(rng, 1)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=0.5)
    assert np.array_equal(o[0, 0], V[0][0, 0])
    assert lse[0, 0] == pytest.approx(0.5 * float(np.dot(q[0, 0], K[0][0, 0])), abs=1e-13)


def test_two_keys_closed_form():
    rng = np.random.default_rng(4)
    q, K, V, indptr, indices, lpl, pool = _single_request(rng, 2, D=4)
    sm = 0.7
    s0 = sm * sum(a * b for a, b in zip(q[0, 0], K[0][0, 0]))
    s1 = sm * sum(a * b for a, b in zip(q[0, 0], K[0][1, 0]))
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = [w0 * a + w1 * b for a, b in zip(V[0][0, 0], V[0][1, 0])]
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", sm_scale=sm)
    np.testing.assert_allclose(o[0, 0], expect, atol=1e-14)
    assert lse[0, 0] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                                      abs=1e-13)


def test_window_zero_returns_last_value():
    rng = np.random.default_rng(5)
    q, K, V, indptr, indices, lpl, pool = _single_request(rng, 23)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", window_left=0, sm_scale=0.3)
    assert np.array_equal(o[0, 0], V[0][22, 0])
    assert lse[0, 0] == pytest.approx(0.3 * float(np.dot(q[0, 0], K[0][22, 0])), abs=1e-13)


def test_constant_v_is_returned_unchanged():
    rng = np.random.default_rng(6)
    n, D = 37, 8
    q, K, V = _rand_problem(rng, [n], 2, 1, D)
    c = rng.standard_normal(D)
    V = [np.broadcast_to(c, (n, 1, D)).copy()]
    indptr, indices, lpl, pool = _scatter([n], K, V, 8, "HND", rng)
    o, _ = _run_f64(indptr, indices, lpl, q, pool, "HND", sm_scale=1.3)
    np.testing.assert_allclose(o[0, 0], c, atol=1e-12)
    np.testing.assert_allclose(o[0, 1], c, atol=1e-12)


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(9)
    n, D, wl = 29, 8, 10
    q, K, V = _rand_problem(rng, [n], 1, 1, D)
    q[:] = 0.0
    indptr, indices, lpl, pool = _scatter([n], K, V, 4, "NHD", rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD", window_left=wl)
    np.testing.assert_allclose(o[0, 0], V[0][n - 1 - wl:, 0].mean(axis=0), atol=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(wl + 1), abs=1e-13)


def test_empty_request_gives_zero_and_minus_inf():
    rng = np.random.default_rng(10)
    q, K, V = _rand_problem(rng, [0, 5], 2, 1, 8)
    indptr, indices, lpl, pool = _scatter([0, 5], K, V, 4, "NHD", rng)
    o, lse = _run_f64(indptr, indices, lpl, q, pool, "NHD")
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.isfinite(lse[1]).all()


# ---------------------------------------------------------------- invariants

def test_page_permutation_invariance_bitwise():
    rng = np.random.default_rng(11)
    kv_lens, Hq, Hkv, D, ps = [13, 40, 7], 4, 2, 8, 4
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    a = _run_f64(*_scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(1))[:3], q,
                 _scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(1))[3], "NHD")
    ip, ix, lpl, pool = _scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(2))
    b = _run_f64(ip, ix, lpl, q, pool, "NHD")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_unused_slots_never_matter():
    """Slots past last_page_len and pages no request owns may hold NaN / Inf."""
    rng = np.random.default_rng(12)
    kv_lens, Hq, Hkv, D, ps = [13, 6, 21], 4, 2, 8, 8
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    ip, ix, lpl, clean = _scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(5), fill=0.0)
    _, _, _, dirty = _scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(5), fill=np.nan)
    dirty[-1] = np.inf
    a = _run_f64(ip, ix, lpl, q, clean, "NHD", window_left=9)
    b = _run_f64(ip, ix, lpl, q, dirty, "NHD", window_left=9)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(13)
    kv_lens, Hq, Hkv, D, ps = [19, 8], 6, 2, 8, 4
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    G = Hq // Hkv
    ip, ix, lpl, pool = _scatter(kv_lens, K, V, ps, "NHD", np.random.default_rng(3))
    gqa = _run_f64(ip, ix, lpl, q, pool, "NHD", num_qo_heads=Hq)
    K2 = [np.repeat(k, G, axis=1) for k in K]
    V2 = [np.repeat(v, G, axis=1) for v in V]
    ip2, ix2, lpl2, pool2 = _scatter(kv_lens, K2, V2, ps, "NHD", np.random.default_rng(3))
    mha = _run_f64(ip2, ix2, lpl2, q, pool2, "NHD")
    np.testing.assert_allclose(gqa[0], mha[0], atol=1e-13)
    np.testing.assert_allclose(gqa[1], mha[1], atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 4, 7, 16, 1000])
def test_split_and_merge_equals_unsplit(chunk):
    rng = np.random.default_rng(14)
    kv_lens, Hq, Hkv, D, ps = [33, 1, 60, 0], 4, 2, 8, 4
    q, K, V = _rand_problem(rng, kv_lens, Hq, Hkv, D)
    ip, ix, lpl, pool = _scatter(kv_lens, K, V, ps, "HND", rng)
    for wl, cap in ((-1, 0.0), (20, 3.0)):
        a = _run_f64(ip, ix, lpl, q, pool, "HND", window_left=wl, logits_soft_cap=cap)
        b = _run_f64(ip, ix, lpl, q, pool, "HND", window_left=wl, logits_soft_cap=cap,
                     chunk_tokens=chunk)
        np.testing.assert_allclose(b[0], a[0], atol=1e-12)
        np.testing.assert_allclose(b[1], a[1], atol=1e-12)


def test_merge_states_against_concatenation():
    """Merging two disjoint key sets equals attending over their union (brute force)."""
    rng = np.random.default_rng(15)
    s = rng.standard_normal(11) * 3
    v = rng.standard_normal((11, 5))
    parts_o, parts_lse = [], []
    for lo, hi in ((0, 4), (4, 11)):
        w = scipy.special.softmax(s[lo:hi])
        parts_o.append(w @ v[lo:hi])
        parts_lse.append(scipy.special.logsumexp(s[lo:hi]))
    o, lse = oracle.merge_states(np.array(parts_o), np.array(parts_lse))
    np.testing.assert_allclose(o, scipy.special.softmax(s) @ v, atol=1e-14)
    assert lse == pytest.approx(scipy.special.logsumexp(s), abs=1e-14)
    o2, lse2 = oracle.merge_states(np.array(parts_o + [np.zeros(5)]),
                                   np.array(parts_lse + [-np.inf]))
    np.testing.assert_array_equal(o2, o)
    assert lse2 == lse


def test_window_at_least_length_is_no_window_and_large_cap_is_no_cap():
    rng = np.random.default_rng(16)
    kv_lens = [12, 30]
    q, K, V = _rand_problem(rng, kv_lens, 2, 1, 8)
    ip, ix, lpl, pool = _scatter(kv_lens, K, V, 4, "NHD", rng)
    base = _run_f64(ip, ix, lpl, q, pool, "NHD")
    for wl in (29, 30, 10 ** 6):
        a = _run_f64(ip, ix, lpl, q, pool, "NHD", window_left=wl)
        assert np.array_equal(a[0], base[0]) and np.array_equal(a[1], base[1])
    b = _run_f64(ip, ix, lpl, q, pool, "NHD", logits_soft_cap=1e6)
    np.testing.assert_allclose(b[0], base[0], atol=1e-9)
    np.testing.assert_allclose(b[1], base[1], atol=1e-9)


def test_soft_cap_bounds_lse():
    """With cap c every logit lies in [-c, c], so lse lies in [-c, c] + ln(#keys)."""
    rng = np.random.default_rng(17)
    kv_lens = [50]
    q, K, V = _rand_problem(rng, kv_lens, 2, 1, 8)
    q *= 40.0
    ip, ix, lpl, pool = _scatter(kv_lens, K, V, 8, "NHD", rng)
    cap = 2.0
    _, lse = _run_f64(ip, ix, lpl, q, pool, "NHD", logits_soft_cap=cap, sm_scale=1.0)
    assert np.all(lse <= cap + math.log(50) + 1e-12)
    assert np.all(lse >= -cap + math.log(50) - 1e-12)


def test_rejects_malformed_tables():
    rng = np.random.default_rng(18)
    q, K, V = _rand_problem(rng, [5], 3, 2, 8)   # 3 qo heads, 2 kv heads: not a multiple
    ip, ix, lpl, pool = _scatter([5], K, V, 4, "NHD", rng)
    with pytest.raises(ValueError):
        _run_f64(ip, ix, lpl, q, pool, "NHD")
    q, K, V = _rand_problem(rng, [5], 2, 2, 8)
    ip, ix, lpl, pool = _scatter([5], K, V, 4, "NHD", rng)
    bad = lpl.copy()
    bad[0] = 5                                  # last_page_len > page_size
    with pytest.raises(ValueError):
        _run_f64(ip, ix, bad, q, pool, "NHD")


# ---------------------------------------------------------------- MLA decode

def _mla_problem(rng, kv_lens, H, dc, dp, ps, extra_pages=5):
    pages = [(n + ps - 1) // ps for n in kv_lens]
    P = sum(pages) + extra_pages
    perm = rng.permutation(P)
    kv_indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    kv_indices = perm[:kv_indptr[-1]].astype(np.int32)
    ckv = rng.standard_normal((P, ps, dc))
    kpe = rng.standard_normal((P, ps, dp))
    q_nope = rng.standard_normal((len(kv_lens), H, dc))
    q_pe = rng.standard_normal((len(kv_lens), H, dp))
    return kv_indptr, kv_indices, np.asarray(kv_lens, np.int32), q_nope, q_pe, ckv, kpe


@pytest.mark.parametrize("case", [dict(kv_lens=[1, 7, 33, 0], H=4, dc=16, dp=8, ps=1),
                                  dict(kv_lens=[50, 3], H=3, dc=32, dp=8, ps=4)])
def test_mla_against_dense_latent_attention(case):
    """Key = [ckv, kpe], value = ckv, one latent cache shared by every head (the page's
    matrix-absorbed MLA), computed densely with numpy."""
    rng = np.random.default_rng(123)
    ip, ix, lens, qn, qp, ckv, kpe = _mla_problem(rng, case["kv_lens"], case["H"], case["dc"],
                                                  case["dp"], case["ps"])
    sm = 0.21
    o, lse = oracle.mla_decode(ip, ix, lens, qn, qp, oracle.F64, ckv, kpe, oracle.F64,
                               case["ps"], sm)
    for i, n in enumerate(lens):
        if n == 0:
            assert np.all(o[i] == 0) and np.all(np.isneginf(lse[i]))
            continue
        t = np.arange(n)
        rows = ix[ip[i] + t // case["ps"]], t % case["ps"]
        C, Pe = ckv[rows], kpe[rows]          # [n, dc], [n, dp]
        logits = sm * (qn[i] @ C.T + qp[i] @ Pe.T)
        np.testing.assert_allclose(o[i], scipy.special.softmax(logits, axis=1) @ C, atol=1e-12)
        np.testing.assert_allclose(lse[i], scipy.special.logsumexp(logits, axis=1), atol=1e-12)


def test_mla_is_decode_with_one_concatenated_kv_head():
    """MLA equals the (separately pinned) GQA decode oracle with one kv head of dim dc + dp,
    K = [ckv, kpe], V = [ckv, 0], q = [q_nope, q_pe], on the first dc output dims."""
    rng = np.random.default_rng(7)
    H, dc, dp, ps = 4, 16, 8, 2
    ip, ix, lens, qn, qp, ckv, kpe = _mla_problem(rng, [9, 1, 20], H, dc, dp, ps)
    o, lse = oracle.mla_decode(ip, ix, lens, qn, qp, oracle.F64, ckv, kpe, oracle.F64, ps, 0.4)
    P = ckv.shape[0]
    pool = np.zeros((P, 2, ps, 1, dc + dp))
    pool[:, 0, :, 0, :dc] = ckv
    pool[:, 0, :, 0, dc:] = kpe
    pool[:, 1, :, 0, :dc] = ckv
    lpl = np.array([n - (ip[i + 1] - ip[i] - 1) * ps for i, n in enumerate(lens)], np.int32)
    q = np.concatenate([qn, qp], axis=2)
    o2, lse2 = _run_f64(ip, ix, lpl, q, pool, "NHD", sm_scale=0.4)
    np.testing.assert_allclose(o, o2[:, :, :dc], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_mla_single_token_returns_its_latent_row():
    rng = np.random.default_rng(8)
    ip, ix, lens, qn, qp, ckv, kpe = _mla_problem(rng, [1], 2, 8, 4, 1)
    o, lse = oracle.mla_decode(ip, ix, lens, qn, qp, oracle.F64, ckv, kpe, oracle.F64, 1, 0.5)
    row = ckv[ix[0], 0]
    np.testing.assert_array_equal(o[0], np.stack([row, row]))
    np.testing.assert_allclose(lse[0], 0.5 * (qn[0] @ row + qp[0] @ kpe[ix[0], 0]), atol=1e-13)
