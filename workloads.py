"""Seeded synthetic inputs for batch decode over a paged KV cache.

This module only draws random numbers and lays them out as page tables, query tensors and
paged K/V pools.  It holds none of the attention arithmetic, so both the CUDA path's tests
and the CPU oracle can take their inputs from it without sharing any of the method.

Workload recipes (shapes follow the FlashInfer attention API page, BatchDecodeWithPaged-
KVCacheWrapper: the worked example of its class docstring and the plan()/run() shapes):

  worked    batch 7, indptr [0,17,29,44,48,66,100,128], indices arange(128),
            last_page_len [1,7,14,4,3,1,16], page 16, 64/8 heads, D 128, fp16, NHD
  uniform   batch 64, kv_len ~ U{512..4096}, page 16, 32/8 heads, D 128, bf16, NHD,
            32 layers of independent pools, one plan
  lognormal batch 256, kv_len = clip(round(exp(N(ln 2048, 1))), 16, 32768), page 16,
            64/8 heads, D 128, fp16, NHD, split-KV by heuristic
  long      batch 4, kv_len 131072, page 64, 32/8 heads, D 128, bf16, HND,
            fixed split of 256 pages
  mix       batch 128, kv_len ~ U{1..8192}, page 32, 16/2 heads, D 256, fp8 e4m3 K/V
            stored as e4m3(x / 0.5) with k_scale = v_scale = 0.5, bf16 q and o,
            logits soft cap 30, window_left 4096, NHD

Every pool except the worked example's holds twice the pages the batch needs; the pages a
request uses are the leading entries of a seeded random permutation of the pool, handed out
in request order.  Values are N(0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

WORKED_INDPTR = [0, 17, 29, 44, 48, 66, 100, 128]
WORKED_LAST_PAGE_LEN = [1, 7, 14, 4, 3, 1, 16]

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


@dataclass
class Workload:
    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str
    q_dtype: str
    kv_dtype: str
    o_dtype: str
    kv_lens: np.ndarray            # requested lengths, int64 [batch]
    indptr: np.ndarray             # int32 [batch + 1]
    indices: np.ndarray            # int32 [indptr[-1]]
    last_page_len: np.ndarray      # int32 [batch]
    num_pages: int                 # pages in the pool
    sm_scale: float | None = None
    logits_soft_cap: float = 0.0
    window_left: int = -1
    fixed_split_size: int = 0
    disable_split_kv: bool = False
    kv_store_scale: float = 1.0    # stored K/V = value / kv_store_scale (fp8 only)
    k_scale: float = 1.0
    v_scale: float = 1.0
    layers: int = 1
    seed: int = 0
    meta: dict = field(default_factory=dict)


def page_table(kv_lens, page_size: int, pool_factor: float = 2.0, permute: bool = True,
               seed: int = 0, min_pool_pages: int = 1):
    """Page table for the given per-request token counts.

    A request of n > 0 tokens gets ceil(n / page_size) pages and a last page holding
    n - (pages - 1) * page_size tokens; a request of 0 tokens gets no page and a
    last_page_len of 0.  Returns (indptr, indices, last_page_len, num_pages).
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    pages = np.where(kv_lens > 0, (kv_lens + page_size - 1) // page_size, 0)
    lpl = np.where(kv_lens > 0, kv_lens - (pages - 1) * page_size, 0)
    indptr = np.zeros(len(kv_lens) + 1, dtype=np.int64)
    np.cumsum(pages, out=indptr[1:])
    total = int(indptr[-1])
    num_pages = max(min_pool_pages, int(np.ceil(total * pool_factor)))
    if permute:
        rng = np.random.Generator(np.random.PCG64(seed + 7919))
        order = rng.permutation(num_pages)
    else:
        order = np.arange(num_pages)
    indices = order[:total].astype(np.int32)
    return indptr.astype(np.int32), indices, lpl.astype(np.int32), num_pages


def _lengths(kind: str, batch: int, rng: np.random.Generator) -> np.ndarray:
    if kind == "uniform":
        return rng.integers(512, 4096, size=batch, endpoint=True)
    if kind == "lognormal":
        x = np.exp(rng.normal(np.log(2048.0), 1.0, size=batch))
        return np.clip(np.round(x), 16, 32768).astype(np.int64)
    if kind == "mix":
        return rng.integers(1, 8192, size=batch, endpoint=True)
    raise ValueError(kind)


def workload(name: str, seed: int = 0, batch: int | None = None) -> Workload:
    """The named workload's page table and parameters (tensors are made separately)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "worked":
        indptr = np.array(WORKED_INDPTR, dtype=np.int32)
        lpl = np.array(WORKED_LAST_PAGE_LEN, dtype=np.int32)
        lens = 16 * (np.diff(indptr).astype(np.int64) - 1) + lpl
        return Workload(name, 7, 64, 8, 128, 16, "NHD", "f16", "f16", "f16", lens, indptr,
                        np.arange(128, dtype=np.int32), lpl, 128,
                        sm_scale=1.0 / np.sqrt(128.0), seed=seed)
    if name == "uniform":
        b = batch or 64
        lens = _lengths("uniform", b, rng)
        ip, ix, lpl, npg = page_table(lens, 16, seed=seed)
        return Workload(name, b, 32, 8, 128, 16, "NHD", "bf16", "bf16", "bf16", lens, ip, ix,
                        lpl, npg, layers=32, seed=seed)
    if name == "lognormal":
        b = batch or 256
        lens = _lengths("lognormal", b, rng)
        ip, ix, lpl, npg = page_table(lens, 16, seed=seed)
        return Workload(name, b, 64, 8, 128, 16, "NHD", "f16", "f16", "f16", lens, ip, ix,
                        lpl, npg, seed=seed)
    if name == "long":
        b = batch or 4
        lens = np.full(b, 131072, dtype=np.int64)
        ip, ix, lpl, npg = page_table(lens, 64, seed=seed)
        return Workload(name, b, 32, 8, 128, 64, "HND", "bf16", "bf16", "bf16", lens, ip, ix,
                        lpl, npg, fixed_split_size=256, seed=seed)
    if name == "mix":
        b = batch or 128
        lens = _lengths("mix", b, rng)
        ip, ix, lpl, npg = page_table(lens, 32, seed=seed)
        return Workload(name, b, 16, 2, 256, 32, "NHD", "bf16", "e4m3", "bf16", lens, ip, ix,
                        lpl, npg, logits_soft_cap=30.0, window_left=4096,
                        kv_store_scale=0.5, k_scale=0.5, v_scale=0.5, seed=seed)
    raise ValueError(f"unknown workload {name!r}")


def custom(kv_lens, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
           layout: str = "NHD", q_dtype: str = "f16", kv_dtype: str | None = None,
           seed: int = 0, pool_factor: float = 2.0, **kw) -> Workload:
    """A small workload with explicit lengths, for parity and edge-case tests."""
    kv_dtype = kv_dtype or q_dtype
    ip, ix, lpl, npg = page_table(kv_lens, page_size, pool_factor=pool_factor, seed=seed)
    o_dtype = kw.pop("o_dtype", q_dtype)
    return Workload("custom", len(ip) - 1, num_qo_heads, num_kv_heads, head_dim, page_size,
                    layout, q_dtype, kv_dtype, o_dtype, np.asarray(kv_lens, dtype=np.int64),
                    ip, ix, lpl, npg, seed=seed, **kw)


def pool_shape(w: Workload):
    if w.layout == "NHD":
        return (w.num_pages, 2, w.page_size, w.num_kv_heads, w.head_dim)
    return (w.num_pages, 2, w.num_kv_heads, w.page_size, w.head_dim)


def _normal(shape, device, gen):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def make_q(w: Workload, device="cpu", layer: int = 0) -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + 17 + layer)
    q = _normal((w.batch, w.num_qo_heads, w.head_dim), device, gen)
    return q.to(TORCH_DTYPES[w.q_dtype])


def _to_storage(x: torch.Tensor, w: Workload) -> torch.Tensor:
    if w.kv_dtype == "e4m3":
        x = (x / w.kv_store_scale).clamp_(-448.0, 448.0)
    return x.to(TORCH_DTYPES[w.kv_dtype])


def make_pool(w: Workload, device="cpu", layer: int = 0, chunk_pages: int = 4096) -> torch.Tensor:
    """The 5-D paged K/V pool of one layer, filled page-block by page-block with N(0,1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + 100003 + layer)
    shape = pool_shape(w)
    pool = torch.empty(shape, dtype=TORCH_DTYPES[w.kv_dtype], device=device)
    for p0 in range(0, w.num_pages, chunk_pages):
        p1 = min(w.num_pages, p0 + chunk_pages)
        pool[p0:p1] = _to_storage(_normal((p1 - p0,) + shape[1:], device, gen), w)
    return pool


def raw_bits(t: torch.Tensor) -> np.ndarray:
    """Element bit patterns of a CPU tensor as a numpy array (uint16 or uint8)."""
    t = t.contiguous().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


# ----------------------------------------------------------------------------- MLA
@dataclass
class MlaWorkload:
    """MLA paged decode (latent cache): per-request kv lengths, a CSR page table over a pool
    of pages of ``page_size`` latent rows (ckv 512 + kpe 64), ``num_heads`` query heads."""
    name: str
    batch: int
    num_heads: int
    page_size: int
    dtype: str
    kv_lens: np.ndarray     # int32 [batch]
    kv_indptr: np.ndarray   # int32 [batch + 1]
    kv_indices: np.ndarray  # int32 [kv_indptr[-1]]
    num_pages: int
    sm_scale: float
    layers: int = 1
    seed: int = 0
    head_dim_ckv: int = 512
    head_dim_kpe: int = 64


def mla_custom(kv_lens, num_heads: int, page_size: int, dtype: str = "bf16", seed: int = 0,
               pool_factor: float = 2.0, extra_pages: int = 0) -> MlaWorkload:
    """An MLA workload with explicit lengths; ``extra_pages`` gives every request that many
    unused pages past its last one (the page table may hold more pages than the length)."""
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    need = np.where(kv_lens > 0, (kv_lens + page_size - 1) // page_size, 0) + extra_pages
    indptr = np.zeros(len(kv_lens) + 1, dtype=np.int64)
    np.cumsum(need, out=indptr[1:])
    total = int(indptr[-1])
    num_pages = max(1, int(np.ceil(total * pool_factor)))
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    indices = rng.permutation(num_pages)[:total].astype(np.int32)
    return MlaWorkload("mla-custom", len(kv_lens), num_heads, page_size, dtype,
                       kv_lens.astype(np.int32), indptr.astype(np.int32), indices, num_pages,
                       sm_scale=1.0 / np.sqrt(128.0 + 64.0), seed=seed)


def mla_workload(seed: int = 0) -> MlaWorkload:
    """The MLA example of the pages' BatchMLAPagedAttentionWrapper: batch 114, 128 heads,
    kv_len 999 per request, page_size 1, bf16, sm_scale 1/sqrt(128 + 64).  Pages are the
    leading entries of a seeded permutation of a pool twice the size needed."""
    w = mla_custom([999] * 114, 128, 1, "bf16", seed=seed)
    w.name = "mla"
    return w


def make_mla_q(w: MlaWorkload, device="cpu", layer: int = 0):
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + 29 + layer)
    qn = _normal((w.batch, w.num_heads, w.head_dim_ckv), device, gen)
    qp = _normal((w.batch, w.num_heads, w.head_dim_kpe), device, gen)
    return qn.to(TORCH_DTYPES[w.dtype]), qp.to(TORCH_DTYPES[w.dtype])


def make_mla_cache(w: MlaWorkload, device="cpu", layer: int = 0):
    """ckv [pages, page_size, 512] and kpe [pages, page_size, 64], N(0, 1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + 200003 + layer)
    ckv = _normal((w.num_pages, w.page_size, w.head_dim_ckv), device, gen)
    kpe = _normal((w.num_pages, w.page_size, w.head_dim_kpe), device, gen)
    return ckv.to(TORCH_DTYPES[w.dtype]), kpe.to(TORCH_DTYPES[w.dtype])
