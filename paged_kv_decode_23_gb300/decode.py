"""Python face of libpkd: ``BatchDecodePagedKV`` with FlashInfer-style plan()/run().

Mirrors BatchDecodeWithPagedKVCacheWrapper from the FlashInfer attention API page
(constructor with a float workspace and a KV layout; plan(indptr, indices, last_page_len,
num_qo_heads, num_kv_heads, head_dim, page_size, ...); run(q, paged_kv_cache, q_scale,
k_scale, v_scale, out, lse, return_lse)).  This module only checks shapes and marshals
pointers: every step of the computation runs in libpkd's CUDA kernels.  PyTorch supplies
device memory and the current stream.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple, Union

import numpy as np
import torch

from . import _lib as L

_DTYPE_CODE = {torch.float16: L.DTYPE_F16, torch.bfloat16: L.DTYPE_BF16,
               torch.float8_e4m3fn: L.DTYPE_E4M3}
_STR_DTYPE = {"float16": torch.float16, "half": torch.float16, "bfloat16": torch.bfloat16,
              "float8_e4m3fn": torch.float8_e4m3fn, "e4m3": torch.float8_e4m3fn}


def _as_dtype(x):
    if x is None or isinstance(x, torch.dtype):
        return x
    return _STR_DTYPE[str(x).replace("torch.", "")]


def _host_i32(t) -> np.ndarray:
    """A contiguous host int32 array of `t` (no copy when it already is one)."""
    if isinstance(t, torch.Tensor):
        if t.device.type != "cpu":
            t = t.to("cpu")
        a = t.detach().numpy()
    else:
        a = np.asarray(t)
    if a.dtype != np.int32 or not a.flags.c_contiguous:
        a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _i32p(a: np.ndarray) -> int:
    """The address of a contiguous int32 array, for a pointer argument of the C ABI."""
    return a.ctypes.data


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_POS_CODE = {"NONE": 0, "ROPE_LLAMA": 1, "ALIBI": 2}


def _graph_buffer(t, name: str, need: int) -> torch.Tensor:
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
            and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
    if t.numel() < need:
        raise ValueError(f"{name} holds {t.numel()} entries, needs at least {need}")
    return t


class BatchDecodePagedKV:
    """Batch decode attention over a paged KV cache (one query token per request and head).

    ``float_workspace_buffer``: a CUDA uint8 tensor for split-KV partials (128 MiB is the
    usual size).  ``int_workspace_buffer``: CUDA uint8 tensor for the work list (allocated
    here, 8 MiB, if not given).  ``kv_layout``: "NHD" or "HND".

    ``use_cuda_graph=True`` (with the three ``paged_kv_*_buffer`` device int32 tensors: indptr
    ``[max_batch + 1]``, indices ``[max_pages]``, last_page_len ``[max_batch]``) makes ``run``
    capturable in a CUDA graph whose replays stay valid across later ``plan`` calls: ``plan``
    copies the page table into those buffers, the batch size is fixed by the first plan (pad
    with zero-length requests), and the work list holds at most ``max_items`` chunks
    (default: max_batch + 2 x the SM count).

    ``use_tensor_cores``: None (auto: the tensor-core kernel, measured at least as fast at
    every GQA group), True, or False (the fp32 CUDA-core kernel); ``plan`` may override it.
    """

    def __init__(self, float_workspace_buffer: torch.Tensor, kv_layout: str = "NHD",
                 use_cuda_graph: bool = False, use_tensor_cores: Optional[bool] = None,
                 paged_kv_indptr_buffer: Optional[torch.Tensor] = None,
                 paged_kv_indices_buffer: Optional[torch.Tensor] = None,
                 paged_kv_last_page_len_buffer: Optional[torch.Tensor] = None,
                 int_workspace_buffer: Optional[torch.Tensor] = None,
                 max_items: Optional[int] = None, backend: str = "auto",
                 jit_args: Optional[list] = None):
        if kv_layout not in ("NHD", "HND"):
            raise ValueError("kv_layout must be 'NHD' or 'HND'")
        # the page's backends name other libraries' kernels; this library has one of its own
        if backend not in ("auto", "fa2"):
            raise NotImplementedError(f"backend {backend!r} is not built (auto / fa2 run this "
                                      "library's kernels)")
        if jit_args is not None:
            raise NotImplementedError("JIT variants are not built")
        if not float_workspace_buffer.is_cuda:
            raise ValueError("the float workspace must be a CUDA tensor")
        if int_workspace_buffer is None:
            int_workspace_buffer = torch.empty(8 << 20, dtype=torch.uint8,
                                               device=float_workspace_buffer.device)
        self.kv_layout = kv_layout
        self._use_tc = use_tensor_cores
        self._float_ws = float_workspace_buffer
        self._int_ws = int_workspace_buffer
        self._plan_args = None
        self._indices = None
        self.use_cuda_graph = bool(use_cuda_graph)
        h = ctypes.c_void_p()
        L.check(L.lib().pkd_create(ctypes.byref(h), self._float_ws.data_ptr(),
                                   self._float_ws.numel() * self._float_ws.element_size(),
                                   self._int_ws.data_ptr(),
                                   self._int_ws.numel() * self._int_ws.element_size(),
                                   L.LAYOUT_NHD if kv_layout == "NHD" else L.LAYOUT_HND))
        self._h = h
        if self.use_cuda_graph:
            lpl = paged_kv_last_page_len_buffer
            if lpl is None or paged_kv_indptr_buffer is None or paged_kv_indices_buffer is None:
                raise ValueError("use_cuda_graph=True needs paged_kv_indptr_buffer, "
                                 "paged_kv_indices_buffer and paged_kv_last_page_len_buffer")
            max_batch = _graph_buffer(lpl, "paged_kv_last_page_len_buffer", 1).numel()
            ip = _graph_buffer(paged_kv_indptr_buffer, "paged_kv_indptr_buffer", max_batch + 1)
            ix = _graph_buffer(paged_kv_indices_buffer, "paged_kv_indices_buffer", 0)
            self._graph_buffers = (ip, ix, lpl)
            L.check(L.lib().pkd_enable_cuda_graph(self._h, ip.data_ptr(), ix.data_ptr(),
                                                  lpl.data_ptr(), max_batch, ix.numel(),
                                                  int(max_items or 0)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                L.lib().pkd_destroy(h)
            except Exception:
                pass
            self._h = None

    def reset_workspace_buffer(self, float_workspace_buffer: torch.Tensor,
                               int_workspace_buffer: torch.Tensor) -> None:
        L.check(L.lib().pkd_reset_workspace(
            self._h, float_workspace_buffer.data_ptr(),
            float_workspace_buffer.numel() * float_workspace_buffer.element_size(),
            int_workspace_buffer.data_ptr(),
            int_workspace_buffer.numel() * int_workspace_buffer.element_size()))
        self._float_ws, self._int_ws = float_workspace_buffer, int_workspace_buffer
        self._plan_args = None

    # ------------------------------------------------------------------ plan
    def plan(self, indptr, indices: torch.Tensor, last_page_len, num_qo_heads: int,
             num_kv_heads: int, head_dim: int, page_size: int, pos_encoding_mode: str = "NONE",
             window_left: int = -1, logits_soft_cap: Optional[float] = None,
             q_data_type=torch.float16, kv_data_type=None, o_data_type=None, data_type=None,
             sm_scale: Optional[float] = None, non_blocking: bool = True,
             fixed_split_size: Optional[int] = None, disable_split_kv: bool = False,
             use_tensor_cores: Optional[bool] = None, stream=None,
             q_len_per_req: int = 1, rope_scale: Optional[float] = None,
             rope_theta: Optional[float] = None, block_tables: Optional[torch.Tensor] = None,
             seq_lens: Optional[torch.Tensor] = None) -> None:
        """Plan a batch; ``indptr`` / ``last_page_len`` may live on the host or the device
        (a device copy is read back once here), ``indices`` must be a CUDA int32 tensor and
        stay unchanged while runs of this plan are in flight.  ``q_len_per_req`` query tokens
        per request (run's parameter of that name; the work list depends on it, so it is fixed
        here): the request's last positions, each attending causally; q / o then have
        ``batch * q_len_per_req`` rows, request-major.  ``pos_encoding_mode``: "NONE",
        "ROPE_LLAMA" (with ``rope_scale`` / ``rope_theta``, defaults 1 and 1e4) or
        "ALIBI"."""
        if block_tables is not None or seq_lens is not None:
            raise NotImplementedError("block_tables / seq_lens (the trtllm-gen backend's page "
                                      "table form) are not built; pass indptr / indices / "
                                      "last_page_len")
        pos_code = _POS_CODE.get(pos_encoding_mode)
        if pos_code is None:
            raise ValueError("pos_encoding_mode must be 'NONE', 'ROPE_LLAMA' or 'ALIBI'")
        if data_type is not None:
            q_data_type = data_type
        q_dt = _as_dtype(q_data_type)
        kv_dt = _as_dtype(kv_data_type) or q_dt
        o_dt = _as_dtype(o_data_type) or q_dt
        if not (isinstance(indices, torch.Tensor) and indices.is_cuda
                and indices.dtype == torch.int32 and indices.is_contiguous()):
            raise ValueError("indices must be a contiguous CUDA int32 tensor")
        ip = _host_i32(indptr)
        lpl = _host_i32(last_page_len)
        batch = len(lpl)
        if len(ip) != batch + 1:
            raise ValueError("indptr must have batch + 1 entries")
        utc = use_tensor_cores if use_tensor_cores is not None else self._use_tc
        kernel = L.KERNEL_AUTO if utc is None else (L.KERNEL_TENSOR_CORE if utc else L.KERNEL_CUDA_CORE)
        sm = float("nan") if sm_scale is None else float(sm_scale)
        L.check(L.lib().pkd_plan(
            self._h, _i32p(ip), _i32p(lpl), batch, indices.data_ptr(), indices.numel(),
            num_qo_heads, num_kv_heads, head_dim, page_size, sm,
            float(logits_soft_cap or 0.0), int(window_left), int(fixed_split_size or 0),
            int(bool(disable_split_kv)), _DTYPE_CODE[q_dt], _DTYPE_CODE[kv_dt], _DTYPE_CODE[o_dt],
            kernel, int(q_len_per_req), pos_code,
            1.0 if rope_scale is None else float(rope_scale),
            1e4 if rope_theta is None else float(rope_theta), _stream_ptr(stream)))
        self._indices = indices
        self._plan_args = dict(batch=batch, q_len=int(q_len_per_req),
                               num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                               head_dim=head_dim, page_size=page_size, q_dtype=q_dt,
                               kv_dtype=kv_dt, o_dtype=o_dt)

    # ------------------------------------------------------------------ run
    def _kv_pointers(self, paged_kv_cache):
        a = self._plan_args
        if isinstance(paged_kv_cache, (tuple, list)):
            k, v = paged_kv_cache
            if k.dim() != 4 or v.dim() != 4 or k.shape != v.shape or k.stride() != v.stride():
                raise ValueError("(k_cache, v_cache) must be 4-D tensors of one shape and stride")
            if self.kv_layout == "NHD":
                exp = (a["page_size"], a["num_kv_heads"], a["head_dim"])
                strides = (k.stride(0), k.stride(1), k.stride(2))
            else:
                exp = (a["num_kv_heads"], a["page_size"], a["head_dim"])
                strides = (k.stride(0), k.stride(2), k.stride(1))
            if tuple(k.shape[1:]) != exp or k.stride(3) != 1:
                raise ValueError(f"k/v cache shape {tuple(k.shape)} does not match the plan")
            return k, k.data_ptr(), v.data_ptr(), k.shape[0], strides
        kv = paged_kv_cache
        if kv.dim() != 5 or kv.shape[1] != 2 or kv.stride(4) != 1:
            raise ValueError("paged_kv_cache must be [pages, 2, ...] with head_dim contiguous")
        if self.kv_layout == "NHD":
            exp = (a["page_size"], a["num_kv_heads"], a["head_dim"])
            strides = (kv.stride(0), kv.stride(2), kv.stride(3))
        else:
            exp = (a["num_kv_heads"], a["page_size"], a["head_dim"])
            strides = (kv.stride(0), kv.stride(3), kv.stride(2))
        if tuple(kv.shape[2:]) != exp:
            raise ValueError(f"paged_kv_cache shape {tuple(kv.shape)} does not match the plan")
        base = kv.data_ptr()
        return kv, base, base + kv.stride(1) * kv.element_size(), kv.shape[0], strides

    def run(self, q: torch.Tensor, paged_kv_cache: Union[torch.Tensor, Tuple[torch.Tensor, torch.Tensor]],
            q_scale: Optional[float] = None, k_scale: Optional[float] = None,
            v_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, return_lse: bool = False, stream=None,
            timing_events=None, enable_pdl: Optional[bool] = None,
            q_len_per_req: Optional[int] = None):
        """Decode attention for the planned batch on one layer's pool: returns ``o`` or
        ``(o, lse)`` (lse: float32 natural log, ``[batch, num_qo_heads]``).  ``enable_pdl``
        switches programmatic dependent launch for this and later runs (on by default)."""
        a = self._plan_args
        if a is None:
            raise RuntimeError("plan() must be called before run()")
        if q_len_per_req is not None and int(q_len_per_req) != a["q_len"]:
            raise ValueError(f"q_len_per_req={q_len_per_req} differs from the plan's "
                             f"{a['q_len']} (the work list depends on it: re-plan)")
        exp_q = (a["batch"] * a["q_len"], a["num_qo_heads"], a["head_dim"])
        if tuple(q.shape) != exp_q or q.dtype != a["q_dtype"] or not q.is_contiguous():
            raise ValueError(f"q must be a contiguous {a['q_dtype']} tensor of shape {exp_q}")
        kv, k_ptr, v_ptr, num_pages, strides = self._kv_pointers(paged_kv_cache)
        if kv.dtype != a["kv_dtype"]:
            raise ValueError(f"KV dtype {kv.dtype} does not match the plan ({a['kv_dtype']})")
        if out is None:
            out = torch.empty(exp_q, dtype=a["o_dtype"], device=q.device)
        elif tuple(out.shape) != exp_q or out.dtype != a["o_dtype"] or not out.is_contiguous():
            raise ValueError("out has the wrong shape, dtype or layout")
        if lse is None and return_lse:
            lse = torch.empty(exp_q[:2], dtype=torch.float32, device=q.device)
        if lse is not None and (tuple(lse.shape) != exp_q[:2] or lse.dtype != torch.float32):
            raise ValueError("lse must be float32 [batch * q_len_per_req, num_qo_heads]")
        st = (ctypes.c_int64 * 3)(*strides)
        if enable_pdl is not None:
            L.check(L.lib().pkd_set_pdl(self._h, int(bool(enable_pdl))))
        ev0, ev1 = timing_events if timing_events is not None else (None, None)
        L.check(L.lib().pkd_run_timed(
            self._h, q.data_ptr(), k_ptr, v_ptr, num_pages, st,
            1.0 if q_scale is None else float(q_scale), 1.0 if k_scale is None else float(k_scale),
            1.0 if v_scale is None else float(v_scale), out.data_ptr(),
            lse.data_ptr() if lse is not None else None, _stream_ptr(stream),
            ev0.cuda_event if ev0 is not None else None,
            ev1.cuda_event if ev1 is not None else None))
        return (out, lse) if return_lse else out

    def run_return_lse(self, q: torch.Tensor, paged_kv_cache, *args, **kw):
        """``run(..., return_lse=True)``: returns ``(o, lse)``."""
        kw["return_lse"] = True
        return self.run(q, paged_kv_cache, *args, **kw)

    def check_status(self, stream=None) -> int:
        """Read and clear the device status word (synchronises the stream); 0 = no error,
        else STATUS_TIMEOUT / STATUS_BAD_PAGE bits (include/pkd.h, pkd_check_status)."""
        v = ctypes.c_uint32()
        L.check(L.lib().pkd_check_status(self._h, ctypes.byref(v), _stream_ptr(stream)))
        return v.value

    def plan_info(self) -> dict:
        """The current plan's launch shape: grid (CTAs per launch), ctas_per_sm, tasks, merges."""
        g, c = ctypes.c_int(), ctypes.c_int()
        t, m = ctypes.c_int64(), ctypes.c_int64()
        L.check(L.lib().pkd_plan_info(self._h, ctypes.byref(g), ctypes.byref(c), ctypes.byref(t),
                                      ctypes.byref(m)))
        return dict(grid=g.value, ctas_per_sm=c.value, tasks=t.value, merges=m.value)

    def set_wait_limit(self, limit_ns: int) -> None:
        """Limit of the decode kernel's pipeline waits for later runs, in ns (default and
        maximum 2e9); a wait that runs out sets STATUS_TIMEOUT and its CTA gives up."""
        L.check(L.lib().pkd_set_wait_limit(self._h, int(limit_ns)))


def check_page_table(indptr, indices, num_pages: int) -> None:
    """Host validation of a page table (pkd_check_page_table): raises PkdError
    (PKD_ERR_INVALID_ARG) naming the first request whose page id lies outside
    [0, num_pages).  Device tensors are copied to the host first."""
    ip = _host_i32(indptr)
    ix = _host_i32(indices) if len(indices) else np.zeros(1, dtype=np.int32)
    L.check(L.lib().pkd_check_page_table(_i32p(ip), len(ip) - 1, _i32p(ix), len(indices),
                                         int(num_pages)))


def noalloc_check_status(stream=None) -> int:
    """Read and clear the status word of pkd_decode_noalloc's built-in scratch on the current
    device (pkd_check_status with a null handle); 0 = the last call reported nothing."""
    v = ctypes.c_uint32()
    L.check(L.lib().pkd_check_status(None, ctypes.byref(v), _stream_ptr(stream)))
    return v.value


def plan_host(indptr, last_page_len, num_qo_heads: int, num_kv_heads: int, head_dim: int,
              page_size: int, window_left: int = -1, fixed_split_size: int = 0,
              disable_split_kv: bool = False, kv_dtype: int = L.DTYPE_F16,
              use_tensor_cores: int = L.KERNEL_AUTO, num_sms: int = 152,
              work_capacity: int = 0, q_len_per_req: int = 1):
    """Run the decode planner alone (no GPU): returns a dict with the tasks ``[n, 12]``
    (row, first page index, chunk start, begin, end, slot, merge entry, query position,
    kv head, slice, CTA, 0) grouped by CTA, the merge entries ``[m, 4]`` (row, first slot,
    chunk count, unit), the slot count, the CTAs with work, the chosen kernel and the tile
    size.  ``work_capacity`` > 0 bounds the work list as CUDA-graph mode does."""
    ip = _host_i32(indptr)
    lpl = _host_i32(last_page_len)
    batch = len(lpl)
    n_tasks, n_merges, n_slots = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    kern, tile, n_ctas = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    args = (_i32p(ip), _i32p(lpl), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
            window_left, fixed_split_size, int(disable_split_kv), kv_dtype, use_tensor_cores,
            num_sms)
    L.check(L.lib().pkd_plan_host(*args, None, 0, None, 0, ctypes.byref(n_tasks),
                                  ctypes.byref(n_merges), ctypes.byref(n_slots),
                                  ctypes.byref(kern), ctypes.byref(tile), int(work_capacity),
                                  int(q_len_per_req), ctypes.byref(n_ctas)))
    tasks = np.zeros((max(1, n_tasks.value), 12), dtype=np.int32)
    merges = np.zeros((max(1, n_merges.value), 4), dtype=np.int32)
    L.check(L.lib().pkd_plan_host(*args, _i32p(tasks), n_tasks.value, _i32p(merges),
                                  n_merges.value, ctypes.byref(n_tasks), ctypes.byref(n_merges),
                                  ctypes.byref(n_slots), ctypes.byref(kern), ctypes.byref(tile),
                                  int(work_capacity), int(q_len_per_req), ctypes.byref(n_ctas)))
    return dict(tasks=tasks[:n_tasks.value], merges=merges[:n_merges.value],
                num_slots=n_slots.value, num_ctas=n_ctas.value, kernel=kern.value,
                tile_tokens=tile.value)


def mla_graph_workspace_bytes(max_items: int, num_heads: int, backend: str = "auto"):
    """(float, int) workspace bytes BatchMLAPagedAttention needs in CUDA-graph mode for a work
    list of max_items chunks."""
    if backend not in _MLA_BACKEND:
        raise ValueError(f"backend must be one of {sorted(_MLA_BACKEND)}")
    fb, ib = ctypes.c_size_t(), ctypes.c_size_t()
    L.check(L.lib().pkd_mla_graph_workspace_bytes(int(max_items), num_heads,
                                                  _MLA_BACKEND[backend], ctypes.byref(fb),
                                                  ctypes.byref(ib)))
    return fb.value, ib.value


def mla_plan_host(kv_indptr, kv_len_arr, num_heads: int, page_size: int,
                  dtype: int = L.DTYPE_BF16, backend: str = "auto", num_sms: int = 152):
    """The MLA work list ``BatchMLAPagedAttention.plan`` would upload, built on the host alone
    (no GPU): items ``[n, 8]`` (row, first page index, chunk start, begin, end, slot, merge
    entry, query position), merge entries ``[m, 4]``, slot count, CTAs per item and the
    float / int workspace bytes the plan needs."""
    if backend not in _MLA_BACKEND:
        raise ValueError(f"backend must be one of {sorted(_MLA_BACKEND)}")
    ip = _host_i32(kv_indptr)
    kl = _host_i32(kv_len_arr)
    batch = len(kl)
    n_items, n_merges, n_slots, cpi = (ctypes.c_int() for _ in range(4))
    fb, ib = ctypes.c_size_t(), ctypes.c_size_t()
    args = (_i32p(ip), _i32p(kl), batch, num_heads, page_size, dtype, _MLA_BACKEND[backend],
            num_sms)
    outs = (ctypes.byref(n_items), ctypes.byref(n_merges), ctypes.byref(n_slots),
            ctypes.byref(cpi), ctypes.byref(fb), ctypes.byref(ib))
    L.check(L.lib().pkd_mla_plan_host(*args, None, 0, None, 0, *outs))
    items = np.zeros((max(1, n_items.value), 8), dtype=np.int32)
    merges = np.zeros((max(1, n_merges.value), 4), dtype=np.int32)
    L.check(L.lib().pkd_mla_plan_host(*args, _i32p(items), n_items.value, _i32p(merges),
                                      n_merges.value, *outs))
    return dict(items=items[:n_items.value], merges=merges[:n_merges.value],
                num_slots=n_slots.value, ctas_per_item=cpi.value, float_ws_bytes=fb.value,
                int_ws_bytes=ib.value)


def workspace_bytes(indptr, last_page_len, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                    page_size: int, window_left: int = -1, fixed_split_size: int = 0,
                    disable_split_kv: bool = False, kv_dtype: int = L.DTYPE_F16,
                    use_tensor_cores: int = L.KERNEL_AUTO, num_sms: int = 152,
                    q_len_per_req: int = 1):
    ip = _host_i32(indptr)
    lpl = _host_i32(last_page_len)
    fb, ib = ctypes.c_size_t(), ctypes.c_size_t()
    L.check(L.lib().pkd_workspace_bytes(_i32p(ip), _i32p(lpl), len(lpl), num_qo_heads,
                                        num_kv_heads, head_dim, page_size, window_left,
                                        fixed_split_size, int(disable_split_kv), kv_dtype,
                                        use_tensor_cores, num_sms, int(q_len_per_req),
                                        ctypes.byref(fb), ctypes.byref(ib)))
    return fb.value, ib.value


def graph_workspace_bytes(max_items: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                          use_tensor_cores: int = L.KERNEL_AUTO):
    """(float, int) workspace bytes that CUDA-graph mode needs for ``max_items`` chunks."""
    fb, ib = ctypes.c_size_t(), ctypes.c_size_t()
    L.check(L.lib().pkd_graph_workspace_bytes(int(max_items), num_qo_heads, num_kv_heads,
                                              head_dim, use_tensor_cores, ctypes.byref(fb),
                                              ctypes.byref(ib)))
    return fb.value, ib.value


class CUDAGraphBatchDecodePagedKV(BatchDecodePagedKV):
    """The pages' CUDAGraphBatchDecodeWithPagedKVCacheWrapper: BatchDecodePagedKV in CUDA-graph
    mode with the page-table buffers given up front (``indptr_buffer [max_batch + 1]``,
    ``indices_buffer [max_pages]``, ``last_page_len_buffer [max_batch]``, device int32)."""

    def __init__(self, workspace_buffer: torch.Tensor, indptr_buffer: torch.Tensor,
                 indices_buffer: torch.Tensor, last_page_len_buffer: torch.Tensor,
                 kv_layout: str = "NHD", use_tensor_cores: Optional[bool] = None,
                 int_workspace_buffer: Optional[torch.Tensor] = None,
                 max_items: Optional[int] = None):
        super().__init__(workspace_buffer, kv_layout, use_cuda_graph=True,
                         use_tensor_cores=use_tensor_cores,
                         paged_kv_indptr_buffer=indptr_buffer,
                         paged_kv_indices_buffer=indices_buffer,
                         paged_kv_last_page_len_buffer=last_page_len_buffer,
                         int_workspace_buffer=int_workspace_buffer, max_items=max_items)


_MLA_BACKEND = {"auto": 0, "fa2": 1, "tcgen05": 2}


class BatchMLAPagedAttention:
    """MLA paged decode (the pages' BatchMLAPagedAttentionWrapper): every query head attends
    over one latent cache; key = [ckv, kpe] (512 + 64), value = ckv.  Decode only: every
    query length in ``qo_indptr`` must be 1.

    ``backend``: "auto" (the tcgen05 kernel for more than 32 heads, else "fa2"), "fa2" (32
    heads per CTA on mma.sync with register accumulators) or "tcgen05" (128 heads per 2-CTA
    cluster on the 5th-generation tensor cores, accumulators in tensor memory).

    ``use_cuda_graph=True`` with the device int32 buffers ``qo_indptr`` / ``kv_indptr``
    ``[max_batch + 1]``, ``kv_indices`` ``[max_pages]`` and ``kv_len_arr`` ``[max_batch]``
    makes ``run`` capturable in a CUDA graph whose replays stay valid across later ``plan``
    calls: ``plan`` copies the page table into those buffers; the first plan fixes the batch
    size (pad with zero-length requests), the head count, page size, sm_scale and dtype; the
    work list holds at most ``max_items`` chunks (default: max_batch + the SM count)."""

    def __init__(self, float_workspace_buffer: torch.Tensor, use_cuda_graph: bool = False,
                 qo_indptr: Optional[torch.Tensor] = None,
                 kv_indptr: Optional[torch.Tensor] = None,
                 kv_indices: Optional[torch.Tensor] = None,
                 kv_len_arr: Optional[torch.Tensor] = None, backend: str = "auto",
                 int_workspace_buffer: Optional[torch.Tensor] = None,
                 max_items: Optional[int] = None):
        if backend not in _MLA_BACKEND:
            raise ValueError(f"backend must be one of {sorted(_MLA_BACKEND)}")
        if not float_workspace_buffer.is_cuda:
            raise ValueError("the float workspace must be a CUDA tensor")
        if int_workspace_buffer is None:
            int_workspace_buffer = torch.empty(8 << 20, dtype=torch.uint8,
                                               device=float_workspace_buffer.device)
        self._float_ws = float_workspace_buffer
        self._int_ws = int_workspace_buffer
        self._plan_args = None
        self.use_cuda_graph = bool(use_cuda_graph)
        h = ctypes.c_void_p()
        L.check(L.lib().pkd_create(ctypes.byref(h), self._float_ws.data_ptr(),
                                   self._float_ws.numel() * self._float_ws.element_size(),
                                   self._int_ws.data_ptr(),
                                   self._int_ws.numel() * self._int_ws.element_size(),
                                   L.LAYOUT_NHD))
        self._h = h
        L.check(L.lib().pkd_mla_set_backend(h, _MLA_BACKEND[backend]))
        if self.use_cuda_graph:
            if kv_indptr is None or kv_indices is None or kv_len_arr is None:
                raise ValueError("use_cuda_graph=True needs kv_indptr, kv_indices and kv_len_arr "
                                 "buffers")
            lens = _graph_buffer(kv_len_arr, "kv_len_arr", 1)
            max_batch = lens.numel()
            ip = _graph_buffer(kv_indptr, "kv_indptr", max_batch + 1)
            ix = _graph_buffer(kv_indices, "kv_indices", 0)
            qo = _graph_buffer(qo_indptr, "qo_indptr", max_batch + 1) if qo_indptr is not None \
                else None
            self._graph_buffers = (qo, ip, ix, lens)
            if max_items is None:
                props = torch.cuda.get_device_properties(float_workspace_buffer.device)
                max_items = max_batch + props.multi_processor_count
            L.check(L.lib().pkd_enable_cuda_graph(self._h, ip.data_ptr(), ix.data_ptr(),
                                                  lens.data_ptr(), max_batch, ix.numel(),
                                                  int(max_items)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                L.lib().pkd_destroy(h)
            except Exception:
                pass
            self._h = None

    def plan(self, qo_indptr, kv_indptr, kv_indices: torch.Tensor, kv_len_arr, num_heads: int,
             head_dim_ckv: int, head_dim_kpe: int, page_size: int, causal: bool, sm_scale: float,
             q_data_type=torch.bfloat16, kv_data_type=None, use_profiler: bool = False,
             stream=None) -> None:
        q_ip = _host_i32(qo_indptr)
        kv_ip = _host_i32(kv_indptr)
        kv_len = _host_i32(kv_len_arr)
        batch = len(kv_len)
        if len(kv_ip) != batch + 1 or len(q_ip) != batch + 1:
            raise ValueError("qo_indptr and kv_indptr must have batch + 1 entries")
        if not np.array_equal(np.diff(q_ip), np.ones(batch, dtype=np.int32)):
            raise NotImplementedError("only decode (one query per request) is built for MLA")
        if use_profiler:
            raise NotImplementedError("the in-kernel profiler is not built")
        if not (isinstance(kv_indices, torch.Tensor) and kv_indices.is_cuda
                and kv_indices.dtype == torch.int32 and kv_indices.is_contiguous()):
            raise ValueError("kv_indices must be a contiguous CUDA int32 tensor")
        q_dt = _as_dtype(q_data_type)
        kv_dt = _as_dtype(kv_data_type) or q_dt
        L.check(L.lib().pkd_mla_plan(
            self._h, _i32p(kv_ip), _i32p(kv_len), batch, kv_indices.data_ptr(),
            kv_indices.numel(), num_heads, head_dim_ckv, head_dim_kpe, page_size,
            int(bool(causal)), float(sm_scale), _DTYPE_CODE[q_dt], _DTYPE_CODE[kv_dt],
            _stream_ptr(stream)))
        if self.use_cuda_graph and self._graph_buffers[0] is not None:
            # the qo_indptr buffer holds 0, 1, ..., batch like the page's wrapper (no kernel
            # reads it: one query per request)
            self._graph_buffers[0][:batch + 1].copy_(torch.from_numpy(q_ip), non_blocking=True)
        self._indices = kv_indices
        self._plan_args = dict(batch=batch, num_heads=num_heads, page_size=page_size, dtype=q_dt)

    def run(self, q_nope: torch.Tensor, q_pe: torch.Tensor, ckv_cache: torch.Tensor,
            kpe_cache: torch.Tensor, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, return_lse: bool = False,
            profiler_buffer: Optional[torch.Tensor] = None, kv_len: Optional[torch.Tensor] = None,
            page_table: Optional[torch.Tensor] = None, return_lse_base_on_e: bool = False,
            stream=None, timing_events=None, enable_pdl: Optional[bool] = None):
        """The page's run(): ``kv_len`` and ``page_table`` belong to the cutlass backend, which is
        not built (the plan's lengths and page ids are used), and no profiler is built, so
        all three must be None."""
        if profiler_buffer is not None:
            raise NotImplementedError("no profiler is built (plan with use_profiler=False)")
        if kv_len is not None or page_table is not None:
            raise NotImplementedError("kv_len / page_table are the cutlass backend's run() "
                                      "arguments; that backend is not built")
        a = self._plan_args
        if a is None:
            raise RuntimeError("plan() must be called before run()")
        B, H, dt = a["batch"], a["num_heads"], a["dtype"]
        for name, t, shape in (("q_nope", q_nope, (B, H, 512)), ("q_pe", q_pe, (B, H, 64))):
            if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shape}")
        ps = a["page_size"]
        if (ckv_cache.dim() != 3 or tuple(ckv_cache.shape[1:]) != (ps, 512)
                or ckv_cache.dtype != dt or not ckv_cache.is_contiguous()):
            raise ValueError(f"ckv_cache must be a contiguous {dt} [pages, {ps}, 512] tensor")
        if (tuple(kpe_cache.shape) != (ckv_cache.shape[0], ps, 64) or kpe_cache.dtype != dt
                or not kpe_cache.is_contiguous()):
            raise ValueError(f"kpe_cache must be a contiguous {dt} [pages, {ps}, 64] tensor")
        if out is None:
            out = torch.empty((B, H, 512), dtype=dt, device=q_nope.device)
        if lse is None and return_lse:
            lse = torch.empty((B, H), dtype=torch.float32, device=q_nope.device)
        if enable_pdl is not None:
            L.check(L.lib().pkd_set_pdl(self._h, int(bool(enable_pdl))))
        ev0, ev1 = timing_events if timing_events is not None else (None, None)
        L.check(L.lib().pkd_mla_run(
            self._h, q_nope.data_ptr(), q_pe.data_ptr(), ckv_cache.data_ptr(),
            kpe_cache.data_ptr(), ckv_cache.shape[0], out.data_ptr(),
            lse.data_ptr() if lse is not None else None, int(bool(return_lse_base_on_e)),
            _stream_ptr(stream), ev0.cuda_event if ev0 is not None else None,
            ev1.cuda_event if ev1 is not None else None))
        return (out, lse) if return_lse else out

    def check_status(self, stream=None) -> int:
        v = ctypes.c_uint32()
        L.check(L.lib().pkd_check_status(self._h, ctypes.byref(v), _stream_ptr(stream)))
        return v.value
