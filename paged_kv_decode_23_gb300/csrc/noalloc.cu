// noalloc.cu -- pkd_decode_noalloc: plan + run with scratch built into the library.
//
// For callers that may not allocate device memory and have no workspace to lend (a runtime
// that owns every allocation through its own pool or budget).  The scratch they would have
// passed -- status word, work list, split partials -- lives in one file-scope device array.
// The plan is built in static host storage, so a call allocates nothing.  The kernels are the
// tensor-core decode and merge_states kernels of the rest of the library, instantiated here
// with the same parameters.
//
// The array is shared by every call in the process: calls whose GPU work overlaps race.
#include "../../include/pkd.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <mutex>

#include "decode_kernels.cuh"
#include "merge_kernel.cuh"

namespace pkd {
void set_error_message(const char* msg);  // pkd_api.cpp: what pkd_last_error() returns
}

using namespace pkd;

// One array per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char pkd_noalloc_scratch[PKD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNaItemsOff = kStatusBytes;                           // work list
constexpr size_t kNaMergesOff = kNaItemsOff + PKD_NOALLOC_MAX_ITEMS * sizeof(WorkItem);
constexpr size_t kNaFloatOff = (1u << 20) + 512u;                      // split partials
static_assert(kNaMergesOff + PKD_NOALLOC_MAX_MERGES * sizeof(MergeEntry) <= kNaFloatOff,
              "work list region overlaps the partials");
static_assert(kNaFloatOff + PKD_NOALLOC_PARTIAL_BYTES == PKD_NOALLOC_SCRATCH_BYTES,
              "partials region ends at the end of the array");

struct NaDecode {
  int q_dtype, kv_dtype, head_dim;
  const void* fn;
  int threads, smem, tile;
};

#define PKD_NA_DEC(TQ, FP8, D, TS, NS, QC, KC)                                              \
  NaDecode {                                                                                \
    QC, KC, D, reinterpret_cast<const void*>(&decode_paged_kernel<TQ, FP8, D, TS, NS, kTensorCore, 8>), \
        DecodeGeom<TQ, FP8, D, TS, NS>::THREADS, DecodeGeom<TQ, FP8, D, TS, NS>::SMEM_BYTES, TS \
  }

// The tensor-core kernels of decode_f16.cu / decode_bf16.cu / decode_e4m3.cu.
const NaDecode kNaDecode[] = {
    PKD_NA_DEC(__half, false, 64, 128, 3, kF16, kF16),
    PKD_NA_DEC(__half, false, 128, 64, 3, kF16, kF16),
    PKD_NA_DEC(__half, false, 256, 32, 3, kF16, kF16),
    PKD_NA_DEC(__nv_bfloat16, false, 64, 128, 3, kBF16, kBF16),
    PKD_NA_DEC(__nv_bfloat16, false, 128, 64, 3, kBF16, kBF16),
    PKD_NA_DEC(__nv_bfloat16, false, 256, 32, 3, kBF16, kBF16),
    PKD_NA_DEC(__half, true, 128, 128, 3, kF16, kE4M3),
    PKD_NA_DEC(__half, true, 256, 64, 3, kF16, kE4M3),
    PKD_NA_DEC(__nv_bfloat16, true, 128, 128, 3, kBF16, kE4M3),
    PKD_NA_DEC(__nv_bfloat16, true, 256, 64, 3, kBF16, kE4M3),
};
#undef PKD_NA_DEC

struct NaMerge {
  int o_dtype, head_dim;
  const void* fn;
};
const NaMerge kNaMerge[] = {
    {kF16, 64, reinterpret_cast<const void*>(&merge_states_kernel<__half, 64>)},
    {kF16, 128, reinterpret_cast<const void*>(&merge_states_kernel<__half, 128>)},
    {kF16, 256, reinterpret_cast<const void*>(&merge_states_kernel<__half, 256>)},
    {kBF16, 64, reinterpret_cast<const void*>(&merge_states_kernel<__nv_bfloat16, 64>)},
    {kBF16, 128, reinterpret_cast<const void*>(&merge_states_kernel<__nv_bfloat16, 128>)},
    {kBF16, 256, reinterpret_cast<const void*>(&merge_states_kernel<__nv_bfloat16, 256>)},
};

// ---------------------------------------------------------------- per-device set-up
constexpr int kMaxDevices = 64;
std::mutex g_na_mutex;  // guards the set-up table and the static host plan below
bool g_na_ready[kMaxDevices];
unsigned char* g_na_scratch[kMaxDevices];
int g_na_sms[kMaxDevices];

int na_fail(int code, const char* msg) {
  set_error_message(msg);
  return code;
}

// Runs with the device current.  Returns PKD_OK or an error code.
int na_setup(int dev) {
  if (g_na_ready[dev]) return PKD_OK;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, pkd_noalloc_scratch) != cudaSuccess || !ptr)
    return na_fail(PKD_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch array failed");
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "cudaDeviceGetAttribute(multiProcessorCount) failed");
  for (const NaDecode& k : kNaDecode)
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) !=
        cudaSuccess)
      return na_fail(PKD_ERR_CUDA, "cudaFuncSetAttribute on a decode kernel failed");
  g_na_scratch[dev] = static_cast<unsigned char*>(ptr);
  g_na_sms[dev] = sms;
  g_na_ready[dev] = true;
  return PKD_OK;
}

// ---------------------------------------------------------------- planning into static storage
WorkItem g_na_items[PKD_NOALLOC_MAX_ITEMS];
MergeEntry g_na_merges[PKD_NOALLOC_MAX_MERGES];

struct NaCounts {
  int64_t items = 0, merges = 0, slots = 0;
};

inline int64_t na_len(const int32_t* indptr, const int32_t* lpl, int i, int ps) {
  const int64_t pages = (int64_t)indptr[i + 1] - indptr[i];
  return pages <= 0 ? 0 : (int64_t)ps * (pages - 1) + lpl[i];
}

inline int64_t na_start(int64_t n, int window_left) {
  return (window_left >= 0 && n - 1 - window_left > 0) ? n - 1 - window_left : 0;
}

NaCounts na_count(const int32_t* indptr, const int32_t* lpl, int batch, int ps, int wl, int64_t C) {
  NaCounts c;
  for (int i = 0; i < batch; ++i) {
    const int64_t n = na_len(indptr, lpl, i, ps);
    const int64_t nch = (n == 0 || C == 0) ? 1 : (n - 1) / C - na_start(n, wl) / C + 1;
    c.items += nch;
    if (nch > 1) {
      c.merges += 1;
      c.slots += nch;
    }
  }
  return c;
}

size_t na_partial_bytes(int64_t slots, int hq, int d) {
  const size_t o = (size_t)slots * hq * d * sizeof(float);
  const size_t l = (size_t)slots * hq * sizeof(float);
  return (o + 255) / 256 * 256 + (l + 255) / 256 * 256;
}

bool na_fits(const NaCounts& c, int hq, int d) {
  return c.items <= PKD_NOALLOC_MAX_ITEMS && c.merges <= PKD_NOALLOC_MAX_MERGES &&
         na_partial_bytes(c.slots, hq, d) <= PKD_NOALLOC_PARTIAL_BYTES;
}

// The same rules as the handle-based planner: chunks of C tokens counted from each request's
// token 0 (C = 0: one chunk), chunks the window leaves empty dropped, longest chunks first.
// The heuristic C grows until the plan fits the built-in scratch.
int na_plan(const int32_t* indptr, const int32_t* lpl, int batch, int hq, int hkv, int d, int ps,
            int wl, int fixed, int disable, int sms, NaCounts* out) {
  int64_t total = 0, longest = 0;
  for (int i = 0; i < batch; ++i) {
    if (indptr[i + 1] < indptr[i]) return na_fail(PKD_ERR_INVALID_ARG, "indptr must be non-decreasing");
    const int64_t pages = (int64_t)indptr[i + 1] - indptr[i];
    if (pages > 0 && (lpl[i] < 1 || lpl[i] > ps))
      return na_fail(PKD_ERR_INVALID_ARG,
                     "last_page_len must lie in [1, page_size] for every request with pages");
    const int64_t n = na_len(indptr, lpl, i, ps);
    if (n > (int64_t)std::numeric_limits<int32_t>::max() - 4096)
      return na_fail(PKD_ERR_INVALID_ARG, "a request is longer than 2^31 - 4096 tokens");
    total += n - na_start(n, wl);
    longest = std::max(longest, n - na_start(n, wl));
  }
  int64_t C = 0;
  const bool heuristic = !disable && fixed <= 0;
  if (disable) {
    C = 0;
  } else if (fixed > 0) {
    C = (int64_t)fixed * ps;
  } else {
    const int64_t slots = (int64_t)(sms > 0 ? sms : 152) * 2 * 2;
    const int64_t per_cta = (total * hkv + slots - 1) / slots;  // one head slice per CTA (G <= 8)
    int64_t c = std::max<int64_t>(256, per_cta);
    c = (c + ps - 1) / ps * ps;
    C = longest > c ? c : 0;
  }
  NaCounts cnt = na_count(indptr, lpl, batch, ps, wl, C);
  while (heuristic && C > 0 && !na_fits(cnt, hq, d)) {
    C = C * 2 >= longest ? 0 : C * 2;
    cnt = na_count(indptr, lpl, batch, ps, wl, C);
  }
  if (cnt.items > PKD_NOALLOC_MAX_ITEMS)
    return na_fail(PKD_ERR_WORKSPACE_TOO_SMALL,
                   "plan needs more chunks than the built-in scratch holds (PKD_NOALLOC_MAX_ITEMS)");
  if (cnt.merges > PKD_NOALLOC_MAX_MERGES)
    return na_fail(PKD_ERR_WORKSPACE_TOO_SMALL,
                   "plan splits more requests than the built-in scratch holds (PKD_NOALLOC_MAX_MERGES)");
  if (na_partial_bytes(cnt.slots, hq, d) > PKD_NOALLOC_PARTIAL_BYTES)
    return na_fail(PKD_ERR_WORKSPACE_TOO_SMALL,
                   "split partials exceed the built-in scratch (PKD_NOALLOC_PARTIAL_BYTES); use a "
                   "larger fixed_split_size or disable_split_kv");
  int ni = 0, nm = 0, slot = 0;
  for (int i = 0; i < batch; ++i) {
    WorkItem it;
    std::memset(&it, 0, sizeof it);
    it.req = i;
    it.page_base = indptr[i];
    const int64_t n = na_len(indptr, lpl, i, ps);
    if (n == 0) {
      it.out_slot = -1;
      g_na_items[ni++] = it;
      continue;
    }
    const int64_t w = na_start(n, wl);
    const int64_t k0 = C > 0 ? w / C : 0, k1 = C > 0 ? (n - 1) / C : 0;
    const int64_t nch = k1 - k0 + 1;
    const int first = slot;
    for (int64_t k = k0; k <= k1; ++k) {
      const int64_t c0 = C > 0 ? k * C : 0;
      const int64_t c1 = C > 0 ? std::min(n, (k + 1) * C) : n;
      it.chunk_tok0 = (int32_t)c0;
      it.tok_begin = (int32_t)std::max(c0, w);
      it.tok_end = (int32_t)c1;
      it.out_slot = nch > 1 ? slot++ : -1;
      g_na_items[ni++] = it;
    }
    if (nch > 1) {
      MergeEntry me;
      me.req = i;
      me.first_slot = first;
      me.n_chunks = (int32_t)nch;
      me.pad = 0;
      g_na_merges[nm++] = me;
    }
  }
  std::sort(g_na_items, g_na_items + ni, [](const WorkItem& a, const WorkItem& b) {
    const int la = a.tok_end - a.tok_begin, lb = b.tok_end - b.tok_begin;
    if (la != lb) return la > lb;
    if (a.req != b.req) return a.req < b.req;
    return a.chunk_tok0 < b.chunk_tok0;
  });
  out->items = ni;
  out->merges = nm;
  out->slots = slot;
  return PKD_OK;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*NaEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Same 4-D view as the handle-based path: dims ordered by stride, 128-byte boxes of d by
// `rows` slots of one head of one page, 128-byte swizzle.
int na_tensor_map(CUtensorMap* map, const void* base, int kv_dtype, int d, int ps, int hkv,
                  int64_t num_pages, const int64_t st[3], int layout, int rows) {
  static NaEncodeFn enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return na_fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    enc = reinterpret_cast<NaEncodeFn>(p);
  }
  const int elt = kv_dtype == kE4M3 ? 1 : 2;
  const CUtensorMapDataType dt = kv_dtype == kF16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : kv_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const bool nhd = layout == PKD_LAYOUT_NHD;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)(nhd ? hkv : ps), (cuuint64_t)(nhd ? ps : hkv),
                        (cuuint64_t)num_pages};
  cuuint64_t gstr[3] = {(cuuint64_t)((nhd ? st[2] : st[1]) * elt),
                        (cuuint64_t)((nhd ? st[1] : st[2]) * elt), (cuuint64_t)(st[0] * elt)};
  cuuint32_t box[4] = {(cuuint32_t)(128 / elt), (cuuint32_t)(nhd ? 1 : rows),
                       (cuuint32_t)(nhd ? rows : 1), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (enc(map, dt, 4, const_cast<void*>(base), dims, gstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return na_fail(PKD_ERR_INVALID_ARG, "cuTensorMapEncodeTiled rejected the KV pool view");
  return PKD_OK;
}

bool na_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

// pkd_check_status(NULL, ...): the status word at the start of this device's built-in array,
// read after the stream's earlier work and then cleared.  No allocation either.
int pkd::noalloc_check_status(uint32_t* status, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return na_fail(PKD_ERR_CUDA, "cudaGetDevice failed");
  std::lock_guard<std::mutex> lock(g_na_mutex);
  int rc = na_setup(dev);
  if (rc) return rc;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, g_na_scratch[dev], sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v) e = cudaMemsetAsync(g_na_scratch[dev], 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return na_fail(PKD_ERR_CUDA, "reading the built-in status word failed");
  *status = v;
  return PKD_OK;
}

extern "C" int pkd_decode_noalloc(const int32_t* indptr_host, const int32_t* last_page_len_host,
                                  int batch, const int32_t* indices_dev, int64_t num_indices,
                                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                                  float sm_scale, float logits_soft_cap, int window_left,
                                  int fixed_split_size, int disable_split_kv, int q_dtype,
                                  int kv_dtype, int o_dtype, int use_tensor_cores, int kv_layout,
                                  const void* q, const void* k_base, const void* v_base,
                                  int64_t num_pages, const int64_t kv_strides[3], float q_scale,
                                  float k_scale, float v_scale, void* o, float* lse,
                                  void* stream) {
  // ---- arguments (the rules of pkd_plan and pkd_run)
  if (batch < 0 || (batch > 0 && (!indptr_host || !last_page_len_host || !indices_dev)))
    return na_fail(PKD_ERR_INVALID_ARG, "batch must be >= 0 and the page table pointers non-null");
  if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return na_fail(PKD_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
  if (num_qo_heads / num_kv_heads > 8)
    return na_fail(PKD_ERR_UNSUPPORTED, "this variant serves GQA groups of at most 8 qo heads");
  if (use_tensor_cores != PKD_KERNEL_AUTO && use_tensor_cores != PKD_KERNEL_TENSOR_CORE)
    return na_fail(PKD_ERR_UNSUPPORTED, "this variant is built with the tensor-core kernel only");
  if (kv_layout != PKD_LAYOUT_NHD && kv_layout != PKD_LAYOUT_HND)
    return na_fail(PKD_ERR_INVALID_ARG, "kv_layout must be PKD_LAYOUT_NHD or PKD_LAYOUT_HND");
  if ((q_dtype != kF16 && q_dtype != kBF16) || o_dtype != q_dtype ||
      (kv_dtype != q_dtype && kv_dtype != kE4M3))
    return na_fail(PKD_ERR_UNSUPPORTED, "dtypes: q = o in {F16, BF16}, kv = q or E4M3");
  if ((page_size & (page_size - 1)) != 0 || page_size < 8 || page_size > 256)
    return na_fail(PKD_ERR_UNSUPPORTED, "page_size must be a power of two in [8, 256]");
  const NaDecode* dk = nullptr;
  for (const NaDecode& k : kNaDecode)
    if (k.q_dtype == q_dtype && k.kv_dtype == kv_dtype && k.head_dim == head_dim) dk = &k;
  const NaMerge* mk = nullptr;
  for (const NaMerge& k : kNaMerge)
    if (k.o_dtype == o_dtype && k.head_dim == head_dim) mk = &k;
  if (!dk || !mk)
    return na_fail(PKD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (128 or 256 for e4m3 KV)");
  if (batch > 0 && (indptr_host[0] < 0 || num_indices < (int64_t)indptr_host[batch]))
    return na_fail(PKD_ERR_INVALID_ARG, "indices must hold indptr[batch] page ids from indptr[0] >= 0");
  if (!(std::isnan(sm_scale) || (sm_scale > 0.f && std::isfinite(sm_scale))) ||
      !std::isfinite(logits_soft_cap))
    return na_fail(PKD_ERR_INVALID_ARG, "sm_scale must be positive (or NaN), the soft cap finite");
  if (batch == 0) return PKD_OK;
  if (!q || !k_base || !v_base || !o || !kv_strides || num_pages <= 0 ||
      num_pages > (int64_t(1) << 31))
    return na_fail(PKD_ERR_INVALID_ARG, "null tensor pointer or num_pages outside [1, 2^31]");
  if (!na_aligned(q, 16) || !na_aligned(o, 16) || !na_aligned(k_base, 16) || !na_aligned(v_base, 16))
    return na_fail(PKD_ERR_INVALID_ARG, "q, o and the K/V bases must be 16-byte aligned");
  const int elt = kv_dtype == kE4M3 ? 1 : 2;
  for (int i = 0; i < 3; ++i)
    if (kv_strides[i] <= 0 || (kv_strides[i] * elt) % 16 != 0)
      return na_fail(PKD_ERR_INVALID_ARG, "kv strides must be positive multiples of 16 bytes");
  const bool nhd = kv_layout == PKD_LAYOUT_NHD;
  const int64_t inner = nhd ? kv_strides[2] : kv_strides[1];
  const int64_t outer = nhd ? kv_strides[1] : kv_strides[2];
  if (inner < head_dim || outer < inner * (nhd ? num_kv_heads : page_size) ||
      kv_strides[0] < outer * (nhd ? page_size : num_kv_heads))
    return na_fail(PKD_ERR_INVALID_ARG, "kv strides do not match the layout");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return na_fail(PKD_ERR_CUDA, "cudaGetDevice failed");
  std::lock_guard<std::mutex> lock(g_na_mutex);
  int rc = na_setup(dev);
  if (rc) return rc;
  NaCounts cnt;
  rc = na_plan(indptr_host, last_page_len_host, batch, num_qo_heads, num_kv_heads, head_dim,
               page_size, window_left, fixed_split_size, disable_split_kv, g_na_sms[dev], &cnt);
  if (rc) return rc;

  // ---- upload: clear the status word, copy the work list (pageable source: the copy has
  // left the host buffers when cudaMemcpyAsync returns, so they may be rewritten next call)
  unsigned char* scratch = g_na_scratch[dev];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "clearing the status word failed");
  if (cudaMemcpyAsync(scratch + kNaItemsOff, g_na_items, cnt.items * sizeof(WorkItem),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "uploading the work list failed");
  if (cnt.merges > 0 &&
      cudaMemcpyAsync(scratch + kNaMergesOff, g_na_merges, cnt.merges * sizeof(MergeEntry),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "uploading the merge list failed");

  // ---- decode
  DecodeParams prm;
  std::memset(&prm, 0, sizeof prm);
  const int rows = page_size < dk->tile ? page_size : dk->tile;
  rc = na_tensor_map(&prm.tmap_k, k_base, kv_dtype, head_dim, page_size, num_kv_heads, num_pages,
                     kv_strides, kv_layout, rows);
  if (rc) return rc;
  rc = na_tensor_map(&prm.tmap_v, v_base, kv_dtype, head_dim, page_size, num_kv_heads, num_pages,
                     kv_strides, kv_layout, rows);
  if (rc) return rc;
  const size_t part_o_bytes =
      ((size_t)cnt.slots * num_qo_heads * head_dim * sizeof(float) + 255) / 256 * 256;
  prm.items = reinterpret_cast<const WorkItem*>(scratch + kNaItemsOff);
  prm.indices = indices_dev;
  prm.q = q;
  prm.o = o;
  prm.lse = lse;
  prm.part_o = reinterpret_cast<float*>(scratch + kNaFloatOff);
  prm.part_lse = reinterpret_cast<float*>(scratch + kNaFloatOff + part_o_bytes);
  prm.status = reinterpret_cast<uint32_t*>(scratch);
  prm.wait_ns = kWaitLimitNs;
  prm.num_pages = (uint32_t)num_pages;
  prm.num_qo_heads = num_qo_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = num_qo_heads / num_kv_heads;
  prm.gslices = 1;
  prm.page_size = page_size;
  prm.hnd = nhd ? 0 : 1;
  const double sm = (std::isnan(sm_scale) ? 1.0 / std::sqrt((double)head_dim) : (double)sm_scale) *
                    q_scale * k_scale;
  const double log2e = 1.4426950408889634;
  if (logits_soft_cap > 0.f) {
    prm.scale_qk = (float)(sm / logits_soft_cap);
    prm.cap_log2 = (float)(logits_soft_cap * log2e);
  } else {
    prm.scale_qk = (float)(sm * log2e);
    prm.cap_log2 = 0.f;
  }
  prm.v_scale = v_scale;
  void* args[] = {&prm};
  const unsigned grid = (unsigned)(cnt.items * num_kv_heads);
  if (cudaLaunchKernel(dk->fn, dim3(grid), dim3(dk->threads), args, (size_t)dk->smem, s) !=
      cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "decode kernel launch failed");

  // ---- merge_states for split requests
  if (cnt.merges > 0) {
    MergeParams mp;
    mp.merges = reinterpret_cast<const MergeEntry*>(scratch + kNaMergesOff);
    mp.part_o = prm.part_o;
    mp.part_lse = prm.part_lse;
    mp.o = o;
    mp.lse = lse;
    mp.status = prm.status;
    mp.num_merges = (int)cnt.merges;
    mp.num_qo_heads = num_qo_heads;
    void* margs[] = {&mp};
    const unsigned blocks = (unsigned)((cnt.merges * num_qo_heads + 3) / 4);
    if (cudaLaunchKernel(mk->fn, dim3(blocks), dim3(128), margs, 0, s) != cudaSuccess)
      return na_fail(PKD_ERR_CUDA, "merge kernel launch failed");
  }
  return PKD_OK;
}
