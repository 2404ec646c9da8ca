// noalloc.cu -- pkd_decode_noalloc: plan + run with scratch built into the library.
//
// For callers that may not allocate device memory and have no workspace to lend (a runtime
// that owns every allocation through its own pool or budget).  The scratch they would have
// passed -- status word, merge counters, tasks, merge entries, split partials --
// lives in one file-scope device array.  The plan is built by the library's decode planner
// into static host storage, so a call allocates nothing.  The kernel is the tensor-core decode
// kernel of the rest of the library (split units are merged inside it), instantiated here with
// the same parameters.
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

namespace pkd {
void set_error_message(const char* msg);  // pkd_api.cpp: what pkd_last_error() returns
}

using namespace pkd;

// One array per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char pkd_noalloc_scratch[PKD_NOALLOC_SCRATCH_BYTES];

namespace {

// The array: [status block | counters | tasks | merge entries | partials].
constexpr size_t kNaCountersOff = kStatusBytes;
constexpr size_t kNaTasksOff = kNaCountersOff + (PKD_NOALLOC_MAX_MERGES * 4 + 255) / 256 * 256;
constexpr size_t kNaMergesOff = kNaTasksOff + PKD_NOALLOC_MAX_ITEMS * sizeof(DecodeTask);
constexpr size_t kNaFloatOff = PKD_NOALLOC_SCRATCH_BYTES - PKD_NOALLOC_PARTIAL_BYTES;
static_assert(kNaMergesOff + PKD_NOALLOC_MAX_MERGES * sizeof(MergeEntry) <= kNaFloatOff,
              "work list region overlaps the partials");
static_assert(kNaFloatOff % 256 == 0, "partials region is 256-byte aligned");

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
constexpr int kNaKernels = sizeof(kNaDecode) / sizeof(kNaDecode[0]);

// ---------------------------------------------------------------- per-device set-up
constexpr int kMaxDevices = 64;
std::mutex g_na_mutex;  // guards the set-up table and the static host plan below
bool g_na_ready[kMaxDevices];
unsigned char* g_na_scratch[kMaxDevices];
int g_na_sms[kMaxDevices];
int g_na_per_sm[kMaxDevices][kNaKernels];  // resident CTAs per SM of each kernel

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
  for (int i = 0; i < kNaKernels; ++i) {
    const NaDecode& k = kNaDecode[i];
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) !=
        cudaSuccess)
      return na_fail(PKD_ERR_CUDA, "cudaFuncSetAttribute on a decode kernel failed");
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.fn, k.threads, (size_t)k.smem) !=
        cudaSuccess)
      return na_fail(PKD_ERR_CUDA, "cudaOccupancyMaxActiveBlocksPerMultiprocessor failed");
    g_na_per_sm[dev][i] = std::max(1, std::min(n, kDecodeCtasPerSm));
  }
  g_na_scratch[dev] = static_cast<unsigned char*>(ptr);
  g_na_sms[dev] = sms;
  g_na_ready[dev] = true;
  return PKD_OK;
}

// ---------------------------------------------------------------- static host plan storage
DecodeTask g_na_tasks[PKD_NOALLOC_MAX_ITEMS];
MergeEntry g_na_merges[PKD_NOALLOC_MAX_MERGES];
DecodeChunk g_na_chunks[PKD_NOALLOC_MAX_ITEMS];  // planner scratch

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
  if (!dk)
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
  const int kidx = (int)(dk - kNaDecode);
  const int ctas = g_na_sms[dev] * g_na_per_sm[dev][kidx];

  // ---- plan with the library's decode planner, into the static host storage
  PlanRequest r;
  r.indptr = indptr_host;
  r.last_page_len = last_page_len_host;
  r.batch = batch;
  r.num_qo_heads = num_qo_heads;
  r.num_kv_heads = num_kv_heads;
  r.head_dim = head_dim;
  r.page_size = page_size;
  r.window_left = window_left;
  r.fixed_split_size = fixed_split_size;
  r.disable_split_kv = disable_split_kv;
  r.kv_dtype = kv_dtype;
  r.use_tensor_cores = PKD_KERNEL_TENSOR_CORE;
  r.num_sms = g_na_sms[dev];
  const char* err = "";
  DecodeSchedule sch;
  sch.tasks = g_na_tasks;
  sch.tasks_cap = PKD_NOALLOC_MAX_ITEMS;
  sch.merges = g_na_merges;
  sch.merges_cap = PKD_NOALLOC_MAX_MERGES;
  sch.chunks = g_na_chunks;
  sch.chunks_cap = PKD_NOALLOC_MAX_ITEMS;
  // partial slots: kSlotHeads rows of head_dim + 1 floats each, in the partials region
  sch.max_slots = (int64_t)((PKD_NOALLOC_PARTIAL_BYTES - 512) /
                            ((size_t)kSlotHeads * (head_dim + 1) * sizeof(float)));
  rc = build_decode_schedule(r, ctas, &sch, &err);
  if (rc == PKD_ERR_WORKSPACE_TOO_SMALL) {
    // name the limit of the built-in scratch that the plan ran into
    const bool merges_full = std::strstr(err, "merge") != nullptr;
    const bool partials_full = std::strstr(err, "partials") != nullptr;
    return na_fail(rc, merges_full ? "plan splits more units than the built-in scratch holds "
                                     "(PKD_NOALLOC_MAX_MERGES)"
                       : partials_full
                           ? "split partials exceed the built-in scratch "
                             "(PKD_NOALLOC_PARTIAL_BYTES); use a larger fixed_split_size or "
                             "disable_split_kv"
                           : "plan needs more tasks than the built-in scratch holds "
                             "(PKD_NOALLOC_MAX_ITEMS)");
  }
  if (rc) return na_fail(rc, err);

  // ---- upload: clear the status word and the merge counters, copy the tasks and the merge
  // entries (pageable sources: each copy has left the host buffers when
  // cudaMemcpyAsync returns, so they may be rewritten by the next call)
  unsigned char* scratch = g_na_scratch[dev];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, kNaTasksOff, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "clearing the status word and the merge counters failed");
  if (sch.n_tasks > 0 &&
      cudaMemcpyAsync(scratch + kNaTasksOff, g_na_tasks, (size_t)sch.n_tasks * sizeof(DecodeTask),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "uploading the tasks failed");
  if (sch.n_merges > 0 &&
      cudaMemcpyAsync(scratch + kNaMergesOff, g_na_merges,
                      (size_t)sch.n_merges * sizeof(MergeEntry), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "uploading the merge list failed");

  // ---- decode (split units are merged inside the launch)
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
      ((size_t)sch.n_slots * kSlotHeads * head_dim * sizeof(float) + 255) / 256 * 256;
  prm.tasks = reinterpret_cast<const DecodeTask*>(scratch + kNaTasksOff);
  prm.merges = reinterpret_cast<const MergeEntry*>(scratch + kNaMergesOff);
  prm.counters = reinterpret_cast<uint32_t*>(scratch + kNaCountersOff);
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
  if (sch.n_tasks == 0) return PKD_OK;
  void* args[] = {&prm};
  if (cudaLaunchKernel(dk->fn, dim3((unsigned)sch.n_tasks), dim3(dk->threads), args,
                       (size_t)dk->smem, s) != cudaSuccess)
    return na_fail(PKD_ERR_CUDA, "decode kernel launch failed");
  return PKD_OK;
}
