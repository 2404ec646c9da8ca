// pkd_api.cpp -- the C ABI declared in include/pkd.h: handle, plan, run, status.
//
// Mirrors FlashInfer's BatchDecodeWithPagedKVCacheWrapper (FlashInfer attention API page):
// the constructor takes the workspaces and KV layout, plan() runs once per batch on the host
// and leaves the auxiliary data in the int workspace, run() launches the kernels for one
// layer's pool and may be called any number of times per plan.
#include "../../include/pkd.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <mutex>
#include <string>
#include <vector>

#include "pkd_internal.h"

using namespace pkd;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

std::once_flag g_registry_once;
std::vector<DecodeKernel> g_decode;
std::vector<MlaKernel> g_mla;

void init_registry() {
  std::call_once(g_registry_once, [] {
    register_decode_f16(g_decode);
    register_decode_bf16(g_decode);
    register_decode_e4m3(g_decode);
    register_decode_rope(g_decode);
    register_decode_rope_cc(g_decode);
    register_decode_rope_cc_e4m3(g_decode);
    register_mla(g_mla);
    register_mla_tc(g_mla);
  });
}

const MlaKernel* find_mla(int dtype, int variant) {
  init_registry();
  for (const auto& k : g_mla)
    if (k.dtype == dtype && k.variant == variant) return &k;
  return nullptr;
}

const DecodeKernel* find_decode(int kind, int q_dtype, int kv_dtype, int head_dim, int heads,
                                int rope) {
  init_registry();
  for (const auto& k : g_decode)
    if (k.kind == kind && k.q_dtype == q_dtype && k.kv_dtype == kv_dtype &&
        k.head_dim == head_dim && k.heads_per_cta == heads && k.rope == rope)
      return &k;
  return nullptr;
}

// ALiBi slope of qo head g of H heads (the ALiBi paper's set): with m the largest power of two
// <= H, heads below m take 2^(-8 (g + 1) / m); the others take the odd-indexed slopes of the
// 2m-head sequence, 2^(-4 (2 (g - m) + 1) / m).
double alibi_slope_of(int g, int H) {
  int m = 1;
  while (2 * m <= H) m *= 2;
  return g < m ? std::exp2(-8.0 * (g + 1) / m) : std::exp2(-4.0 * (2 * (g - m) + 1) / m);
}


// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn(std::string* why) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static std::string err;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      err = "cuTensorMapEncodeTiled is not available from the driver";
    else
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) *why = err;
  return fn;
}

}  // namespace

struct pkd_handle {
  void* float_ws = nullptr;
  size_t float_bytes = 0;
  void* int_ws = nullptr;
  size_t int_bytes = 0;
  int layout = PKD_LAYOUT_NHD;
  int device = 0;
  int num_sms = 152;

  bool planned = false;
  Plan plan;
  int batch = 0, num_qo_heads = 0, num_kv_heads = 0, head_dim = 0, page_size = 0;
  int q_len = 1;  // query tokens per request: q / o / lse have batch * q_len rows
  int pos_mode = 0;  // PKD_POS_*
  bool mla = false;  // the current plan is an MLA plan (pkd_mla_plan)
  const MlaKernel* mla_kernel = nullptr;
  int mla_backend = PKD_MLA_BACKEND_AUTO;  // pkd_mla_set_backend
  int q_dtype = 0, kv_dtype = 0, o_dtype = 0;
  float sm_scale = 0.f, cap = 0.f;
  const int32_t* indices = nullptr;
  const DecodeKernel* kernel = nullptr;

  // The decode plan: tasks grouped by CTA, merge entries, CTA ranges, and the grid that runs
  // them (CUDA-graph mode: fixed by the first plan).
  std::vector<DecodeTask> tasks;     // the plan's tasks (the first n_tasks entries)
  std::vector<MergeEntry> dmerges;   // its merge entries (the first n_merges)
  std::vector<DecodeChunk> dchunks;  // planner scratch
  DecodeWsLayout dlayout{};
  int64_t n_dmerges = 0;
  int grid = 0;       // CTAs pkd_run launches (one per task; CUDA-graph mode: the capacity)
  // K / V tensor maps of the pools runs have used, so a run on a pool seen before (every layer
  // of every later step) skips the encoding: a map depends only on these fields
  struct TmapEntry {
    const void* base;
    int64_t num_pages;
    int64_t strides[3];
    int kv_dtype, head_dim, page_size, num_kv_heads, layout, box_rows;
    CUtensorMap map;
  };
  static constexpr size_t kTmapCacheSize = 256;
  std::vector<TmapEntry> tmaps;
  size_t tmap_next = 0;
  int gslices = 1;
  int64_t n_tasks = 0;

  // Pinned copies of the work list for the async uploads, used in turn: plan() waits only for
  // the upload of kStagingSlots plans ago, so a host that plans ahead of the GPU is not held up.
  struct StagingSlot {
    void* ptr = nullptr;
    size_t bytes = 0;
    cudaEvent_t done = nullptr;
    bool pending = false;
  };
  static constexpr int kStagingSlots = 4;
  StagingSlot staging[kStagingSlots];
  int staging_next = 0;
  bool pdl = true;  // launch the decode kernel as a programmatic dependent of its predecessor
  unsigned long long wait_ns = kWaitLimitNs;  // decode pipeline wait limit (pkd_set_wait_limit)

  // The workspace layout the current plan was uploaded in (its own counts, or capacities).
  WsLayout ws_layout{};

  // CUDA-graph mode (pkd_enable_cuda_graph): the page table lives in the caller's fixed
  // buffers, the workspaces are cut for fixed capacities, and every run launches the same
  // grid, so a captured run stays valid across later plans of the same batch size.
  bool graph = false;
  int32_t* g_indptr = nullptr;
  int32_t* g_indices = nullptr;
  int32_t* g_lpl = nullptr;
  int g_max_batch = 0;
  int64_t g_max_pages = 0;
  int g_max_items = 0;
  int g_batch = -1;  // fixed by the first plan in graph mode
  int planned_heads = 0;  // MLA: num_heads of the last plan (fixed in graph mode)
};

namespace {

// The next staging slot with room for `bytes`, once its previous upload has completed.
int staging_acquire(pkd_handle* h, size_t bytes, char** out, int* slot_out) {
  const int slot = h->staging_next;
  auto& st = h->staging[slot];
  cudaError_t e;
  if (st.pending) {
    e = cudaEventSynchronize(st.done);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    st.pending = false;
  }
  if (bytes > st.bytes) {
    if (st.ptr) cudaFreeHost(st.ptr);
    st.ptr = nullptr;
    st.bytes = 0;
    const size_t cap = std::max<size_t>(bytes * 2, 1 << 16);
    e = cudaHostAlloc(&st.ptr, cap, cudaHostAllocDefault);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
    st.bytes = cap;
  }
  *out = static_cast<char*>(st.ptr);
  *slot_out = slot;
  return PKD_OK;
}

// Marks the slot's upload (already enqueued on `s`) and moves to the next slot.
int staging_release(pkd_handle* h, int slot, cudaStream_t s) {
  auto& st = h->staging[slot];
  cudaError_t e = cudaEventRecord(st.done, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  st.pending = true;
  h->staging_next = (slot + 1) % pkd_handle::kStagingSlots;
  return PKD_OK;
}

// 4-D TMA view of one K or V pool: dims (d, head, slot, page) for NHD and (d, slot, head, page)
// for HND, i.e. ordered by increasing stride; a box is 128 bytes of d by `box_rows` slots of
// one head of one page, landing 128-byte swizzled in shared memory.
int make_kv_tensor_map(CUtensorMap* map, const void* base, int kv_dtype, int head_dim, int page_size,
                       int num_kv_heads, int64_t num_pages, const int64_t strides[3], int layout,
                       int box_rows) {
  std::string why;
  EncodeTiledFn enc = get_encode_fn(&why);
  if (!enc) return fail(PKD_ERR_CUDA, why);
  const int elt = kv_dtype == kE4M3 ? 1 : 2;
  const CUtensorMapDataType dt = kv_dtype == kF16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : kv_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int64_t page_b = strides[0] * elt, slot_b = strides[1] * elt, head_b = strides[2] * elt;
  cuuint64_t dims[4], gstr[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  if (layout == PKD_LAYOUT_NHD) {
    dims[1] = (cuuint64_t)num_kv_heads;
    dims[2] = (cuuint64_t)page_size;
    gstr[0] = (cuuint64_t)head_b;
    gstr[1] = (cuuint64_t)slot_b;
    box[1] = 1;
    box[2] = (cuuint32_t)box_rows;
  } else {
    dims[1] = (cuuint64_t)page_size;
    dims[2] = (cuuint64_t)num_kv_heads;
    gstr[0] = (cuuint64_t)slot_b;
    gstr[1] = (cuuint64_t)head_b;
    box[1] = (cuuint32_t)box_rows;
    box[2] = 1;
  }
  dims[0] = (cuuint64_t)head_dim;
  dims[3] = (cuuint64_t)num_pages;
  gstr[2] = (cuuint64_t)page_b;
  box[0] = (cuuint32_t)(128 / elt);
  box[3] = 1;
  CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[256];
    std::snprintf(buf, sizeof buf,
                  "cuTensorMapEncodeTiled failed (%d) for strides page=%lld slot=%lld head=%lld "
                  "bytes",
                  (int)r, (long long)page_b, (long long)slot_b, (long long)head_b);
    return fail(PKD_ERR_INVALID_ARG, buf);
  }
  return PKD_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Raise a decode kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t set_smem_limit_once(const DecodeKernel* k, int device) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == k->fn && d.second == device) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k->smem_bytes);
  if (e == cudaSuccess) done.emplace_back(k->fn, device);
  return e;
}

int fill_plan_request(PlanRequest* r, const int32_t* indptr, const int32_t* lpl, int batch,
                      int hq, int hkv, int d, int ps, int window_left, int fixed_split,
                      int disable_split, int kv_dtype, int use_tc, int num_sms, int q_len) {
  r->indptr = indptr;
  r->last_page_len = lpl;
  r->batch = batch;
  r->num_qo_heads = hq;
  r->num_kv_heads = hkv;
  r->head_dim = d;
  r->page_size = ps;
  r->window_left = window_left;
  r->fixed_split_size = fixed_split;
  r->disable_split_kv = disable_split;
  r->kv_dtype = kv_dtype;
  r->use_tensor_cores = use_tc;
  r->num_sms = num_sms;
  r->q_len = q_len;
  if (use_tc < -1 || use_tc > 1) return fail(PKD_ERR_INVALID_ARG, "use_tensor_cores must be -1, 0 or 1");
  if (q_len < 1) return fail(PKD_ERR_INVALID_ARG, "q_len_per_req must be >= 1");
  return PKD_OK;
}

}  // namespace

namespace {

// Resident CTAs per SM of a decode kernel (its shared memory raised first), cached per kernel
// and device.  The persistent grid is this times the SM count.
int decode_ctas_per_sm(const DecodeKernel* k, int device, int* out) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<const void*, int>, int>> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& c : cache)
    if (c.first.first == k->fn && c.first.second == device) {
      *out = c.second;
      return PKD_OK;
    }
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k->fn, k->threads,
                                                                (size_t)k->smem_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  n = std::max(1, std::min(n, kDecodeCtasPerSm));
  cache.push_back({{k->fn, device}, n});
  *out = n;
  return PKD_OK;
}

// Storage for one decode schedule (host vectors, reused across plans).
struct ScheduleStore {
  std::vector<DecodeTask> tasks;
  std::vector<MergeEntry> merges;
  std::vector<DecodeChunk> chunks;
};

// Plans the batch (the GPU holding `ctas` CTAs at once) into `st`, growing its vectors when a
// plan needs more; *s holds the counts.
int plan_decode(const PlanRequest& r, int ctas, ScheduleStore& st, DecodeSchedule* s) {
  const char* err = "";
  for (int attempt = 0;; ++attempt) {
    s->tasks = st.tasks.data();
    s->tasks_cap = (int64_t)st.tasks.size();
    s->merges = st.merges.data();
    s->merges_cap = (int64_t)st.merges.size();
    s->chunks = st.chunks.data();
    s->chunks_cap = (int64_t)st.chunks.size();
    const int rc = build_decode_schedule(r, ctas, s, &err);
    if (rc == 0) return PKD_OK;
    if (!s->storage_short || attempt > 0) return fail(rc, err);
    st.tasks.resize((size_t)std::max<int64_t>(s->n_tasks, (int64_t)st.tasks.size()));
    st.merges.resize((size_t)std::max<int64_t>(s->n_merges, (int64_t)st.merges.size()));
    st.chunks.resize((size_t)std::max<int64_t>(s->n_chunks, (int64_t)st.chunks.size()));
  }
}

}  // namespace

namespace pkd {
// Lets other translation units of the library report a failure through pkd_last_error().
void set_error_message(const char* msg) { g_last_error.assign(msg); }
}  // namespace pkd

extern "C" {

const char* pkd_last_error(void) { return g_last_error.c_str(); }

int pkd_create(pkd_handle** out, void* float_ws, size_t float_ws_bytes, void* int_ws,
               size_t int_ws_bytes, int kv_layout) {
  if (!out) return fail(PKD_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (kv_layout != PKD_LAYOUT_NHD && kv_layout != PKD_LAYOUT_HND)
    return fail(PKD_ERR_INVALID_ARG, "kv_layout must be PKD_LAYOUT_NHD or PKD_LAYOUT_HND");
  if (!aligned(float_ws, 256) || !aligned(int_ws, 256))
    return fail(PKD_ERR_INVALID_ARG, "workspaces must be 256-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  pkd_handle* h = new pkd_handle();
  h->float_ws = float_ws;
  h->float_bytes = float_ws_bytes;
  h->int_ws = int_ws;
  h->int_bytes = int_ws_bytes;
  h->layout = kv_layout;
  h->device = dev;
  h->num_sms = sms;
  for (auto& st : h->staging) {
    e = cudaEventCreateWithFlags(&st.done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (auto& t : h->staging)
        if (t.done) cudaEventDestroy(t.done);
      delete h;
      return cuda_fail(e, "cudaEventCreate");
    }
  }
  *out = h;
  g_last_error.clear();
  return PKD_OK;
}

int pkd_reset_workspace(pkd_handle* h, void* float_ws, size_t float_ws_bytes, void* int_ws,
                        size_t int_ws_bytes) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (!aligned(float_ws, 256) || !aligned(int_ws, 256))
    return fail(PKD_ERR_INVALID_ARG, "workspaces must be 256-byte aligned");
  h->float_ws = float_ws;
  h->float_bytes = float_ws_bytes;
  h->int_ws = int_ws;
  h->int_bytes = int_ws_bytes;
  h->planned = false;
  return PKD_OK;
}

int pkd_destroy(pkd_handle* h) {
  if (!h) return PKD_OK;
  for (auto& st : h->staging) {
    if (st.pending) cudaEventSynchronize(st.done);
    if (st.ptr) cudaFreeHost(st.ptr);
    if (st.done) cudaEventDestroy(st.done);
  }
  delete h;
  return PKD_OK;
}

int pkd_plan_host(const int32_t* indptr_host, const int32_t* last_page_len_host, int batch,
                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                  int window_left, int fixed_split_size, int disable_split_kv, int kv_dtype,
                  int use_tensor_cores, int num_sms, int32_t* tasks_out, int max_tasks,
                  int32_t* merges_out, int max_merges, int* n_tasks, int* n_merges, int* n_slots,
                  int* kernel_out, int* tile_tokens_out, int work_capacity, int q_len_per_req,
                  int* n_ctas) {
  PlanRequest r;
  int rc = fill_plan_request(&r, indptr_host, last_page_len_host, batch, num_qo_heads,
                             num_kv_heads, head_dim, page_size, window_left, fixed_split_size,
                             disable_split_kv, kv_dtype, use_tensor_cores, num_sms,
                             q_len_per_req);
  if (rc) return rc;
  r.max_items = work_capacity > 0 ? work_capacity : 0;
  ScheduleStore st;
  DecodeSchedule sch;
  rc = plan_decode(r, (num_sms > 0 ? num_sms : 152) * kDecodeCtasPerSm, st, &sch);
  if (rc) return rc;
  if (n_tasks) *n_tasks = (int)sch.n_tasks;
  if (n_merges) *n_merges = (int)sch.n_merges;
  if (n_slots) *n_slots = (int)sch.n_slots;
  if (kernel_out) *kernel_out = sch.kind;
  if (tile_tokens_out) *tile_tokens_out = sch.tile_tokens;
  if (n_ctas) *n_ctas = (int)sch.n_tasks;
  if (tasks_out)
    std::memcpy(tasks_out, st.tasks.data(),
                sizeof(DecodeTask) *
                    std::min<size_t>((size_t)sch.n_tasks, (size_t)std::max(0, max_tasks)));
  if (merges_out)
    std::memcpy(merges_out, st.merges.data(),
                sizeof(MergeEntry) *
                    std::min<size_t>((size_t)sch.n_merges, (size_t)std::max(0, max_merges)));
  g_last_error.clear();
  return PKD_OK;
}

int pkd_workspace_bytes(const int32_t* indptr_host, const int32_t* last_page_len_host, int batch,
                        int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                        int window_left, int fixed_split_size, int disable_split_kv, int kv_dtype,
                        int use_tensor_cores, int num_sms, int q_len_per_req,
                        size_t* float_ws_bytes, size_t* int_ws_bytes) {
  PlanRequest r;
  int rc = fill_plan_request(&r, indptr_host, last_page_len_host, batch, num_qo_heads,
                             num_kv_heads, head_dim, page_size, window_left, fixed_split_size,
                             disable_split_kv, kv_dtype, use_tensor_cores, num_sms,
                             q_len_per_req);
  if (rc) return rc;
  ScheduleStore st;
  DecodeSchedule sch;
  const int ctas = (num_sms > 0 ? num_sms : 152) * kDecodeCtasPerSm;
  rc = plan_decode(r, ctas, st, &sch);
  if (rc) return rc;
  DecodeWsLayout lay{(size_t)sch.n_tasks, (size_t)sch.n_merges, (size_t)sch.n_slots};
  lay.pos_floats = 2 * (size_t)head_dim + num_qo_heads;  // room for a positional encoding
  if (float_ws_bytes) *float_ws_bytes = dws_float_bytes(lay, head_dim);
  if (int_ws_bytes) *int_ws_bytes = dws_int_bytes(lay);
  return PKD_OK;
}

int pkd_plan(pkd_handle* h, const int32_t* indptr_host, const int32_t* last_page_len_host,
             int batch, const int32_t* indices_dev, int64_t num_indices, int num_qo_heads,
             int num_kv_heads, int head_dim, int page_size, float sm_scale, float logits_soft_cap,
             int window_left, int fixed_split_size, int disable_split_kv, int q_dtype,
             int kv_dtype, int o_dtype, int use_tensor_cores, int q_len_per_req,
             int pos_encoding_mode, float rope_scale, float rope_theta, void* stream) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  h->planned = false;
  if (q_dtype != PKD_DTYPE_F16 && q_dtype != PKD_DTYPE_BF16)
    return fail(PKD_ERR_INVALID_ARG, "q_dtype must be F16 or BF16");
  if (o_dtype != q_dtype) return fail(PKD_ERR_UNSUPPORTED, "o_dtype must equal q_dtype");
  if (kv_dtype != q_dtype && kv_dtype != PKD_DTYPE_E4M3)
    return fail(PKD_ERR_UNSUPPORTED, "kv_dtype must equal q_dtype or be E4M3");
  if (batch > 0 && !indices_dev) return fail(PKD_ERR_INVALID_ARG, "indices_dev is null");
  if (batch > 0 && num_indices < (int64_t)indptr_host[batch])
    return fail(PKD_ERR_INVALID_ARG, "indices holds fewer than indptr[batch] page ids");
  if (!(std::isnan(sm_scale) || (sm_scale > 0.f && std::isfinite(sm_scale))))
    return fail(PKD_ERR_INVALID_ARG, "sm_scale must be positive and finite, or NaN for the default");
  if (!std::isfinite(logits_soft_cap))
    return fail(PKD_ERR_INVALID_ARG, "logits_soft_cap must be finite");
  if (pos_encoding_mode != PKD_POS_NONE && pos_encoding_mode != PKD_POS_ROPE_LLAMA &&
      pos_encoding_mode != PKD_POS_ALIBI)
    return fail(PKD_ERR_INVALID_ARG, "pos_encoding_mode must be PKD_POS_NONE, _ROPE_LLAMA or _ALIBI");
  if (pos_encoding_mode == PKD_POS_ROPE_LLAMA &&
      !(rope_scale > 0.f && std::isfinite(rope_scale) && rope_theta > 0.f &&
        std::isfinite(rope_theta)))
    return fail(PKD_ERR_INVALID_ARG, "rope_scale and rope_theta must be positive and finite");

  if (h->graph) {
    if (batch < 1 || batch > h->g_max_batch)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: batch must lie in [1, max_batch]");
    if (h->g_batch >= 0 && batch != h->g_batch)
      return fail(PKD_ERR_INVALID_ARG,
                  "CUDA-graph mode: the batch size is fixed by the first plan (pad the batch "
                  "with zero-length requests instead)");
    if ((int64_t)indptr_host[batch] > h->g_max_pages)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: indptr[batch] exceeds max_pages");
    if (h->g_batch >= 0 && q_len_per_req != h->q_len)
      return fail(PKD_ERR_INVALID_ARG,
                  "CUDA-graph mode: q_len_per_req is fixed by the first plan");
    if (h->g_batch >= 0 && h->mla)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: the handle holds MLA plans");
  }

  PlanRequest r;
  int rc = fill_plan_request(&r, indptr_host, last_page_len_host, batch, num_qo_heads,
                             num_kv_heads, head_dim, page_size, window_left, fixed_split_size,
                             disable_split_kv, kv_dtype, use_tensor_cores, h->num_sms,
                             q_len_per_req);
  if (rc) return rc;
  if (h->graph) r.max_items = h->g_max_items;
  r.rope = pos_encoding_mode == PKD_POS_ROPE_LLAMA ? 1 : 0;
  DecodeSchedule sch;
  const char* err = "";
  rc = decode_geometry(r, &sch, &err);
  if (rc) return fail(rc, err);
  const DecodeKernel* k =
      find_decode(sch.kind, q_dtype, kv_dtype, head_dim, sch.heads_per_cta, r.rope);
  if (!k) return fail(PKD_ERR_UNSUPPORTED, "no decode kernel built for this dtype / head_dim");
  cudaError_t e = set_smem_limit_once(k, h->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  // every resident CTA slot of the GPU: the persistent grid of the balanced layout
  int per_sm = 0;
  if (int rc2 = decode_ctas_per_sm(k, h->device, &per_sm)) return rc2;
  const int ctas = h->num_sms * per_sm;
  ScheduleStore st;
  st.tasks.swap(h->tasks);
  st.merges.swap(h->dmerges);
  st.chunks.swap(h->dchunks);
  rc = plan_decode(r, ctas, st, &sch);
  st.tasks.swap(h->tasks);
  st.merges.swap(h->dmerges);
  st.chunks.swap(h->dchunks);
  if (rc) return rc;
  // one CTA per task; CUDA-graph mode launches the capacity's grid for every plan and the CTAs
  // past a plan's tasks leave at once
  const int64_t grid64 = h->graph ? (int64_t)h->g_max_items * num_kv_heads * sch.gslices
                                  : sch.n_tasks;
  if (grid64 > std::numeric_limits<int32_t>::max() / 2)
    return fail(PKD_ERR_INVALID_ARG, "too many work items for one grid");
  const int grid = (int)grid64;

  DecodeWsLayout lay = h->graph ? decode_capacity_layout(h->g_max_items, num_kv_heads,
                                                         sch.gslices)
                                : DecodeWsLayout{(size_t)sch.n_tasks, (size_t)sch.n_merges,
                                                 (size_t)sch.n_slots};
  if (pos_encoding_mode != PKD_POS_NONE) lay.pos_floats = 2 * (size_t)head_dim + num_qo_heads;
  const size_t need_f = dws_float_bytes(lay, head_dim);
  const size_t need_i = dws_int_bytes(lay);
  if (need_f > h->float_bytes || need_i > h->int_bytes) {
    char buf[200];
    std::snprintf(buf, sizeof buf, "workspace too small: need %zu float / %zu int bytes", need_f,
                  need_i);
    return fail(PKD_ERR_WORKSPACE_TOO_SMALL, buf);
  }

  // Upload the int workspace image -- zeroed status block and merge counters, the CTA ranges,
  // the tasks and the merge entries at the layout's offsets (and the positional-encoding
  // table) -- with one copy (graph mode adds the page table's copies into the fixed buffers);
  // wait for the upload of four plans ago to leave its pinned buffer first.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tasks_off = dws_tasks_offset(lay);
  const size_t merges_off = dws_merges_offset(lay);
  const size_t pos_off = dws_pos_offset(lay);
  const size_t tasks_b = (size_t)sch.n_tasks * sizeof(DecodeTask);
  const size_t merges_b = (size_t)sch.n_merges * sizeof(MergeEntry);
  const size_t img_bytes = lay.pos_floats ? pos_off + lay.pos_floats * sizeof(float)
                                          : merges_off + merges_b;
  const size_t table_b = h->graph ? (size_t)(2 * batch + 1) * sizeof(int32_t) : 0;
  const size_t bytes = img_bytes + table_b;
  char* img = nullptr;
  int slot = 0;
  if (int rc2 = staging_acquire(h, bytes, &img, &slot)) return rc2;
  std::memset(img, 0, tasks_off);
  if (h->graph) {
    const int32_t count = (int32_t)sch.n_tasks;
    std::memcpy(img + kItemCountOffset, &count, sizeof count);
  }
  if (tasks_b) std::memcpy(img + tasks_off, h->tasks.data(), tasks_b);
  if (merges_b) std::memcpy(img + merges_off, h->dmerges.data(), merges_b);
  if (lay.pos_floats) {
    // [head_dim / 2] x {rate hi, rate lo}: the RoPE angle rate theta^(-2i/D) / rope_scale of
    // dim pair i as a float pair (head_dim floats); from float 2 * head_dim, [num_qo_heads]
    // ALiBi slopes in score units (per unit of t - pos)
    float* tbl = reinterpret_cast<float*>(img + pos_off);
    std::memset(tbl, 0, lay.pos_floats * sizeof(float));
    if (pos_encoding_mode == PKD_POS_ROPE_LLAMA) {
      for (int i = 0; i < head_dim / 2; ++i) {
        const double rate = std::pow((double)rope_theta, -2.0 * i / head_dim) / rope_scale;
        const float hi = (float)rate;
        tbl[2 * i] = hi;
        tbl[2 * i + 1] = (float)(rate - (double)hi);
      }
    } else {
      const double unit = logits_soft_cap > 0.f ? 1.0 / logits_soft_cap : 1.4426950408889634;
      for (int g = 0; g < num_qo_heads; ++g)
        tbl[2 * head_dim + g] = (float)(alibi_slope_of(g, num_qo_heads) * unit);
    }
  }
  e = cudaMemcpyAsync(h->int_ws, img, img_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  if (h->graph) {
    int32_t* tbl = reinterpret_cast<int32_t*>(img + img_bytes);
    std::memcpy(tbl, indptr_host, (size_t)(batch + 1) * sizeof(int32_t));
    std::memcpy(tbl + batch + 1, last_page_len_host, (size_t)batch * sizeof(int32_t));
    e = cudaMemcpyAsync(h->g_indptr, tbl, (size_t)(batch + 1) * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->g_lpl, tbl + batch + 1, (size_t)batch * sizeof(int32_t),
                          cudaMemcpyHostToDevice, s);
    const int64_t n_ids = indptr_host[batch];
    if (e == cudaSuccess && n_ids > 0 && indices_dev != h->g_indices)
      e = cudaMemcpyAsync(h->g_indices, indices_dev, (size_t)n_ids * sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "copying the page table into the graph buffers");
  }
  if (int rc2 = staging_release(h, slot, s)) return rc2;

  h->n_tasks = sch.n_tasks;
  h->n_dmerges = sch.n_merges;
  h->gslices = sch.gslices;
  h->grid = grid;
  h->batch = batch;
  h->q_len = q_len_per_req;
  h->num_qo_heads = num_qo_heads;
  h->num_kv_heads = num_kv_heads;
  h->head_dim = head_dim;
  h->page_size = page_size;
  h->q_dtype = q_dtype;
  h->kv_dtype = kv_dtype;
  h->o_dtype = o_dtype;
  h->sm_scale = std::isnan(sm_scale) ? 1.0f / std::sqrt((float)head_dim) : sm_scale;
  h->cap = logits_soft_cap > 0.f ? logits_soft_cap : 0.f;
  h->indices = h->graph ? h->g_indices : indices_dev;
  h->dlayout = lay;
  if (h->graph) h->g_batch = batch;
  h->kernel = k;
  h->pos_mode = pos_encoding_mode;
  h->mla = false;
  h->planned = true;
  g_last_error.clear();
  return PKD_OK;
}

}  // extern "C"

namespace {

// make_kv_tensor_map through the handle's cache of maps.
int cached_kv_tensor_map(pkd_handle* h, CUtensorMap* map, const void* base, int64_t num_pages,
                         const int64_t strides[3], int box_rows) {
  for (const auto& t : h->tmaps)
    if (t.base == base && t.num_pages == num_pages && t.strides[0] == strides[0] &&
        t.strides[1] == strides[1] && t.strides[2] == strides[2] && t.kv_dtype == h->kv_dtype &&
        t.head_dim == h->head_dim && t.page_size == h->page_size &&
        t.num_kv_heads == h->num_kv_heads && t.layout == h->layout && t.box_rows == box_rows) {
      *map = t.map;
      return PKD_OK;
    }
  int rc = make_kv_tensor_map(map, base, h->kv_dtype, h->head_dim, h->page_size,
                              h->num_kv_heads, num_pages, strides, h->layout, box_rows);
  if (rc) return rc;
  pkd_handle::TmapEntry e{base, num_pages, {strides[0], strides[1], strides[2]}, h->kv_dtype,
                          h->head_dim, h->page_size, h->num_kv_heads, h->layout, box_rows, *map};
  if (h->tmaps.size() < pkd_handle::kTmapCacheSize) {
    h->tmaps.push_back(e);
  } else {
    h->tmaps[h->tmap_next] = e;
    h->tmap_next = (h->tmap_next + 1) % pkd_handle::kTmapCacheSize;
  }
  return PKD_OK;
}

}  // namespace

extern "C" {

int pkd_run_timed(pkd_handle* h, const void* q, const void* k_base, const void* v_base,
                  int64_t num_pages, const int64_t kv_strides[3], float q_scale, float k_scale,
                  float v_scale, void* o, float* lse, void* stream, void* ev_start, void* ev_end) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (!h->planned || h->mla)
    return fail(PKD_ERR_NOT_PLANNED, "pkd_run called before a successful pkd_plan");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->n_tasks == 0 && !h->graph) return PKD_OK;  // empty batch
  if (!q || !k_base || !v_base || !o || !kv_strides)
    return fail(PKD_ERR_INVALID_ARG, "null q / k_base / v_base / o / kv_strides");
  if (num_pages <= 0 || num_pages > (int64_t(1) << 31))
    return fail(PKD_ERR_INVALID_ARG, "num_pages must lie in [1, 2^31]");
  if (!aligned(k_base, 16) || !aligned(v_base, 16) || !aligned(q, 16) || !aligned(o, 16))
    return fail(PKD_ERR_INVALID_ARG, "q, o and the K/V bases must be 16-byte aligned");
  const int elt = h->kv_dtype == kE4M3 ? 1 : 2;
  for (int i = 0; i < 3; ++i)
    if (kv_strides[i] <= 0 || (kv_strides[i] * elt) % 16 != 0)
      return fail(PKD_ERR_INVALID_ARG, "kv strides must be positive multiples of 16 bytes");
  const int64_t D = h->head_dim;
  const bool nhd = h->layout == PKD_LAYOUT_NHD;
  const int64_t inner = nhd ? kv_strides[2] : kv_strides[1];  // stride of the faster of slot/head
  const int64_t outer = nhd ? kv_strides[1] : kv_strides[2];
  const int64_t inner_n = nhd ? h->num_kv_heads : h->page_size;
  const int64_t outer_n = nhd ? h->page_size : h->num_kv_heads;
  if (inner < D || outer < inner * inner_n || kv_strides[0] < outer * outer_n)
    return fail(PKD_ERR_INVALID_ARG,
                "kv strides do not match the handle's layout (NHD: page > slot > head >= "
                "head_dim; HND: page > head > slot >= head_dim, without overlap)");

  DecodeParams prm;
  std::memset(&prm, 0, sizeof prm);
  const int tile = h->kernel->tile_tokens;
  const int box_rows = h->page_size < tile ? h->page_size : tile;
  int rc = cached_kv_tensor_map(h, &prm.tmap_k, k_base, num_pages, kv_strides, box_rows);
  if (rc) return rc;
  rc = cached_kv_tensor_map(h, &prm.tmap_v, v_base, num_pages, kv_strides, box_rows);
  if (rc) return rc;

  char* iws = static_cast<char*>(h->int_ws);
  char* fws = static_cast<char*>(h->float_ws);
  const DecodeWsLayout& lay = h->dlayout;
  prm.tasks = reinterpret_cast<const DecodeTask*>(iws + dws_tasks_offset(lay));
  prm.task_count = h->graph ? reinterpret_cast<const int32_t*>(iws + kItemCountOffset) : nullptr;
  prm.merges = reinterpret_cast<const MergeEntry*>(iws + dws_merges_offset(lay));
  prm.counters = reinterpret_cast<uint32_t*>(iws + dws_counters_offset());
  prm.pos_table =
      lay.pos_floats ? reinterpret_cast<const float*>(iws + dws_pos_offset(lay)) : nullptr;
  prm.alibi = h->pos_mode == PKD_POS_ALIBI ? 1 : 0;
  prm.indices = h->indices;
  prm.q = q;
  prm.o = o;
  prm.lse = lse;
  prm.part_o = reinterpret_cast<float*>(fws);
  prm.part_lse = reinterpret_cast<float*>(fws + dws_part_lse_offset(lay, h->head_dim));
  prm.status = reinterpret_cast<uint32_t*>(iws);
  prm.wait_ns = h->wait_ns;
  prm.num_pages = (uint32_t)num_pages;
  prm.num_qo_heads = h->num_qo_heads;
  prm.num_kv_heads = h->num_kv_heads;
  prm.group = h->num_qo_heads / h->num_kv_heads;
  prm.page_size = h->page_size;
  prm.hnd = nhd ? 0 : 1;
  const double log2e = 1.4426950408889634;
  const double sm = (double)h->sm_scale * q_scale * k_scale;
  if (h->cap > 0.f) {
    prm.scale_qk = (float)(sm / h->cap);
    prm.cap_log2 = (float)(h->cap * log2e);
  } else {
    prm.scale_qk = (float)(sm * log2e);
    prm.cap_log2 = 0.f;
  }
  prm.v_scale = v_scale;

  const int64_t grid = h->grid;  // persistent CTAs (CUDA-graph mode: the fixed grid)
  void* args[] = {&prm};
  cudaError_t e;
  if (ev_start && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_start), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");
  {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(h->kernel->threads);
    cfg.dynamicSmemBytes = (size_t)h->kernel->smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = h->pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, h->kernel->fn, args);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  if (ev_end && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_end), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");

  // split (row, kv head, slice) units are merged by the CTA that finishes their last chunk
  return PKD_OK;
}

int pkd_run(pkd_handle* h, const void* q, const void* k_base, const void* v_base,
            int64_t num_pages, const int64_t kv_strides[3], float q_scale, float k_scale,
            float v_scale, void* o, float* lse, void* stream) {
  return pkd_run_timed(h, q, k_base, v_base, num_pages, kv_strides, q_scale, k_scale, v_scale, o,
                       lse, stream, nullptr, nullptr);
}

namespace {

// The kernel `backend` names; auto takes the tcgen05 pair kernel above 32 heads.  Measured on
// GB300 (page 1, bf16): the pair kernel's time barely depends on the head count (its row
// gathers set the pace), while the mma.sync kernel re-reads the rows for every 32-head slice --
// at 64 heads the pair kernel is 1.5-1.7x faster, at 16-32 heads the two are within 10 %.
int mla_variant_for(int backend, int num_heads) {
  return backend == PKD_MLA_BACKEND_MMA_SYNC  ? kMlaMmaSync
         : backend == PKD_MLA_BACKEND_TCGEN05 ? kMlaTcgen05
         : num_heads > 32                     ? kMlaTcgen05
                                              : kMlaMmaSync;
}

// The MLA work list and the kernel that runs it (shared by pkd_mla_plan and the host-only
// pkd_mla_plan_host).
int build_mla_plan(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int batch,
                   int num_heads, int page_size, int dtype, int backend, int num_sms,
                   const MlaKernel** kernel, Plan* plan, int max_items = 0) {
  const int variant = mla_variant_for(backend, num_heads);
  const MlaKernel* k = find_mla(dtype, variant);
  if (!k) return fail(PKD_ERR_UNSUPPORTED, "no MLA kernel built for this dtype");
  PlanRequest r;
  std::memset(&r, 0, sizeof r);
  r.indptr = kv_indptr_host;
  r.kv_len = kv_len_host;
  r.batch = batch;
  r.num_qo_heads = num_heads;
  r.num_kv_heads = 1;
  r.head_dim = 512;
  r.page_size = page_size;
  r.window_left = -1;
  r.kv_dtype = dtype;
  r.use_tensor_cores = 1;
  r.num_sms = num_sms;
  r.q_len = 1;
  r.mla = 1;
  r.mla_heads_per_cta = k->heads_per_cta;
  r.mla_tile_tokens = k->tile_tokens;
  r.mla_ctas_per_head_tile = k->ctas_per_head_tile;
  r.ctas_per_sm = 1;  // both MLA kernels take most of an SM's shared memory
  r.max_items = max_items;
  const char* err = "";
  const int rc = build_plan(r, plan, &err);
  if (rc) return fail(rc, err);
  *kernel = k;
  return PKD_OK;
}

}  // namespace

int pkd_mla_plan_host(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int batch,
                      int num_heads, int page_size, int dtype, int backend, int num_sms,
                      int32_t* items_out, int max_items, int32_t* merges_out, int max_merges,
                      int* n_items, int* n_merges, int* n_slots, int* ctas_per_item,
                      size_t* float_ws_bytes, size_t* int_ws_bytes) {
  if (batch < 0 || (batch > 0 && (!kv_indptr_host || !kv_len_host)))
    return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0 and the tables non-null");
  if (num_heads <= 0) return fail(PKD_ERR_INVALID_ARG, "num_heads must be positive");
  if (dtype != PKD_DTYPE_F16 && dtype != PKD_DTYPE_BF16)
    return fail(PKD_ERR_UNSUPPORTED, "MLA takes F16 or BF16");
  if (backend != PKD_MLA_BACKEND_AUTO && backend != PKD_MLA_BACKEND_MMA_SYNC &&
      backend != PKD_MLA_BACKEND_TCGEN05)
    return fail(PKD_ERR_INVALID_ARG, "backend must be PKD_MLA_BACKEND_AUTO, _MMA_SYNC or _TCGEN05");
  const MlaKernel* k = nullptr;
  Plan plan;
  const int rc = build_mla_plan(kv_indptr_host, kv_len_host, batch, num_heads, page_size, dtype,
                                backend, num_sms > 0 ? num_sms : 152, &k, &plan);
  if (rc) return rc;
  const int cph = k->ctas_per_head_tile;
  const WsLayout lay = layout_of(plan, 1);
  if (n_items) *n_items = (int)plan.items.size();
  if (n_merges) *n_merges = (int)plan.merges.size();
  if (n_slots) *n_slots = plan.num_slots;
  if (ctas_per_item) *ctas_per_item = plan.gslices;
  if (float_ws_bytes) *float_ws_bytes = float_ws_bytes_of(lay, num_heads * cph, 512 / cph);
  if (int_ws_bytes) *int_ws_bytes = int_ws_bytes_of(lay);
  if (items_out)
    std::memcpy(items_out, plan.items.data(),
                sizeof(WorkItem) * std::min<size_t>(plan.items.size(), (size_t)std::max(0, max_items)));
  if (merges_out)
    std::memcpy(merges_out, plan.merges.data(),
                sizeof(MergeEntry) *
                    std::min<size_t>(plan.merges.size(), (size_t)std::max(0, max_merges)));
  g_last_error.clear();
  return PKD_OK;
}

int pkd_mla_plan(pkd_handle* h, const int32_t* kv_indptr_host, const int32_t* kv_len_host,
                 int batch, const int32_t* kv_indices_dev, int64_t num_indices, int num_heads,
                 int head_dim_ckv, int head_dim_kpe, int page_size, int causal, float sm_scale,
                 int q_dtype, int kv_dtype, void* stream) {
  (void)causal;  // one query per request: nothing is masked
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  h->planned = false;
  if (head_dim_ckv != 512 || head_dim_kpe != 64)
    return fail(PKD_ERR_UNSUPPORTED, "MLA is built for head_dim_ckv 512 and head_dim_kpe 64");
  if (q_dtype != kv_dtype || (q_dtype != PKD_DTYPE_F16 && q_dtype != PKD_DTYPE_BF16))
    return fail(PKD_ERR_UNSUPPORTED, "MLA takes F16 or BF16 q and caches of the same dtype");
  if (num_heads <= 0) return fail(PKD_ERR_INVALID_ARG, "num_heads must be positive");
  if (!(sm_scale > 0.f && std::isfinite(sm_scale)))
    return fail(PKD_ERR_INVALID_ARG, "sm_scale must be positive and finite");
  if (batch < 0 || (batch > 0 && (!kv_indptr_host || !kv_len_host)))
    return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0 and the tables non-null");
  if (batch > 0 && (!kv_indices_dev || num_indices < (int64_t)kv_indptr_host[batch]))
    return fail(PKD_ERR_INVALID_ARG, "kv_indices holds fewer than kv_indptr[batch] page ids");
  if (h->graph) {
    if (batch < 1 || batch > h->g_max_batch)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: batch must lie in [1, max_batch]");
    if (h->g_batch >= 0 && batch != h->g_batch)
      return fail(PKD_ERR_INVALID_ARG,
                  "CUDA-graph mode: the batch size is fixed by the first plan (pad the batch "
                  "with zero-length requests instead)");
    if ((int64_t)kv_indptr_host[batch] > h->g_max_pages)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: kv_indptr[batch] exceeds max_pages");
    if (h->g_batch >= 0 && !h->mla)
      return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: the handle holds decode plans");
    if (h->g_batch >= 0 &&
        (h->planned_heads != num_heads || h->page_size != page_size || h->sm_scale != sm_scale))
      return fail(PKD_ERR_INVALID_ARG,
                  "CUDA-graph mode: num_heads, page_size and sm_scale are fixed by the first "
                  "plan (a captured run holds them)");
  }

  const MlaKernel* k = nullptr;
  Plan plan;
  int rc = build_mla_plan(kv_indptr_host, kv_len_host, batch, num_heads, page_size, q_dtype,
                          h->mla_backend, h->num_sms, &k, &plan, h->graph ? h->g_max_items : 0);
  if (rc) return rc;
  if (h->graph && h->g_batch >= 0 && h->mla && k != h->mla_kernel)
    return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode: the kernel is fixed by the first plan");

  // partials: [slots, H * cph, 512 / cph] fp32 and [slots, H * cph] lse (cph CTAs per head tile
  // each keep their own lse copy); CUDA-graph mode cuts the workspaces for the capacities
  const int cph = k->ctas_per_head_tile;
  const WsLayout lay =
      h->graph ? capacity_layout(h->g_max_items, 1, plan.gslices) : layout_of(plan, 1);
  const size_t need_f = float_ws_bytes_of(lay, num_heads * cph, head_dim_ckv / cph);
  const size_t need_i = int_ws_bytes_of(lay);
  if (need_f > h->float_bytes || need_i > h->int_bytes) {
    char buf[200];
    std::snprintf(buf, sizeof buf, "workspace too small: need %zu float / %zu int bytes", need_f,
                  need_i);
    return fail(PKD_ERR_WORKSPACE_TOO_SMALL, buf);
  }
  static std::once_flag smem_once;
  cudaError_t e = cudaSuccess;
  std::call_once(smem_once, [&] {
    for (const auto& m : g_mla)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(m.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, m.smem_bytes);
  });
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");

  // one upload of the int workspace image: zeroed status block and counters, items, merges
  // (CUDA-graph mode: also the item count, and the page table into the caller's buffers)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t items_off = items_offset(lay), merges_off = merges_offset(lay);
  const size_t items_b = plan.items.size() * sizeof(WorkItem);
  const size_t merges_b = plan.merges.size() * sizeof(MergeEntry);
  const size_t img_bytes = merges_off + merges_b;
  const size_t table_b = h->graph ? (size_t)(2 * batch + 1) * sizeof(int32_t) : 0;
  char* img = nullptr;
  int slot = 0;
  if (int rc2 = staging_acquire(h, img_bytes + table_b, &img, &slot)) return rc2;
  std::memset(img, 0, merges_off);
  if (h->graph) {
    const int32_t count = (int32_t)plan.items.size();
    std::memcpy(img + kItemCountOffset, &count, sizeof count);
  }
  if (items_b) std::memcpy(img + items_off, plan.items.data(), items_b);
  if (merges_b) std::memcpy(img + merges_off, plan.merges.data(), merges_b);
  e = cudaMemcpyAsync(h->int_ws, img, img_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  if (h->graph) {
    int32_t* tbl = reinterpret_cast<int32_t*>(img + img_bytes);
    std::memcpy(tbl, kv_indptr_host, (size_t)(batch + 1) * sizeof(int32_t));
    std::memcpy(tbl + batch + 1, kv_len_host, (size_t)batch * sizeof(int32_t));
    e = cudaMemcpyAsync(h->g_indptr, tbl, (size_t)(batch + 1) * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->g_lpl, tbl + batch + 1, (size_t)batch * sizeof(int32_t),
                          cudaMemcpyHostToDevice, s);
    const int64_t n_ids = kv_indptr_host[batch];
    if (e == cudaSuccess && n_ids > 0 && kv_indices_dev != h->g_indices)
      e = cudaMemcpyAsync(h->g_indices, kv_indices_dev, (size_t)n_ids * sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "copying the page table into the graph buffers");
  }
  if (int rc2 = staging_release(h, slot, s)) return rc2;

  h->plan = std::move(plan);
  h->batch = batch;
  h->q_len = 1;
  h->num_qo_heads = num_heads;
  h->num_kv_heads = 1;
  h->head_dim = head_dim_ckv;
  h->page_size = page_size;
  h->q_dtype = q_dtype;
  h->kv_dtype = kv_dtype;
  h->o_dtype = q_dtype;
  h->sm_scale = sm_scale;
  h->cap = 0.f;
  h->indices = h->graph ? h->g_indices : kv_indices_dev;
  h->ws_layout = lay;
  if (h->graph) h->g_batch = batch;
  h->planned_heads = num_heads;
  h->pos_mode = PKD_POS_NONE;
  h->kernel = nullptr;
  h->mla = true;
  h->mla_kernel = k;
  h->planned = true;
  g_last_error.clear();
  return PKD_OK;
}

int pkd_mla_run(pkd_handle* h, const void* q_nope, const void* q_pe, const void* ckv_cache,
                const void* kpe_cache, int64_t num_pages, void* o, float* lse, int lse_base_e,
                void* stream, void* ev_start, void* ev_end) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (!h->planned || !h->mla)
    return fail(PKD_ERR_NOT_PLANNED, "pkd_mla_run called without a successful pkd_mla_plan");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->plan.items.empty() && !h->graph) return PKD_OK;
  if (!q_nope || !q_pe || !ckv_cache || !kpe_cache || !o)
    return fail(PKD_ERR_INVALID_ARG, "null q_nope / q_pe / ckv / kpe / o");
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(ckv_cache, 16) ||
      !aligned(kpe_cache, 16) || !aligned(o, 16))
    return fail(PKD_ERR_INVALID_ARG, "q, the caches and o must be 16-byte aligned");
  if (num_pages <= 0) return fail(PKD_ERR_INVALID_ARG, "num_pages must be positive");
  char* iws = static_cast<char*>(h->int_ws);
  char* fws = static_cast<char*>(h->float_ws);
  const WsLayout& lay = h->ws_layout;
  MlaParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.items = reinterpret_cast<const WorkItem*>(iws + items_offset(lay));
  prm.merges = reinterpret_cast<const MergeEntry*>(iws + merges_offset(lay));
  prm.counters = reinterpret_cast<uint32_t*>(iws + kStatusBytes);
  prm.status = reinterpret_cast<uint32_t*>(iws);
  prm.item_count = h->graph ? reinterpret_cast<const int32_t*>(iws + kItemCountOffset) : nullptr;
  prm.indices = h->indices;
  prm.ckv = ckv_cache;
  prm.kpe = kpe_cache;
  prm.q_nope = q_nope;
  prm.q_pe = q_pe;
  prm.o = o;
  prm.lse = lse;
  prm.part_o = reinterpret_cast<float*>(fws);
  const int cph = h->mla_kernel->ctas_per_head_tile;
  prm.part_lse = reinterpret_cast<float*>(
      fws + part_lse_offset(lay, h->num_qo_heads * cph, h->head_dim / cph));
  prm.num_pages = num_pages;
  prm.num_heads = h->num_qo_heads;
  prm.gslices = h->plan.gslices;
  // the tcgen05 kernel runs as CTA pairs (one per head tile); the mma.sync kernel alone
  const int csize = h->mla_kernel->variant == kMlaTcgen05 ? 2 : 1;
  prm.page_size = h->page_size;
  prm.lse_base_e = lse_base_e ? 1 : 0;
  prm.scale_log2 = (float)((double)h->sm_scale * 1.4426950408889634);
  // CUDA-graph mode: the same grid for every plan (the capacity), CTAs past the count exit
  const int64_t grid =
      (h->graph ? (int64_t)h->g_max_items : (int64_t)h->plan.items.size()) * h->plan.gslices;
  void* args[] = {&prm};
  cudaError_t e;
  if (ev_start && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_start), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");
  {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(h->mla_kernel->threads);
    cfg.dynamicSmemBytes = (size_t)h->mla_kernel->smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = h->pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)csize;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelExC(&cfg, h->mla_kernel->fn, args);
  }
  if (e != cudaSuccess) return cuda_fail(e, "MLA decode kernel launch");
  if (ev_end && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_end), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord");
  return PKD_OK;
}

int pkd_mla_set_backend(pkd_handle* h, int backend) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (backend != PKD_MLA_BACKEND_AUTO && backend != PKD_MLA_BACKEND_MMA_SYNC &&
      backend != PKD_MLA_BACKEND_TCGEN05)
    return fail(PKD_ERR_INVALID_ARG, "backend must be PKD_MLA_BACKEND_AUTO, _MMA_SYNC or _TCGEN05");
  h->mla_backend = backend;
  return PKD_OK;
}

int pkd_set_pdl(pkd_handle* h, int enable) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  h->pdl = enable != 0;
  return PKD_OK;
}

int pkd_plan_info(pkd_handle* h, int* grid, int* ctas_per_sm, int64_t* n_tasks,
                  int64_t* n_merges) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (!h->planned || h->mla) return fail(PKD_ERR_NOT_PLANNED, "no decode plan on this handle");
  int per_sm = 0;
  if (int rc = decode_ctas_per_sm(h->kernel, h->device, &per_sm)) return rc;
  if (grid) *grid = h->grid;
  if (ctas_per_sm) *ctas_per_sm = per_sm;
  if (n_tasks) *n_tasks = h->n_tasks;
  if (n_merges) *n_merges = h->n_dmerges;
  return PKD_OK;
}

int pkd_set_wait_limit(pkd_handle* h, uint64_t limit_ns) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (limit_ns > kWaitLimitNs)
    return fail(PKD_ERR_INVALID_ARG, "the wait limit must lie in [0, 2e9] ns");
  h->wait_ns = limit_ns;
  return PKD_OK;
}

int pkd_check_page_table(const int32_t* indptr_host, int batch, const int32_t* indices_host,
                         int64_t num_indices, int64_t num_pages) {
  if (batch < 0 || (batch > 0 && (!indptr_host || (!indices_host && indptr_host[batch] > 0))))
    return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0 and the page table pointers non-null");
  if (batch == 0) return PKD_OK;
  if (indptr_host[0] < 0) return fail(PKD_ERR_INVALID_ARG, "indptr[0] must be >= 0");
  for (int i = 0; i < batch; ++i)
    if (indptr_host[i + 1] < indptr_host[i])
      return fail(PKD_ERR_INVALID_ARG, "indptr must be non-decreasing");
  if ((int64_t)indptr_host[batch] > num_indices)
    return fail(PKD_ERR_INVALID_ARG, "indices holds fewer than indptr[batch] page ids");
  for (int i = 0; i < batch; ++i)
    for (int32_t j = indptr_host[i]; j < indptr_host[i + 1]; ++j)
      if (indices_host[j] < 0 || (int64_t)indices_host[j] >= num_pages) {
        char buf[200];
        std::snprintf(buf, sizeof buf,
                      "request %d: page id %d at indices[%d] lies outside [0, %lld)", i,
                      (int)indices_host[j], (int)j, (long long)num_pages);
        return fail(PKD_ERR_INVALID_ARG, buf);
      }
  g_last_error.clear();
  return PKD_OK;
}

int pkd_enable_cuda_graph(pkd_handle* h, int32_t* indptr_buf, int32_t* indices_buf,
                          int32_t* last_page_len_buf, int max_batch, int64_t max_pages,
                          int max_items) {
  if (!h) return fail(PKD_ERR_INVALID_ARG, "handle is null");
  if (!indptr_buf || !indices_buf || !last_page_len_buf)
    return fail(PKD_ERR_INVALID_ARG, "CUDA-graph mode needs the indptr, indices and "
                                     "last_page_len buffers");
  if (!aligned(indptr_buf, 4) || !aligned(indices_buf, 4) || !aligned(last_page_len_buf, 4))
    return fail(PKD_ERR_INVALID_ARG, "graph buffers must be 4-byte aligned");
  if (max_batch < 1 || max_pages < 0)
    return fail(PKD_ERR_INVALID_ARG, "max_batch must be >= 1 and max_pages >= 0");
  if (max_items <= 0) max_items = max_batch + 2 * h->num_sms;
  if (max_items < max_batch)
    return fail(PKD_ERR_INVALID_ARG, "max_items must be >= max_batch");
  h->graph = true;
  h->g_indptr = indptr_buf;
  h->g_indices = indices_buf;
  h->g_lpl = last_page_len_buf;
  h->g_max_batch = max_batch;
  h->g_max_pages = max_pages;
  h->g_max_items = max_items;
  h->g_batch = -1;
  h->planned = false;
  return PKD_OK;
}

int pkd_graph_workspace_bytes(int max_items, int num_qo_heads, int num_kv_heads, int head_dim,
                              int use_tensor_cores, size_t* float_ws_bytes,
                              size_t* int_ws_bytes) {
  if (max_items < 1 || num_qo_heads <= 0 || num_kv_heads <= 0 ||
      num_qo_heads % num_kv_heads != 0 || head_dim <= 0)
    return fail(PKD_ERR_INVALID_ARG, "bad capacity or head configuration");
  const int G = num_qo_heads / num_kv_heads;
  int hpc = 8;  // heads per CTA: 8 on tensor cores, else the power of two >= G, at most 8
  if (use_tensor_cores == 0) {
    hpc = 2;
    while (hpc < G && hpc < 8) hpc <<= 1;
  }
  DecodeWsLayout lay = decode_capacity_layout(max_items, num_kv_heads, (G + hpc - 1) / hpc);
  lay.pos_floats = 2 * (size_t)head_dim + num_qo_heads;  // room for a positional encoding
  if (float_ws_bytes) *float_ws_bytes = dws_float_bytes(lay, head_dim);
  if (int_ws_bytes) *int_ws_bytes = dws_int_bytes(lay);
  return PKD_OK;
}

int pkd_mla_graph_workspace_bytes(int max_items, int num_heads, int backend,
                                  size_t* float_ws_bytes, size_t* int_ws_bytes) {
  if (max_items < 1 || num_heads <= 0)
    return fail(PKD_ERR_INVALID_ARG, "bad capacity or head count");
  if (backend != PKD_MLA_BACKEND_AUTO && backend != PKD_MLA_BACKEND_MMA_SYNC &&
      backend != PKD_MLA_BACKEND_TCGEN05)
    return fail(PKD_ERR_INVALID_ARG, "backend must be PKD_MLA_BACKEND_AUTO, _MMA_SYNC or _TCGEN05");
  const int variant = mla_variant_for(backend, num_heads);
  const MlaKernel* k = find_mla(kBF16, variant);
  if (!k) return fail(PKD_ERR_UNSUPPORTED, "no MLA kernel built");
  const int cph = k->ctas_per_head_tile;
  const int gslices = (num_heads + k->heads_per_cta - 1) / k->heads_per_cta * cph;
  const WsLayout lay = capacity_layout(max_items, 1, gslices);
  if (float_ws_bytes) *float_ws_bytes = float_ws_bytes_of(lay, num_heads * cph, 512 / cph);
  if (int_ws_bytes) *int_ws_bytes = int_ws_bytes_of(lay);
  return PKD_OK;
}

int pkd_check_status(pkd_handle* h, uint32_t* status, void* stream) {
  if (!status) return fail(PKD_ERR_INVALID_ARG, "status is null");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!h) return noalloc_check_status(status, s);  // pkd_decode_noalloc's built-in status word
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, h->int_ws, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  *status = v;
  if (v) {
    // A kernel that gave up may have left a split request's chunk counter part-way; zero the
    // counters with the status word so the next run of this plan merges at the right count.
    e = cudaMemsetAsync(h->int_ws, 0, sizeof v, s);
    const size_t counters_end = !h->planned ? kStatusBytes
                                : h->mla    ? items_offset(h->ws_layout)
                                            : dws_tasks_offset(h->dlayout);
    if (e == cudaSuccess && counters_end > kStatusBytes)
      e = cudaMemsetAsync(static_cast<char*>(h->int_ws) + kStatusBytes, 0,
                          counters_end - kStatusBytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  }
  return PKD_OK;
}

}  // extern "C"
