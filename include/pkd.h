/*
 * pkd.h -- C ABI of libpkd: batch decode attention over a paged KV cache on one GB300 GPU.
 *
 * The calls mirror the plan/run split of the FlashInfer attention API page
 * (docs.flashinfer.cn, api/attention.html), class BatchDecodeWithPagedKVCacheWrapper:
 *   - the constructor takes a user-owned float workspace for split-KV partial results and a
 *     KV layout (NHD or HND)                                  -> pkd_create
 *   - reset_workspace_buffer(float_ws, int_ws)                -> pkd_reset_workspace
 *   - plan(indptr, indices, last_page_len, num_qo_heads, num_kv_heads, head_dim, page_size,
 *          window_left, logits_soft_cap, q/kv/o data types, sm_scale, fixed_split_size,
 *          disable_split_kv) builds auxiliary data once and reuses it over many run calls
 *                                                             -> pkd_plan
 *   - run(q, paged_kv_cache, q_scale, k_scale, v_scale, out, lse) -> (o, lse)
 *                                                             -> pkd_run
 *
 * Conventions for every call:
 *   - All functions return PKD_OK (0) or a negative PKD_ERR_* code.  No exception, abort or
 *     exit crosses this boundary.  pkd_last_error() returns a message for the most recent
 *     failure on the calling thread.
 *   - "device" pointers are CUDA device (or managed) addresses on the current device;
 *     "host" pointers are ordinary CPU memory.  Every buffer is owned by the caller.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - dtype codes: PKD_DTYPE_F16 (IEEE half), PKD_DTYPE_BF16, PKD_DTYPE_E4M3 (fp8 e4m3fn,
 *     KV only).
 *
 * Semantics (the page fixes the shapes; these readings fill what it leaves open):
 *   kv_len[i] = page_size * (indptr[i+1] - indptr[i] - 1) + last_page_len[i]  (0 if the
 *   request has no page); token t of request i is slot t % page_size of page
 *   indices[indptr[i] + t / page_size]; qo head g reads kv head g / (Hq / Hkv);
 *   x_t = sm_scale * q_scale * k_scale * <q, K_t>; s_t = cap * tanh(x_t / cap) if cap > 0
 *   else x_t; the attended keys are t >= kv_len - 1 - window_left (all keys if
 *   window_left < 0); o = v_scale * sum_t softmax(s)_t V_t; lse = ln(sum_t exp(s_t)).
 *   A request with no attended key gets o = 0 and lse = -inf.
 */
#ifndef PKD_H_
#define PKD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKD_OK 0
#define PKD_ERR_INVALID_ARG (-1)         /* malformed table, shape, dtype or pointer */
#define PKD_ERR_NOT_PLANNED (-2)         /* pkd_run before a successful pkd_plan */
#define PKD_ERR_WORKSPACE_TOO_SMALL (-3) /* see pkd_workspace_bytes */
#define PKD_ERR_CUDA (-4)                /* a CUDA runtime/driver call failed */
#define PKD_ERR_UNSUPPORTED (-5)         /* valid but not built (head_dim, page_size, dtypes) */
#define PKD_ERR_DEVICE (-6)              /* a kernel reported an error in the status word */

/* Bits of the device status word (pkd_check_status). */
#define PKD_STATUS_TIMEOUT 1u  /* a pipeline wait ran out: the kernel gave up, outputs incomplete */
#define PKD_STATUS_BAD_PAGE 2u /* a page id outside [0, num_pages) was read (as zeros) */

#define PKD_DTYPE_F16 0
#define PKD_DTYPE_BF16 1
#define PKD_DTYPE_E4M3 2

#define PKD_LAYOUT_NHD 0 /* page block [page_size, num_kv_heads, head_dim] */
#define PKD_LAYOUT_HND 1 /* page block [num_kv_heads, page_size, head_dim] */

/* pkd_plan's pos_encoding_mode (the page's pos_encoding_mode NONE / ROPE_LLAMA / ALIBI). */
#define PKD_POS_NONE 0
#define PKD_POS_ROPE_LLAMA 1
#define PKD_POS_ALIBI 2

/* Kernel choice for pkd_plan's use_tensor_cores argument (the page's use_tensor_cores).
 * AUTO takes the tensor-core kernel (mma.sync, 8 qo heads per task), measured at least as
 * fast as the CUDA-core kernel (fp32 FMAs, 1 to 8 qo heads per task) at every GQA group. */
#define PKD_KERNEL_AUTO (-1)
#define PKD_KERNEL_CUDA_CORE 0
#define PKD_KERNEL_TENSOR_CORE 1

typedef struct pkd_handle pkd_handle;

/*
 * Create a handle.  float_ws (device, >= 256-byte aligned) receives split-KV partial
 * outputs and lses; int_ws (device, >= 256-byte aligned) receives the work list, the merge
 * list and a device status word.  Their needed sizes depend on the plan
 * (pkd_workspace_bytes); 128 MiB of float workspace covers every plan whose split slots
 * times num_qo_heads times head_dim stays under 32 M floats.  kv_layout: PKD_LAYOUT_*.
 * The handle keeps the pointers; the caller keeps the buffers alive until pkd_destroy.
 */
int pkd_create(pkd_handle** out, void* float_ws, size_t float_ws_bytes, void* int_ws,
               size_t int_ws_bytes, int kv_layout);

/* Replace both workspaces (FlashInfer's reset_workspace_buffer).  Drops the current plan. */
int pkd_reset_workspace(pkd_handle* h, void* float_ws, size_t float_ws_bytes, void* int_ws,
                        size_t int_ws_bytes);

/*
 * Plan a batch.  Host work O(batch + chunks), then one asynchronous host->device copy of
 * the work list into int_ws on `stream`.  Not capturable in a CUDA graph.
 *   indptr_host [batch+1], last_page_len_host [batch]: host int32 copies of the page table
 *     (indptr non-decreasing from 0; 1 <= last_page_len <= page_size for requests that have
 *     pages; ignored for requests without pages).
 *   indices_dev [num_indices]: device int32 physical page ids, num_indices >= indptr[batch].
 *     The pointer is stored and read by every later pkd_run: keep it valid and unchanged.
 *     Ids outside [0, num_pages) read zeros (the hardware bounds-checks them) and set
 *     PKD_STATUS_BAD_PAGE in the status word; pkd_check_page_table checks a host copy of
 *     the table up front.
 *   num_qo_heads must be a multiple of num_kv_heads.  head_dim in {64, 128, 256}
 *   (e4m3 KV: {128, 256}).  page_size a power of two in [8, 256].
 *   sm_scale: NaN selects 1/sqrt(head_dim).  logits_soft_cap <= 0: no cap.
 *   window_left < 0: no window.  fixed_split_size > 0: split every request into chunks of
 *   that many pages counted from its first page, so the result of a request does not depend
 *   on the rest of the batch; disable_split_kv != 0: one chunk per request; otherwise a
 *   heuristic sizes chunks to fill the GPU.
 *   q_dtype / o_dtype: F16 or BF16, equal; kv_dtype: q_dtype or E4M3.
 *   use_tensor_cores: PKD_KERNEL_AUTO, PKD_KERNEL_CUDA_CORE or PKD_KERNEL_TENSOR_CORE.
 *   q_len_per_req >= 1 (the page's run(q_len_per_req), fixed here because the work list
 *     depends on it): query tokens per request.  They are the request's last positions:
 *     token j of a request with kv_len n sits at n - q_len + j and attends the keys up to its
 *     own position (causal inside the request) and its own window.  q, o and lse then have
 *     batch * q_len_per_req rows, request-major (row = request * q_len_per_req + j).
 *   pos_encoding_mode (the page's NONE / ROPE_LLAMA / ALIBI, with rope_scale and rope_theta,
 *     the page's defaults 1 and 1e4; both ignored unless ROPE_LLAMA):
 *     PKD_POS_ROPE_LLAMA rotates q (at its position) and each key (at its token index) in
 *       pairs of dims (i, i + head_dim/2) by the angle pos / rope_scale * rope_theta^(-2i/D)
 *       before the dot product.  The tensor-core kernel rounds the rotated q and K to fp16
 *       for the product; the CUDA-core kernel rotates and multiplies in fp32.
 *       Angles are accurate to ~1e-6 rad for positions below 2^24.
 *     PKD_POS_ALIBI adds slope_g * (t - pos) to the scaled logit of qo head g (before the soft
 *       cap), with the ALiBi paper's slopes 2^(-8 (g+1) / m) for the largest power of two
 *       m <= num_qo_heads and 2^(-4 (2 (g-m) + 1) / m) for the heads beyond m.
 * Errors: INVALID_ARG (shapes, table), UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA.
 */
int pkd_plan(pkd_handle* h, const int32_t* indptr_host, const int32_t* last_page_len_host,
             int batch, const int32_t* indices_dev, int64_t num_indices, int num_qo_heads,
             int num_kv_heads, int head_dim, int page_size, float sm_scale,
             float logits_soft_cap, int window_left, int fixed_split_size,
             int disable_split_kv, int q_dtype, int kv_dtype, int o_dtype,
             int use_tensor_cores, int q_len_per_req, int pos_encoding_mode, float rope_scale,
             float rope_theta, void* stream);

/*
 * Run the planned batch on one layer's KV pool.  Asynchronous on `stream`; never syncs.
 *   q (device) [batch * q_len_per_req, num_qo_heads, head_dim], contiguous, q_dtype.
 *   k_base / v_base (device): element (page, slot, head, 0) of K / V lives at
 *     base + page*kv_strides[0] + slot*kv_strides[1] + head*kv_strides[2] (elements of
 *     kv_dtype, head_dim contiguous).  A 5-D pool [pages, 2, ...] passes v_base =
 *     k_base + its K/V stride; a (k_cache, v_cache) pair passes the two tensors.  Bases must
 *     be 16-byte aligned and the strides multiples of 16 bytes.  The two inner strides must
 *     match the handle's layout (NHD: slot stride > head stride; HND: the reverse).
 *   num_pages: pages in the pool (the extent of the page axis).
 *   q_scale, k_scale, v_scale: calibration scales (1.0 when unused).
 *   o (device) [batch * q_len_per_req, num_qo_heads, head_dim] o_dtype; lse (device)
 *     [batch * q_len_per_req, num_qo_heads] float32 natural log, or NULL to skip it.
 * Launches one decode kernel; the CTA that finishes a split request's last chunk merges the
 * request's partial results inside that launch.
 */
int pkd_run(pkd_handle* h, const void* q, const void* k_base, const void* v_base,
            int64_t num_pages, const int64_t kv_strides[3], float q_scale, float k_scale,
            float v_scale, void* o, float* lse, void* stream);

/* Same as pkd_run, and records ev_start / ev_end (cudaEvent_t as void*, may be NULL)
 * immediately before and after the decode kernel's launch, so a caller can time that
 * kernel alone on its own stream. */
int pkd_run_timed(pkd_handle* h, const void* q, const void* k_base, const void* v_base,
                  int64_t num_pages, const int64_t kv_strides[3], float q_scale,
                  float k_scale, float v_scale, void* o, float* lse, void* stream,
                  void* ev_start, void* ev_end);

/*
 * Programmatic dependent launch (the page's run(enable_pdl=...)), on by default.  When on, the
 * decode kernel is launched with programmatic stream serialization: the GPU may schedule it
 * while the previous kernel in the stream is still finishing, and the kernel waits
 * (griddepcontrol.wait) before it reads anything, so results are the same either way; only
 * the launch gap is hidden.  Off: ordinary stream order.
 */
int pkd_set_pdl(pkd_handle* h, int enable);

/*
 * CUDA-graph mode: the page's BatchDecodeWithPagedKVCacheWrapper(use_cuda_graph=True,
 * paged_kv_indptr_buffer, paged_kv_indices_buffer, paged_kv_last_page_len_buffer),
 * CUDAGraphBatchDecodeWithPagedKVCacheWrapper(workspace, indptr_buffer, indices_buffer,
 * last_page_len_buffer) and BatchMLAPagedAttentionWrapper(use_cuda_graph=True, ...,
 * kv_indptr, kv_indices, kv_len_arr).  After this call (it cannot be undone on the handle):
 *   - pkd_plan copies the page table into the caller's device buffers (indptr_buf: >=
 *     max_batch + 1 int32, indices_buf: >= max_pages int32, last_page_len_buf: >= max_batch
 *     int32) and the kernel reads page ids from indices_buf;
 *   - the batch size is fixed by the first plan (a shorter batch is padded with zero-length
 *     requests: repeat the last indptr value; their o rows are 0 and lse -inf);
 *   - the work list holds at most max_items chunks (<= 0: max_batch + 2 x the SM count); the
 *     heuristic split grows its chunks to fit, a fixed_split_size that does not fit fails with
 *     PKD_ERR_WORKSPACE_TOO_SMALL; the workspaces must hold pkd_graph_workspace_bytes;
 *   - pkd_run launches the same grid with the same kernel arguments for every plan (CTAs past
 *     the plan's chunk count exit at once), so a run captured in a CUDA graph replays
 *     correctly after later plans.  pkd_plan itself is not capturable, as the page notes for
 *     plan().
 *   - MLA (pkd_mla_plan / pkd_mla_run) works the same way: last_page_len_buf receives
 *     kv_len; the first plan also fixes num_heads, page_size, sm_scale, the dtype and the
 *     kernel; the workspaces must hold pkd_mla_graph_workspace_bytes.  A handle holds decode
 *     plans or MLA plans in this mode, not both.
 * The buffers are the caller's and must outlive every run.
 */
int pkd_enable_cuda_graph(pkd_handle* h, int32_t* indptr_buf, int32_t* indices_buf,
                          int32_t* last_page_len_buf, int max_batch, int64_t max_pages,
                          int max_items);

/* Workspace bytes CUDA-graph mode needs for a work list of max_items chunks. */
int pkd_graph_workspace_bytes(int max_items, int num_qo_heads, int num_kv_heads, int head_dim,
                              int use_tensor_cores, size_t* float_ws_bytes,
                              size_t* int_ws_bytes);
/* The same for MLA plans of num_heads heads on the kernel `backend` (PKD_MLA_BACKEND_*) picks. */
int pkd_mla_graph_workspace_bytes(int max_items, int num_heads, int backend,
                                  size_t* float_ws_bytes, size_t* int_ws_bytes);

/*
 * MLA paged decode: the page's flashinfer.mla.BatchMLAPagedAttentionWrapper plan() / run()
 * (decode: qo_indptr = 0, 1, ..., batch, one query per request).  With matrix absorption all
 * num_heads query heads attend over one latent cache: key of token t = [ckv_t, kpe_t],
 * value = ckv_t, logit = sm_scale * (<q_nope, ckv_t> + <q_pe, kpe_t>).
 * pkd_mla_plan:
 *   kv_indptr_host [batch+1] (non-decreasing), kv_len_host [batch] (0 <= kv_len <= pages *
 *     page_size; extra pages are ignored): host int32.  kv_indices_dev [num_indices >=
 *     kv_indptr[batch]]: device int32 page ids, stored and read by later runs.
 *   head_dim_ckv must be 512 and head_dim_kpe 64 (the DeepSeek shapes the page names);
 *   page_size >= 1 (any integer, 1 included); sm_scale > 0 (the page's example uses
 *   1 / sqrt(128 + 64)); q_dtype == kv_dtype in {F16, BF16}; causal is accepted and has no
 *   effect with one query per request.  The handle then holds an MLA plan: pkd_run refuses
 *   it, pkd_mla_run refuses a pkd_plan plan.  pkd_mla_plan is not capturable; in CUDA-graph
 *   mode (pkd_enable_cuda_graph) pkd_mla_run is.
 * pkd_mla_run:
 *   q_nope [batch, num_heads, 512], q_pe [batch, num_heads, 64]; ckv_cache [num_pages,
 *   page_size, 512], kpe_cache [num_pages, page_size, 64] (all device, contiguous, 16-byte
 *   aligned); a page id outside [0, num_pages) reads as a zero row (logit 0, value 0).  o [batch, num_heads, 512];
 *   lse [batch, num_heads] float32 or NULL, base 2 unless lse_base_e (the page's
 *   return_lse_base_on_e).  ev_start / ev_end (cudaEvent_t or NULL) are recorded around the
 *   kernel.  One launch; split requests are merged inside it.
 */
int pkd_mla_plan(pkd_handle* h, const int32_t* kv_indptr_host, const int32_t* kv_len_host,
                 int batch, const int32_t* kv_indices_dev, int64_t num_indices, int num_heads,
                 int head_dim_ckv, int head_dim_kpe, int page_size, int causal, float sm_scale,
                 int q_dtype, int kv_dtype, void* stream);
int pkd_mla_run(pkd_handle* h, const void* q_nope, const void* q_pe, const void* ckv_cache,
                const void* kpe_cache, int64_t num_pages, void* o, float* lse, int lse_base_e,
                void* stream, void* ev_start, void* ev_end);

/*
 * MLA kernel used by later pkd_mla_plan calls on this handle (the wrapper's backend argument):
 *   PKD_MLA_BACKEND_AUTO      the tcgen05 kernel when num_heads > 32, else the mma.sync kernel;
 *   PKD_MLA_BACKEND_MMA_SYNC  32 heads per CTA, mma.sync with register accumulators;
 *   PKD_MLA_BACKEND_TCGEN05   128 heads per 2-CTA cluster (the pair splits the 576 features),
 *                             tcgen05 MMAs with accumulators in tensor memory.
 * Both compute the same result within rounding.  PKD_ERR_INVALID_ARG for other values.
 */
#define PKD_MLA_BACKEND_AUTO 0
#define PKD_MLA_BACKEND_MMA_SYNC 1
#define PKD_MLA_BACKEND_TCGEN05 2
int pkd_mla_set_backend(pkd_handle* h, int backend);

/*
 * Host-only MLA planning (no GPU, no handle): the work list pkd_mla_plan would upload for this
 * batch with this backend, for inspection and tests.  kv_indptr_host / kv_len_host as in
 * pkd_mla_plan; dtype PKD_DTYPE_F16 or _BF16; num_sms <= 0 means 152.  items_out receives up
 * to max_items work items of 8 int32 (output row, offset of the request's first page id,
 * first token of the chunk's first tile, attended begin, attended end, partial slot or -1,
 * merge entry or -1, query position) and merges_out up to max_merges entries of 4 int32
 * (row, first slot, chunk count, 0); either may be NULL.  n_items / n_merges / n_slots receive
 * the counts, ctas_per_item the CTAs each item launches, float_ws_bytes / int_ws_bytes the
 * workspace sizes pkd_mla_plan needs (any of them may be NULL).
 */
int pkd_mla_plan_host(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int batch,
                      int num_heads, int page_size, int dtype, int backend, int num_sms,
                      int32_t* items_out, int max_items, int32_t* merges_out, int max_merges,
                      int* n_items, int* n_merges, int* n_slots, int* ctas_per_item,
                      size_t* float_ws_bytes, size_t* int_ws_bytes);

/* Free the handle (host memory and pinned staging only; the workspaces are the caller's). */
int pkd_destroy(pkd_handle* h);

/* Message of the last failure on this thread ("" if none).  Valid until the next call. */
const char* pkd_last_error(void);

/*
 * Workspace bytes a plan with these arguments needs (host-only; no CUDA call).  Arguments
 * as in pkd_plan; num_sms is the SM count the heuristic assumes (0 = 152).
 */
int pkd_workspace_bytes(const int32_t* indptr_host, const int32_t* last_page_len_host,
                        int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                        int page_size, int window_left, int fixed_split_size,
                        int disable_split_kv, int kv_dtype, int use_tensor_cores, int num_sms,
                        int q_len_per_req, size_t* float_ws_bytes, size_t* int_ws_bytes);

/*
 * The decode planner alone (host-only; no CUDA call), for inspection and tests.  The plan
 * is a list of tasks for a persistent grid of num_sms x 2 CTAs (num_sms <= 0 means 152): a
 * task is a chunk of one output row's attended tokens for one kv head and one slice of its
 * qo-head group (8 qo heads on the tensor-core kernel).  Writes up to max_tasks tasks of 12
 * int32 each:
 *   {output row, first page index into `indices`, first token of the chunk's first tile,
 *    first attended token, end token, partial slot (-1 = final), merge entry (-1 = none),
 *    query position, kv head, slice, CTA, 0}
 *   (tokens count from the request's start), grouped by CTA in the order each CTA runs them,
 * and up to max_merges merge entries of 4 int32 {row, first slot, chunk count, unit} (unit =
 * kv head x slices + slice).  n_tasks / n_merges / n_slots / n_ctas receive the full counts
 * (n_ctas: CTAs with at least one task).  kernel_out receives the chosen PKD_KERNEL_* and
 * tile_tokens_out the tokens per pipeline stage.  work_capacity > 0 bounds the work list the
 * way CUDA-graph mode does (pkd_enable_cuda_graph's max_items, chunks per row summed over
 * rows); 0 leaves it unbounded.
 */
int pkd_plan_host(const int32_t* indptr_host, const int32_t* last_page_len_host, int batch,
                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                  int window_left, int fixed_split_size, int disable_split_kv, int kv_dtype,
                  int use_tensor_cores, int num_sms, int32_t* tasks_out, int max_tasks,
                  int32_t* merges_out, int max_merges, int* n_tasks, int* n_merges,
                  int* n_slots, int* kernel_out, int* tile_tokens_out, int work_capacity,
                  int q_len_per_req, int* n_ctas);

/*
 * Read and clear the device status word (synchronises `stream`).  *status receives 0 if no
 * kernel since the last plan or check reported a problem, else PKD_STATUS_* bits:
 *   PKD_STATUS_TIMEOUT   a pipeline wait ran out (pkd_set_wait_limit): the CTAs that gave up
 *                        wrote none of their outputs, and every later launch on this handle
 *                        returns at once, writing nothing, until this call clears the bit;
 *   PKD_STATUS_BAD_PAGE  a decode launch read a page id outside [0, num_pages) (read as zeros;
 *                        later launches are not affected).
 * When it is nonzero, the split-merge chunk counters in the int workspace are zeroed with it,
 * so later runs of the same plan start clean.
 * h == NULL reads and clears the status word of pkd_decode_noalloc's built-in scratch on the
 * current device instead (the status of the last pkd_decode_noalloc call there).
 */
int pkd_check_status(pkd_handle* h, uint32_t* status, void* stream);

/*
 * The current decode plan's launch shape: *grid receives the CTAs pkd_run launches (the
 * persistent grid, or in CUDA-graph mode the fixed one), *ctas_per_sm the CTAs of the plan's
 * kernel one SM holds, *n_tasks / *n_merges the tasks and split units (any may be NULL).
 * NOT_PLANNED without a decode plan.
 */
int pkd_plan_info(pkd_handle* h, int* grid, int* ctas_per_sm, int64_t* n_tasks,
                  int64_t* n_merges);

/*
 * Limit of the decode kernel's pipeline waits (a consumer waiting for a tile's copies, the
 * producer waiting for a free stage) for later pkd_run calls on this handle, in ns; the
 * default and largest value is 2e9 (2 s).  A wait that runs out sets PKD_STATUS_TIMEOUT and
 * the CTA gives up (see pkd_check_status).  0 makes every wait test its barrier once and give
 * up if the tile is not already there; it exists to exercise that failure path.  A CTA that
 * gives up still waits, with the full 2 s limit, for the copies it has already issued to
 * land before it exits.  INVALID_ARG above 2e9.
 */
int pkd_set_wait_limit(pkd_handle* h, uint64_t limit_ns);

/*
 * Optional host validation of a page table (no handle, no CUDA call): indptr_host [batch+1]
 * non-decreasing from indptr[0] >= 0, indptr[batch] <= num_indices, and every page id a
 * request owns (indices_host[indptr[0] .. indptr[batch])) inside [0, num_pages).  Returns
 * PKD_OK or PKD_ERR_INVALID_ARG with a message naming the first offending request and id.
 * The kernels themselves read such ids as zeros and report PKD_STATUS_BAD_PAGE.
 */
int pkd_check_page_table(const int32_t* indptr_host, int batch, const int32_t* indices_host,
                         int64_t num_indices, int64_t num_pages);

/*
 * pkd_decode_noalloc -- plan + run in one call, using only scratch memory built into the
 * library.  The FlashInfer pages have no counterpart of this call.
 *
 * Who it is for: callers that cannot allocate device memory and have no workspace to lend.
 * A runtime that owns every device allocation (a fixed memory pool, or a hard memory budget
 * shared with other engines) does not let its plug-ins call cudaMalloc: an allocation outside
 * the pool can fail at any point, and it hides memory from the runtime's accounting.  Such a
 * caller passes only its inputs and outputs.
 *
 * Scratch: one file-scope device array of PKD_NOALLOC_SCRATCH_BYTES (16 MiB) inside libpkd.
 * Every GPU that loads the library holds it until the process exits.  It holds the status
 * word, the work list (at most PKD_NOALLOC_MAX_ITEMS chunks and PKD_NOALLOC_MAX_MERGES split
 * requests) and the split partials (4 * slots * num_qo_heads * (head_dim + 1) bytes, at most
 * PKD_NOALLOC_PARTIAL_BYTES).  A plan that needs more fails with PKD_ERR_WORKSPACE_TOO_SMALL
 * and a message saying which limit it hit.  With neither fixed_split_size nor
 * disable_split_kv set, the chunk size grows until the partials fit.
 *
 * A call allocates nothing: no cudaMalloc / cudaFree, no pinned or heap memory (the plan is
 * built in static host storage).  The first call on a device does a one-time set-up with that
 * device current: it reads the array's device address (cudaGetSymbolAddress) and raises the
 * kernels' shared-memory limit.
 *
 * Failures on the GPU: the call's kernels report into the status word at the start of the
 * array, which every call clears first.  pkd_check_status(NULL, &status, stream) reads and
 * clears it after the call (PKD_STATUS_TIMEOUT: a pipeline wait ran out and o / lse are
 * incomplete; PKD_STATUS_BAD_PAGE: a page id outside [0, num_pages) was read as zeros).
 *
 * Every call shares the one array and overwrites what the last call left there.  Calls whose
 * GPU work overlaps (on two streams, or from two host threads) race and corrupt each other's
 * results: serialise them.  The work list is uploaded from pageable host memory, so the call
 * waits for earlier work on `stream` before it returns.
 *
 * Arguments: those of pkd_plan followed by those of pkd_run, with kv_layout as in pkd_create.
 * Only the tensor-core kernel is built into this variant: use_tensor_cores must be
 * PKD_KERNEL_AUTO or PKD_KERNEL_TENSOR_CORE, and a kv head may serve at most 8 qo heads.
 * Returns PKD_OK or a PKD_ERR_* code (a failing call may allocate to format its message).
 */
#define PKD_NOALLOC_SCRATCH_BYTES (16u << 20)
#define PKD_NOALLOC_MAX_ITEMS 24576
#define PKD_NOALLOC_MAX_MERGES 16384
#define PKD_NOALLOC_PARTIAL_BYTES ((16u << 20) - (2u << 20))
int pkd_decode_noalloc(const int32_t* indptr_host, const int32_t* last_page_len_host, int batch,
                       const int32_t* indices_dev, int64_t num_indices, int num_qo_heads,
                       int num_kv_heads, int head_dim, int page_size, float sm_scale,
                       float logits_soft_cap, int window_left, int fixed_split_size,
                       int disable_split_kv, int q_dtype, int kv_dtype, int o_dtype,
                       int use_tensor_cores, int kv_layout, const void* q, const void* k_base,
                       const void* v_base, int64_t num_pages, const int64_t kv_strides[3],
                       float q_scale, float k_scale, float v_scale, void* o, float* lse,
                       void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H_ */
