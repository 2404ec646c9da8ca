// pkd_internal.h -- types shared by the host API/planner and the kernel translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (a 128-byte opaque descriptor; no driver call is made here)
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace pkd {

// One CTA-group of work: a chunk of one output row's KV tokens (a row is one query token of
// one request; with one query token per request, the request).  Tokens count from the
// request's first token.  The chunk covers pages starting at chunk_tok0 / page_size; the
// attended tokens of the chunk are [tok_begin, tok_end).  out_slot < 0 means the chunk is
// the whole request and the kernel writes the final o / lse; otherwise it writes an fp32
// partial into slot out_slot of the float workspace.
struct WorkItem {
  int32_t req;         // output row: q / o / lse row index
  int32_t page_base;   // indptr[request]: offset of the request's first page id in `indices`
  int32_t chunk_tok0;  // first token of the chunk's first page
  int32_t tok_begin;
  int32_t tok_end;
  int32_t out_slot;
  int32_t merge_idx;   // index of the request's MergeEntry when out_slot >= 0, else -1
  int32_t q_pos;       // the row's query position (its last key, n - 1): ALiBi / RoPE
};
static_assert(sizeof(WorkItem) == 32, "WorkItem is 8 int32");

// A request whose chunks wrote partials into slots [first_slot, first_slot + n_chunks).
struct MergeEntry {
  int32_t req;
  int32_t first_slot;
  int32_t n_chunks;
  int32_t pad;
};
static_assert(sizeof(MergeEntry) == 16, "MergeEntry is 4 int32");

// One task of the persistent decode kernel: a chunk of one output row's attended tokens for
// one kv head and one slice of that head's qo-head group (at most 8 qo heads).  The fields up
// to q_pos mean what they mean in a WorkItem.  A CTA runs a list of tasks back to back.
struct DecodeTask {
  int32_t req;         // output row: q / o / lse row index
  int32_t page_base;   // indptr[request]: offset of the request's first page id in `indices`
  int32_t chunk_tok0;  // first token of the chunk's first tile (a page boundary)
  int32_t tok_begin;   // attended tokens [tok_begin, tok_end)
  int32_t tok_end;
  int32_t out_slot;    // < 0: the task is the whole row for its heads (final o / lse);
                       // else its fp32 partial goes to slot out_slot
  int32_t merge_idx;   // the merge entry of the task's (row, kv head, slice) when split
  int32_t q_pos;       // the row's query position (its last key): ALiBi / RoPE
  int32_t kvh;         // kv head
  int32_t gs;          // slice of the kv head's qo-head group
  int32_t cta;         // the CTA that runs it
  int32_t pad;
};
static_assert(sizeof(DecodeTask) == 48, "DecodeTask is 12 int32");

// Rows of one partial slot: the qo heads of one task (a slice holds at most 8).
constexpr int kSlotHeads = 8;

enum DType { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Default (and largest) limit of a kernel's pipeline waits, in ns of the global timer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Reads and clears the status word of pkd_decode_noalloc's built-in scratch on the current
// device (noalloc.cu), for pkd_check_status(NULL, ...).
int noalloc_check_status(uint32_t* status, cudaStream_t stream);
enum KernelKind { kCudaCore = 0, kTensorCore = 1 };

// Kernel parameters, passed by value as a __grid_constant__ so the tensor maps stay in
// parameter space (where the TMA unit may read them).
struct DecodeParams {
  CUtensorMap tmap_k;  // 4-D view of the K pool, see make_kv_tensor_map
  CUtensorMap tmap_v;
  const DecodeTask* tasks;   // CTA c runs task c (longest first)
  const int32_t* task_count; // CUDA-graph mode: the plan's task count, read on the device (the
                             // grid is cut for a fixed capacity); null: the grid is exact
  const int32_t* indices;
  const void* q;        // [batch, Hq, D] q dtype
  void* o;              // [batch, Hq, D] o dtype
  float* lse;           // [batch, Hq] natural log, may be null
  float* part_o;        // [slots, kSlotHeads, D] fp32, normalised partial outputs
  float* part_lse;      // [slots, kSlotHeads] fp32, base-2 log-sum-exp of the partial
  uint32_t* status;     // device status word (bit 0: a pipeline wait timed out)
  const MergeEntry* merges;  // the split (row, kv head, slice) units: slots and chunk counts
  uint32_t* counters;   // finished chunks per merge entry (the last one merges)
  // Positional-encoding table (plan's pos_encoding_mode), in the int workspace, 256-byte
  // aligned: [head_dim / 2] x {rate hi, rate lo} for the RoPE angle rate
  // rope_theta^(-2i/D) / rope_scale (a float pair), and from float 2 * head_dim the
  // [num_qo_heads] ALiBi slopes in score units.  Null without an encoding.
  const float* pos_table;
  unsigned long long wait_ns;  // limit of every pipeline wait (0: test once); the wait for
                               // copies in flight before a CTA exits keeps its own 2 s limit
  uint32_t num_pages;   // pages in the pool: an id outside [0, num_pages) sets status bit 1
                        // (the load itself reads zeros: the tensor map bounds-checks it)
  int alibi;            // 1: add pos_table[qo head] * (t - q_pos) to every logit
  int num_qo_heads;
  int num_kv_heads;
  int group;            // Hq / Hkv
  int page_size;
  int hnd;              // 1: the tensor map's dims are (d, slot, head, page); 0: (d, head, slot, page)
  float scale_qk;       // multiplies <q, k>: sm_scale*q_scale*k_scale, times log2(e) without a
                        // cap or divided by the cap with one
  float cap_log2;       // cap * log2(e), 0 = no cap
  float v_scale;
};

// A compiled decode kernel and how to launch it.
struct DecodeKernel {
  int kind;         // KernelKind
  int q_dtype;      // DType of q and o
  int kv_dtype;     // DType of K/V
  int head_dim;
  int heads_per_cta;  // qo heads one CTA serves (the CUDA-core kernel is built per power of 2)
  const void* fn;
  int threads;
  int smem_bytes;   // dynamic shared memory
  int tile_tokens;  // tokens per pipeline stage
  int rope;         // 1: rotates q and K (ROPE_LLAMA) before the QK product
  int nstages;      // pipeline stages
};

// Registries filled by the kernel translation units.
void register_decode_f16(std::vector<DecodeKernel>& out);
void register_decode_bf16(std::vector<DecodeKernel>& out);
void register_decode_e4m3(std::vector<DecodeKernel>& out);
void register_decode_rope(std::vector<DecodeKernel>& out);
void register_decode_rope_cc(std::vector<DecodeKernel>& out);
void register_decode_rope_cc_e4m3(std::vector<DecodeKernel>& out);

// MLA decode kernel parameters (pkd_mla_run -> mla_decode_kernel).
struct MlaParams {
  const WorkItem* items;
  const int32_t* indices;
  const void* ckv;        // [pages, page_size, 512]
  const void* kpe;        // [pages, page_size, 64]
  const void* q_nope;     // [rows, H, 512]
  const void* q_pe;       // [rows, H, 64]
  void* o;                // [rows, H, 512]
  float* lse;             // [rows, H] or null
  float* part_o;          // [slots, H, 512] fp32, normalised
  float* part_lse;        // [slots, H] fp32, base 2
  uint32_t* status;
  const MergeEntry* merges;
  uint32_t* counters;     // per (merge entry, head slice)
  const int32_t* item_count;  // CUDA-graph mode: the plan's item count, read on the device (the
                              // grid is cut for a fixed capacity); null: the grid is exact
  int64_t num_pages;      // pages in the caches: ids outside [0, num_pages) read as zeros
  int num_heads;
  int gslices;            // CTAs per item: head tiles x CTAs per head tile
  int page_size;
  int lse_base_e;         // 1: lse as natural log, 0: base 2 (run()'s default)
  float scale_log2;       // sm_scale * log2(e)
};

// MLA decode kernels, latent 512 + rope 64, one per q / cache dtype and variant:
//   kMlaMmaSync (mla.cu): 32 heads per CTA, mma.sync, register accumulators;
//   kMlaTcgen05 (mla_tc.cu): 128 heads per CTA pair (a 2-CTA cluster splitting the features),
//   tcgen05 MMAs with TMEM accumulators.
enum MlaVariant { kMlaAuto = 0, kMlaMmaSync = 1, kMlaTcgen05 = 2 };
struct MlaKernel {
  int dtype;
  int variant;
  const void* fn;
  int threads;
  int smem_bytes;
  int heads_per_cta;
  int tile_tokens;
  int ctas_per_head_tile;  // CTAs sharing one head tile (each with its own lse partials)
};
void register_mla(std::vector<MlaKernel>& out);
void register_mla_tc(std::vector<MlaKernel>& out);

// ----------------------------------------------------------------------------- planner
struct PlanRequest {
  const int32_t* indptr;
  const int32_t* last_page_len;
  int batch;
  int num_qo_heads;
  int num_kv_heads;
  int head_dim;
  int page_size;
  int window_left;
  int fixed_split_size;
  int disable_split_kv;
  int kv_dtype;
  int use_tensor_cores;  // -1 auto, 0, 1
  int num_sms;
  int max_items = 0;     // > 0: the work list may hold at most this many items (CUDA-graph mode;
                         // for decode: chunks per row, counted over all rows)
  int q_len = 1;         // query tokens per request (run's q_len_per_req)
  int rope = 0;          // 1: ROPE_LLAMA
  // MLA plans (pkd_mla_plan): lengths come from kv_len (pages may be more than needed), any
  // page size >= 1, a fixed head tile and token tile, and the kernel's CTAs per SM.
  const int32_t* kv_len = nullptr;
  int mla = 0;
  int mla_heads_per_cta = 32;
  int mla_tile_tokens = 32;
  int mla_ctas_per_head_tile = 1;
  int ctas_per_sm = 2;
};

struct Plan {
  std::vector<WorkItem> items;
  std::vector<MergeEntry> merges;
  int num_slots = 0;
  int kind = kTensorCore;
  int heads_per_cta = 8;
  int gslices = 1;
  int tile_tokens = 64;
  int64_t chunk_tokens = 0;  // 0 = no split
};

// Returns 0 or a PKD_ERR_* code with a message in *err.  MLA plans (r.mla) only.
int build_plan(const PlanRequest& r, Plan* plan, const char** err);

// ----------------------------------------------------------------------- decode schedule
// The decode planner's output, written into storage the caller provides (it allocates
// nothing: the no-allocation entry point passes static arrays, the handle path vectors).
// One chunk of one row: [b, e) of its attended tokens (tiles from tile0), chunk q of k; when
// the row is split (k > 1), unit u of the row takes partial slots slot_base + u k .. + k - 1 and
// merge entry merge_base + u.
struct DecodeChunk {
  int32_t row, b, e, tile0, q, k, slot_base, merge_base;
};

struct DecodeSchedule {
  DecodeTask* tasks = nullptr;  // capacity tasks_cap; task q runs on CTA q (longest first)
  int64_t tasks_cap = 0;
  MergeEntry* merges = nullptr;  // capacity merges_cap; {row, first slot, chunks, unit}
  int64_t merges_cap = 0;
  DecodeChunk* chunks = nullptr;  // scratch, capacity chunks_cap
  int64_t chunks_cap = 0;
  int64_t max_slots = 0;         // > 0: at most this many partial slots
  // results
  int64_t n_tasks = 0, n_merges = 0, n_slots = 0, n_chunks = 0;
  // set with PKD_ERR_WORKSPACE_TOO_SMALL when only the storage above was too small: the
  // counts then hold what the plan needs, and a call with that much storage succeeds
  bool storage_short = false;
  int kind = kTensorCore, heads_per_cta = 8, gslices = 1, tile_tokens = 64;
};

// Kernel geometry a decode plan implies (kind, heads per CTA, slices, tile) and validation of
// the request.  Returns 0 or a PKD_ERR_* code with a message in *err.
int decode_geometry(const PlanRequest& r, DecodeSchedule* s, const char** err);
// Cuts every row's attended tokens into tasks per (kv head, slice), one per CTA, longest first.
int build_decode_schedule(const PlanRequest& r, int ctas, DecodeSchedule* s, const char** err);

// CTAs per SM the decode kernels are sized for.
constexpr int kDecodeCtasPerSm = 2;

// Decode workspaces.  int: [status block (CUDA-graph mode: the task count at
// kItemCountOffset) | one merge counter per merge entry | tasks | merge entries |
// positional-encoding table]; float: [part_o (slots x kSlotHeads x D) | part_lse (slots x
// kSlotHeads)], every region 256-byte aligned.  A plan's own counts, or in CUDA-graph mode
// fixed capacities (every address a captured launch holds stays valid).
struct DecodeWsLayout {
  size_t tasks, merges, slots;
  size_t pos_floats = 0;
};
inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
inline size_t dws_counters_offset() { return 256; }
inline size_t dws_tasks_offset(const DecodeWsLayout& l) {
  return dws_counters_offset() + align256(l.merges * 4);
}
inline size_t dws_merges_offset(const DecodeWsLayout& l) {
  return dws_tasks_offset(l) + align256(l.tasks * sizeof(DecodeTask));
}
inline size_t dws_pos_offset(const DecodeWsLayout& l) {
  return dws_merges_offset(l) + align256(l.merges * sizeof(MergeEntry));
}
inline size_t dws_int_bytes(const DecodeWsLayout& l) {
  return dws_pos_offset(l) + align256(l.pos_floats * sizeof(float));
}
inline size_t dws_part_lse_offset(const DecodeWsLayout& l, int head_dim) {
  return align256(l.slots * kSlotHeads * (size_t)head_dim * sizeof(float));
}
inline size_t dws_float_bytes(const DecodeWsLayout& l, int head_dim) {
  return dws_part_lse_offset(l, head_dim) + align256(l.slots * kSlotHeads * sizeof(float)) + 256;
}
// CUDA-graph mode: a work list of at most max_items chunks per row (summed over rows) holds at
// most max_items x Hkv x slices tasks (the fixed grid), half as many merge entries, as many
// slots.
inline DecodeWsLayout decode_capacity_layout(size_t max_items, int num_kv_heads, int gslices) {
  const size_t tasks = max_items * (size_t)num_kv_heads * gslices;
  return {tasks, tasks / 2, tasks, 0};
}

// Byte offsets inside the int workspace.
constexpr size_t kStatusBytes = 256;
constexpr size_t kItemCountOffset = 64;  // int32 inside the status block (CUDA-graph mode)

// Capacities the workspaces are cut for: a plan's own counts, or in CUDA-graph mode fixed
// maxima, so that every address a captured launch holds stays valid for later plans.
struct WsLayout {
  size_t counters;  // fused-merge counters
  size_t items;
  size_t merges;
  size_t slots;     // split partials
  size_t pos_floats = 0;  // positional-encoding table (2 head_dim + num_qo_heads floats, or 0)
};
inline WsLayout layout_of(const Plan& p, int num_kv_heads) {
  return {p.merges.size() * (size_t)num_kv_heads * p.gslices, p.items.size(), p.merges.size(),
          (size_t)p.num_slots, 0};
}
// A work list of at most max_items items has at most max_items / 2 split requests (each has
// two or more chunks) and at most max_items partial slots.
inline WsLayout capacity_layout(size_t max_items, int num_kv_heads, int gslices) {
  const size_t merges = max_items / 2;
  return {merges * (size_t)num_kv_heads * gslices, max_items, merges, max_items, 0};
}
// int workspace: [status block | merge counters | work items | merge entries]; plan() writes
// everything up to the end of the merge entries in one upload (counters zeroed).
inline size_t items_offset(const WsLayout& l) {
  return kStatusBytes + (l.counters * 4 + 255) / 256 * 256;
}
inline size_t merges_offset(const WsLayout& l) { return items_offset(l) + l.items * sizeof(WorkItem); }
inline size_t pos_table_offset(const WsLayout& l) {
  return (merges_offset(l) + l.merges * sizeof(MergeEntry) + 255) / 256 * 256;
}
inline size_t int_ws_bytes_of(const WsLayout& l) {
  return pos_table_offset(l) + l.pos_floats * sizeof(float) + 256;
}
// float workspace: [part_o (slots x Hq x D) | part_lse (slots x Hq)], each 256-byte aligned
inline size_t part_lse_offset(const WsLayout& l, int num_qo_heads, int head_dim) {
  return (l.slots * num_qo_heads * head_dim * sizeof(float) + 255) / 256 * 256;
}
inline size_t float_ws_bytes_of(const WsLayout& l, int num_qo_heads, int head_dim) {
  return part_lse_offset(l, num_qo_heads, head_dim) +
         (l.slots * num_qo_heads * sizeof(float) + 255) / 256 * 256;
}
inline size_t items_offset(const Plan& p, int num_kv_heads) {
  return items_offset(layout_of(p, num_kv_heads));
}
inline size_t merges_offset(const Plan& p, int num_kv_heads) {
  return merges_offset(layout_of(p, num_kv_heads));
}
inline size_t int_ws_bytes_of(const Plan& p, int num_kv_heads) {
  return int_ws_bytes_of(layout_of(p, num_kv_heads));
}
inline size_t float_ws_bytes_of(const Plan& p, int num_qo_heads, int head_dim) {
  return float_ws_bytes_of(layout_of(p, 1), num_qo_heads, head_dim);
}

}  // namespace pkd
