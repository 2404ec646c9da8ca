// planner.cpp -- host planners: turn a CSR page table into the work a decode launch runs.
//
// FlashInfer attention API page, BatchDecodeWithPagedKVCacheWrapper:
//   - plan() builds auxiliary data structures once and every later run() reuses them
//     (across layers);
//   - indptr / indices / last_page_len describe each request's pages, with
//     kv_len = page_size * (pages - 1) + last_page_len (batch prefill example);
//   - window_left keeps the keys t >= kv_len - 1 - window_left;
//   - fixed_split_size (pages) fixes the split-KV chunk so that the merge, and thus the
//     output, does not depend on the batch; disable_split_kv keeps one chunk per request.
// With a fixed split, chunks are cut at multiples of the chunk size counted from the request's
// first token, so a request's partition depends only on its own length, its window and the
// chunk size.
//
// build_plan: the MLA work list (BatchMLAPagedAttentionWrapper; one CTA, or CTA pair, per
// item and SM, in waves).  build_decode_schedule (below): the persistent decode kernel's task
// lists.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <utility>

#include "pkd_internal.h"

namespace pkd {

namespace {

constexpr int kErrInvalid = -1;
constexpr int kErrUnsupported = -5;
constexpr int kErrWorkspace = -3;
constexpr int64_t kMinChunk = 256;   // never split below this many tokens

}  // namespace

int build_plan(const PlanRequest& r, Plan* plan, const char** err) {
  *plan = Plan();
  if (!r.mla) {
    *err = "build_plan plans MLA batches; decode batches use build_decode_schedule";
    return kErrInvalid;
  }
  if (r.batch < 0 || (r.batch > 0 && (!r.indptr || !r.kv_len))) {
    *err = "batch must be >= 0 and the page table pointers non-null";
    return kErrInvalid;
  }
  if (r.num_qo_heads <= 0 || r.num_kv_heads != 1) {
    *err = "num_heads must be positive";
    return kErrInvalid;
  }
  if (r.kv_dtype != kF16 && r.kv_dtype != kBF16) {
    *err = "the MLA caches must be F16 or BF16";
    return kErrInvalid;
  }
  if (r.page_size < 1) {
    *err = "page_size must be >= 1";
    return kErrUnsupported;
  }
  if (r.batch > 0 && r.indptr[0] < 0) {
    *err = "indptr[0] must be >= 0";
    return kErrInvalid;
  }
  const int ps = r.page_size;
  plan->kind = kTensorCore;
  plan->heads_per_cta = r.mla_heads_per_cta;
  plan->gslices = (r.num_qo_heads + plan->heads_per_cta - 1) / plan->heads_per_cta *
                  r.mla_ctas_per_head_tile;
  plan->tile_tokens = r.mla_tile_tokens;

  // per-request lengths, from kv_len_arr (pages may be more than the length needs)
  std::vector<int64_t> n_req(r.batch);
  for (int i = 0; i < r.batch; ++i) {
    const int64_t pages = (int64_t)r.indptr[i + 1] - r.indptr[i];
    if (pages < 0) {
      *err = "indptr must be non-decreasing";
      return kErrInvalid;
    }
    if (r.kv_len[i] < 0 || (int64_t)r.kv_len[i] > pages * ps) {
      *err = "kv_len must lie in [0, pages * page_size] for every request";
      return kErrInvalid;
    }
    n_req[i] = r.kv_len[i];
  }

  // Output rows: query token j of request i is row i * q_len + j, at position
  // n - q_len + j, and sees the keys up to that position -- a decode query over the
  // request's first n - q_len + j + 1 keys, read through the request's own pages.  Each row
  // is planned as a request of its own (with q_len = 1 the rows are the requests).
  const int ql = r.q_len > 0 ? r.q_len : 1;
  const int64_t rows64 = (int64_t)r.batch * ql;
  if (rows64 > (int64_t)std::numeric_limits<int32_t>::max() / 2) {
    *err = "batch * q_len_per_req is too large";
    return kErrInvalid;
  }
  const int rows = (int)rows64;
  std::vector<int64_t> n(rows), w(rows);
  std::vector<int32_t> base(rows);
  int64_t total = 0, longest = 0;
  for (int row = 0; row < rows; ++row) {
    const int i = row / ql, j = row % ql;
    n[row] = std::max<int64_t>(0, n_req[i] - (ql - 1 - j));
    base[row] = r.indptr[i];
    w[row] = (r.window_left >= 0 && n[row] - 1 - r.window_left > 0)
                 ? n[row] - 1 - r.window_left
                 : 0;
    total += n[row] - w[row];
    longest = std::max(longest, n[row] - w[row]);
  }

  // chunk size in tokens (a multiple of the page size); 0 = one chunk per request.  An MLA
  // plan may instead give every row its own chunk count in kc.
  int64_t C = 0;
  std::vector<int32_t> kc;
  const int64_t ctas_per_item = (int64_t)r.num_kv_heads * plan->gslices;
  // work items with heuristic (equal) chunks of c tokens; an empty request is one item
  auto items_with = [&](int64_t c) {
    int64_t items = 0;
    for (int i = 0; i < rows; ++i) {
      const int64_t a = n[i] - w[i];
      items += a > c ? (a + c - 1) / c : 1;
    }
    return items;
  };
  auto ctas_with = [&](int64_t c) { return items_with(c) * ctas_per_item; };
  const int64_t c_min = (kMinChunk + ps - 1) / ps * ps;
  const int64_t c_max = (longest + ps - 1) / ps * ps;
  if (r.max_items > 0 && rows > r.max_items) {
    *err = "the batch has more query rows (requests x q_len_per_req) than the work-list capacity";
    return kErrInvalid;
  }
  {
    const int sms = r.num_sms > 0 ? r.num_sms : 152;
    const int64_t slots = (int64_t)sms * (r.ctas_per_sm > 0 ? r.ctas_per_sm : 1);
    if ((int64_t)rows * ctas_per_item <= slots) {
      // The unsplit requests already fit in one wave: split only as far as the grid stays
      // one wave, i.e. the smallest page-aligned chunk whose CTAs all start at once.  A second,
      // partial wave of chunks measured slower than no split at all on GB300.
      int64_t lo = c_min, hi = std::max(c_min, c_max);
      while (lo < hi) {
        const int64_t mid = (lo / ps + (hi / ps - lo / ps) / 2) * ps;
        if (ctas_with(mid) <= slots) hi = mid; else lo = mid + ps;
      }
      C = longest > lo ? lo : 0;
    } else {
      // MLA kernels hold one CTA (pair) per SM, so the grid runs in waves of whole items, and
      // every item pays a fixed cost on top of its tokens (Q load, pipeline fill and drain,
      // epilogue: about 11 tiles of 32 tokens measured on GB300).  Candidates: for k = 1..16,
      // chunks of at most C = longest / k tokens (a row cut into ceil(a / C) equal chunks),
      // and the same with the rows of the longest chunks cut once more, as many as fill the
      // last wave.  Each is scored by a wave model -- items launch longest first, and a wave
      // costs its longest item plus the overhead -- and the cheapest kept.  Batch 114 x 999
      // tokens: 76 whole requests, then 38 requests in halves, two full waves (one chunk size
      // for all would take 1.5 waves unsplit or three waves of halves).
      constexpr int64_t kItemOverhead = 352;
      const int64_t item_slots = std::max<int64_t>(1, slots / ctas_per_item);
      // rows by chunk length, longest first, as one integer key each: length << 32 | ~row
      std::vector<uint64_t> by_len(rows);
      std::vector<int32_t> cand(rows);
      std::vector<uint32_t> att(rows);  // attended tokens per row (< 2^31)
      for (int i = 0; i < rows; ++i) att[i] = (uint32_t)(n[i] - w[i]);
      auto chunk_len = [&](int i, int32_t k) -> uint32_t {
        return att[i] > 0 ? (att[i] - 1) / (uint32_t)k + 1 : 0u;
      };
      auto row_of = [](uint64_t key) { return (int)(~(uint32_t)key); };
      auto desc = [](uint64_t x, uint64_t y) { return x > y; };
      // rekey in the previous order (chunk lengths mostly keep it), re-sort only if needed
      auto sort_rows = [&](const std::vector<int32_t>& kk) {
        for (uint64_t& key : by_len) {
          const int i = row_of(key);
          key = ((uint64_t)chunk_len(i, kk[i]) << 32) | (uint64_t)(~(uint32_t)i);
        }
        if (!std::is_sorted(by_len.begin(), by_len.end(), desc))
          std::sort(by_len.begin(), by_len.end(), desc);
      };
      for (int i = 0; i < rows; ++i) by_len[i] = (uint64_t)(~(uint32_t)i);
      // by_len sorted for kk: sum over waves of (first item's length + overhead)
      auto wave_cost = [&](const std::vector<int32_t>& kk) -> int64_t {
        int64_t cost = 0, pos = 0, next_wave = 0;
        for (const uint64_t key : by_len) {
          const int i = row_of(key);
          pos += att[i] > 0 ? kk[i] : 1;
          for (; next_wave < pos; next_wave += item_slots)
            cost += (int64_t)(key >> 32) + kItemOverhead;
        }
        return cost;
      };
      int64_t best_cost = -1;
      for (int64_t k = 1; k <= 16; ++k) {
        const int64_t c = ((longest + k - 1) / k + ps - 1) / ps * ps;
        if (k > 1 && c < c_min) break;
        int64_t items_k = 0;
        const uint32_t c32 = (uint32_t)std::min<int64_t>(c, std::numeric_limits<int32_t>::max());
        for (int i = 0; i < rows; ++i) {
          cand[i] = att[i] > c32 ? (int32_t)((att[i] - 1) / c32 + 1) : 1;
          items_k += cand[i];
        }
        if (r.max_items > 0 && items_k > r.max_items) break;
        sort_rows(cand);
        const int64_t cost0 = wave_cost(cand);
        if (best_cost < 0 || cost0 < best_cost) {
          best_cost = cost0;
          kc = cand;
        }
        // the same with the longest chunks cut once more, to fill the last wave
        int64_t fill = (item_slots - items_k % item_slots) % item_slots;
        if (fill == 0 || (r.max_items > 0 && items_k + fill > r.max_items)) continue;
        for (const uint64_t key : by_len) {
          if (fill == 0) break;
          const int i = row_of(key);
          if ((int64_t)chunk_len(i, cand[i] + 1) < c_min) continue;
          ++cand[i];
          --fill;
        }
        sort_rows(cand);
        const int64_t cost1 = wave_cost(cand);
        if (cost1 < best_cost) {
          best_cost = cost1;
          kc = cand;
        }
      }
      bool any_split = false;
      for (int i = 0; i < rows && !any_split; ++i) any_split = kc[i] > 1;
      if (!any_split) kc.clear();
      int64_t c_big = 0;
      for (int i = 0; i < (int)kc.size(); ++i)
        c_big = std::max<int64_t>(c_big, chunk_len(i, kc[i]));
      C = c_big;
    }
    if (C > 0 && kc.empty() && r.max_items > 0 && items_with(C) > r.max_items) {
      // a bounded work list (CUDA-graph mode): the smallest larger chunk that fits
      int64_t lo = C, hi = std::max(C, c_max);
      while (lo < hi) {
        const int64_t mid = (lo / ps + (hi / ps - lo / ps) / 2) * ps;
        if (items_with(mid) <= r.max_items) hi = mid; else lo = mid + ps;
      }
      C = longest > lo ? lo : 0;
    }
  }
  plan->chunk_tokens = C;

  // work items, partial slots in request order, merge entries
  std::vector<WorkItem>& items = plan->items;
  std::vector<int64_t> bounds, tile0;
  for (int i = 0; i < rows; ++i) {
    WorkItem it;
    std::memset(&it, 0, sizeof it);
    it.req = i;  // the output row
    it.page_base = base[i];
    it.merge_idx = -1;
    it.q_pos = n[i] > 0 ? (int32_t)(n[i] - 1) : 0;
    if (n[i] == 0) {
      it.chunk_tok0 = 0;
      it.tok_begin = 0;
      it.tok_end = 0;
      it.out_slot = -1;
      items.push_back(it);
      continue;
    }
    // chunk boundaries: [bounds[j], bounds[j+1]); chunk j's tiles start at tile0[j]
    bounds.clear();
    tile0.clear();
    if (C == 0 && kc.empty()) {
      bounds = {w[i], n[i]};
      tile0 = {0};
    } else {
      // heuristic: k equal page-aligned chunks, so no short remainder chunk (which would
      // launch last and do the request's merge at the very end of the grid)
      const int64_t a = n[i] - w[i];
      const int64_t k = kc.empty() ? (a + C - 1) / C : kc[i];
      bounds.push_back(w[i]);
      tile0.push_back(w[i] / ps * ps);
      for (int64_t j = 1; j < k; ++j) {
        const int64_t b = (w[i] + a * j / k) / ps * ps;
        if (b > bounds.back() && b < n[i]) {
          bounds.push_back(b);
          tile0.push_back(b);
        }
      }
      bounds.push_back(n[i]);
    }
    const int64_t nchunks = (int64_t)tile0.size();
    const int first_slot = plan->num_slots;
    it.merge_idx = nchunks > 1 ? (int32_t)plan->merges.size() : -1;
    for (int64_t k = 0; k < nchunks; ++k) {
      it.chunk_tok0 = (int32_t)tile0[k];
      it.tok_begin = (int32_t)bounds[k];
      it.tok_end = (int32_t)bounds[k + 1];
      it.out_slot = nchunks > 1 ? plan->num_slots++ : -1;
      items.push_back(it);
    }
    if (nchunks > 1) {
      MergeEntry me;
      me.req = i;
      me.first_slot = first_slot;
      me.n_chunks = (int32_t)nchunks;
      me.pad = 0;
      plan->merges.push_back(me);
    }
  }
  // longest chunks launch first (their CTAs bound the tail of the grid)
  std::stable_sort(items.begin(), items.end(), [](const WorkItem& a, const WorkItem& b) {
    return (a.tok_end - a.tok_begin) > (b.tok_end - b.tok_begin);
  });
  const int64_t ctas = (int64_t)items.size() * r.num_kv_heads * plan->gslices;
  if (ctas > (int64_t)std::numeric_limits<int32_t>::max()) {
    *err = "too many work items for one grid";
    return kErrInvalid;
  }
  *err = "";
  return 0;
}

}  // namespace pkd

// ============================================================================ decode schedule
//
// The decode kernel runs one task per CTA: a chunk of one output row's attended tokens for one
// kv head and one slice of its qo-head group.  Tasks launch longest first and the hardware
// hands each free CTA slot the next one; the kv heads (and slices) of one chunk are neighbours
// in that order, so they stream the same tokens at the same time (in the NHD layout they share
// every slot's row of memory).  Chunks:
//   - fixed_split_size: at multiples of C tokens from the row's token 0 (the result of a row
//     does not depend on the batch);
//   - disable_split_kv: whole rows;
//   - otherwise: when the unsplit rows' CTAs fit in one wave of CTA slots, the smallest
//     page-aligned chunk whose CTAs all still fit in one wave (a second, partial wave measured
//     slower); else chunks of about one CTA slot's average load; a row longer than the chunk
//     is cut into equal page-aligned parts, so no short remainder launches last.
// A unit (row, kv head, slice) cut into k > 1 chunks gets k partial slots and a merge entry; the
// CTA that finishes its last chunk merges them.  The planner writes into storage the caller
// provides and allocates nothing, so the no-allocation entry point shares it.
namespace pkd {

namespace {

constexpr int kErrInvalidD = -1;
constexpr int kErrUnsupportedD = -5;
constexpr int kErrWorkspaceD = -3;

int64_t request_len(const PlanRequest& r, int i) {
  const int64_t pages = (int64_t)r.indptr[i + 1] - r.indptr[i];
  return pages <= 0 ? 0 : (int64_t)r.page_size * (pages - 1) + r.last_page_len[i];
}

// Output row `row` (query token j of request i): its key count n, first attended token w and
// the offset of its request's page ids.
struct RowSpan {
  int64_t n, w;
  int32_t base;
};
RowSpan row_span(const PlanRequest& r, int row) {
  const int ql = r.q_len > 0 ? r.q_len : 1;
  const int i = row / ql, j = row % ql;
  RowSpan s;
  s.n = std::max<int64_t>(0, request_len(r, i) - (ql - 1 - j));
  s.w = (r.window_left >= 0 && s.n - 1 - r.window_left > 0) ? s.n - 1 - r.window_left : 0;
  s.base = r.indptr[i];
  return s;
}

int rows_of(const PlanRequest& r) { return r.batch * (r.q_len > 0 ? r.q_len : 1); }

// chunks of a row with a fixed chunk of C tokens (C = 0: one)
int64_t fixed_chunks(const RowSpan& s, int64_t C) {
  if (s.n == 0 || C == 0) return 1;
  return (s.n - 1) / C - s.w / C + 1;
}

}  // namespace

int decode_geometry(const PlanRequest& r, DecodeSchedule* s, const char** err) {
  if (r.batch < 0 || (r.batch > 0 && (!r.indptr || !r.last_page_len))) {
    *err = "batch must be >= 0 and the page table pointers non-null";
    return kErrInvalidD;
  }
  if (r.num_qo_heads <= 0 || r.num_kv_heads <= 0 || r.num_qo_heads % r.num_kv_heads != 0) {
    *err = "num_qo_heads must be a positive multiple of num_kv_heads";
    return kErrInvalidD;
  }
  if (r.kv_dtype != kF16 && r.kv_dtype != kBF16 && r.kv_dtype != kE4M3) {
    *err = "kv_dtype must be F16, BF16 or E4M3";
    return kErrInvalidD;
  }
  if (r.head_dim != 64 && r.head_dim != 128 && r.head_dim != 256) {
    *err = "head_dim must be 64, 128 or 256";
    return kErrUnsupportedD;
  }
  if (r.kv_dtype == kE4M3 && r.head_dim == 64) {
    *err = "e4m3 KV needs head_dim 128 or 256 (rows of whole 128-byte blocks)";
    return kErrUnsupportedD;
  }
  if (r.page_size < 8 || r.page_size > 256 || (r.page_size & (r.page_size - 1)) != 0) {
    *err = "page_size must be a power of two in [8, 256]";
    return kErrUnsupportedD;
  }
  if (r.q_len < 1) {
    *err = "q_len_per_req must be >= 1";
    return kErrInvalidD;
  }
  if ((int64_t)r.batch * r.q_len > (int64_t)std::numeric_limits<int32_t>::max() / 2) {
    *err = "batch * q_len_per_req is too large";
    return kErrInvalidD;
  }
  if (r.batch > 0 && r.indptr[0] < 0) {
    *err = "indptr[0] must be >= 0";
    return kErrInvalidD;
  }
  for (int i = 0; i < r.batch; ++i) {
    const int64_t pages = (int64_t)r.indptr[i + 1] - r.indptr[i];
    if (pages < 0) {
      *err = "indptr must be non-decreasing";
      return kErrInvalidD;
    }
    if (pages > 0 && (r.last_page_len[i] < 1 || r.last_page_len[i] > r.page_size)) {
      *err = "last_page_len must lie in [1, page_size] for every request with pages";
      return kErrInvalidD;
    }
    if (request_len(r, i) > (int64_t)std::numeric_limits<int32_t>::max() - 4096) {
      *err = "a request is longer than 2^31 - 4096 tokens";
      return kErrInvalidD;
    }
  }
  const int G = r.num_qo_heads / r.num_kv_heads;
  // use_tensor_cores auto takes the tensor-core kernel at every group size: measured on GB300,
  // it streams faster than the CUDA-core kernel for groups of 1, 2, 4 and 8 alike
  s->kind = r.use_tensor_cores == 0 ? kCudaCore : kTensorCore;
  if (s->kind == kTensorCore) {
    s->heads_per_cta = 8;
  } else {
    int gp = 1;
    while (gp < G && gp < 8) gp <<= 1;
    s->heads_per_cta = gp;
  }
  s->gslices = (G + s->heads_per_cta - 1) / s->heads_per_cta;
  s->tile_tokens = 16384 / (r.head_dim * (r.kv_dtype == kE4M3 ? 1 : 2));
  return 0;
}

namespace {

// The chunking of a batch.
enum ChunkMode {
  kChunkFixed,  // multiples of C counted from token 0 (fixed_split_size)
  kChunkEqual,  // rows longer than C in equal page-aligned parts
  kChunkHead,   // rows longer than C cut once, after their first C tokens (page-aligned end)
};
struct DecodeChunking {
  int64_t C;  // chunk tokens (0 = whole rows)
  int mode;
};

// End of the first chunk of a row longer than C under kChunkHead (C >= one page).
int64_t head_cut(const RowSpan& sp, int64_t C, int ps) { return (sp.w + C) / ps * ps; }

int64_t chunks_of(const RowSpan& sp, int64_t C, int mode) {
  const int64_t a = sp.n - sp.w;
  if (mode == kChunkFixed) return fixed_chunks(sp, C);
  if (sp.n == 0 || C == 0 || a <= C) return 1;
  if (mode == kChunkHead) return 2;
  return (a + C - 1) / C;
}

// chunks of every row, the rows split in more than one, and their partial slots
struct ChunkCounts {
  int64_t chunks = 0, split = 0, slots = 0;
};
ChunkCounts count_chunks(const PlanRequest& r, int64_t C, int mode) {
  ChunkCounts c;
  for (int row = 0; row < rows_of(r); ++row) {
    const int64_t k = chunks_of(row_span(r, row), C, mode);
    c.chunks += k;
    if (k > 1) {
      ++c.split;
      c.slots += k;
    }
  }
  return c;
}

// Fixed cost of a decode task in tokens: prologue, pipeline fill and drain, epilogue and merge,
// about 8 us at the ~24 ns per token of one CTA of the e4m3 head_dim-256 kernel with RoPE
// (fitted to fixed-split measurements of a 128-row batch on GB300).
constexpr int64_t kDecodeTaskOverhead = 352;
// Largest slot count and row count the list-scheduling score handles (its storage is on the
// stack); beyond them only the one-wave equal split is considered.
constexpr int kMaxScoredSlots = 1024;

// Finish-time buckets of the list-scheduling score (on the stack).
constexpr int kSpanBuckets = 1024;

// Makespan, in tokens plus kDecodeTaskOverhead per task, of a batch whose rows (attended
// lengths `len`, longest first, all at most 2C) are cut under kChunkHead at C, when the tasks
// (per_row per chunk) launch longest first and each starts on the CTA slot that frees first:
// how the hardware hands a grid's CTAs to free slots.  Finish times are counted in buckets of
// q tokens (q chosen so that 3 (C + overhead) / q fits kSpanBuckets; the slots that free first
// are the lowest non-empty bucket, which never moves down).  `pieces` holds 2 * rows entries.
int64_t head_cut_makespan(const int32_t* len, int rows, int64_t C, int per_row, int slots,
                          int32_t* pieces, uint16_t* count) {
  // chunk lengths, longest first: the cut rows' first chunks (C), then the merge of their
  // remainders and the uncut rows (both already in descending order, all at most C)
  int n_cut = 0;
  while (n_cut < rows && len[n_cut] > C) ++n_cut;
  int np = 0;
  for (int i = 0; i < n_cut; ++i) pieces[np++] = (int32_t)C;
  for (int i = 0, j = n_cut; i < n_cut || j < rows;) {
    if (j >= rows || (i < n_cut && len[i] - C >= len[j])) pieces[np++] = (int32_t)(len[i++] - C);
    else pieces[np++] = len[j++];
  }
  const int64_t ntask = (int64_t)np * per_row;
  const int m = (int)std::min<int64_t>(slots, ntask);
  if (m == 0) return 0;
  const int64_t q = (3 * (C + kDecodeTaskOverhead)) / (kSpanBuckets - 8) + 1;
  const double per_q = 1.0 / (double)q;
  auto units = [&](int32_t piece) {
    return (int)((double)(piece + kDecodeTaskOverhead) * per_q + 0.5);
  };
  // every task of the batch costs at most units(C); a slot never holds more than 2 C of work
  // past its first task (at most 2 slots' worth of tasks in all), so finish < 3 units(C)
  const int top = units((int32_t)C);
  std::memset(count, 0, sizeof(uint16_t) * (size_t)(3 * top + 2));
  int p = 0, u = 0, lo = 0;  // the next task: unit u of chunk p; lo: the lowest finish time
  for (int i = 0; i < m; ++i) {
    lo = units(pieces[p]);
    ++count[lo];
    if (++u == per_row) { u = 0; ++p; }
  }
  int span = units(pieces[0]);
  for (; p < np; ++p, u = 0) {
    const int c = units(pieces[p]);
    for (; u < per_row; ++u) {
      while (count[lo] == 0) ++lo;
      --count[lo];
      const int f = std::min(lo + c, 3 * top + 1);
      ++count[f];
      span = std::max(span, f);
    }
  }
  return (int64_t)span * q;
}

// `slots` CTA slots on the GPU; `max_slots` > 0 bounds the partial slots (per unit).
DecodeChunking choose_chunking(const PlanRequest& r, const DecodeSchedule& g, int64_t slots,
                               int64_t max_slots) {
  const int rows = rows_of(r);
  const int64_t per_row = (int64_t)r.num_kv_heads * g.gslices;
  const int ps = r.page_size;
  if (r.disable_split_kv) return {0, kChunkEqual};
  if (r.fixed_split_size > 0) return {(int64_t)r.fixed_split_size * ps, kChunkFixed};
  int64_t total = 0, longest = 0;
  for (int row = 0; row < rows; ++row) {
    const RowSpan sp = row_span(r, row);
    total += sp.n - sp.w;
    longest = std::max(longest, sp.n - sp.w);
  }
  const int64_t c_min = (kMinChunk + ps - 1) / ps * ps;
  const int64_t c_max = std::max(c_min, (longest + ps - 1) / ps * ps);
  // the smallest page-aligned chunk in [lo, c_max] for which `fits` holds (fits(c_max) does)
  auto smallest = [&](int64_t lo, auto fits) {
    int64_t hi = c_max;
    while (lo < hi) {
      const int64_t mid = (lo / ps + (hi / ps - lo / ps) / 2) * ps;
      if (fits(mid)) hi = mid; else lo = mid + ps;
    }
    return lo;
  };
  // bounded work lists (CUDA-graph capacity, partial-slot storage)
  auto fits_caps = [&](int64_t c, int mode) {
    const ChunkCounts k = count_chunks(r, c, mode);
    return (r.max_items <= 0 || k.chunks <= r.max_items) &&
           (max_slots <= 0 || k.slots * per_row <= max_slots);
  };
  int64_t C;
  if ((int64_t)rows * per_row <= slots && slots <= kMaxScoredSlots) {
    // The unsplit rows fit in one wave.  Candidates: the smallest equal split whose CTAs all
    // start at once (its time is about its longest chunk), and cutting every row longer than
    // C once, for C from half the longest row up to all of it, which lets a second, partial
    // wave of short remainders fill the slots the short rows free early.  Each is scored by
    // its list-scheduling makespan; the cheapest is kept (ties: the one-wave split).
    int32_t len[kMaxScoredSlots], pieces[2 * kMaxScoredSlots];
    uint16_t buckets[kSpanBuckets];
    for (int row = 0; row < rows; ++row) {
      const RowSpan sp = row_span(r, row);
      len[row] = (int32_t)(sp.n - sp.w);
    }
    // chunks and partial slots (per unit) of the rows under an equal or a head cut at c
    auto counts = [&](int64_t c, int mode) {
      ChunkCounts k;
      for (int row = 0; row < rows; ++row) {
        const uint32_t a = (uint32_t)len[row], c32 = (uint32_t)c;
        const int64_t n = a <= c32 ? 1 : mode == kChunkHead ? 2 : (a - 1) / c32 + 1;
        k.chunks += n;
        if (n > 1) {
          ++k.split;
          k.slots += n;
        }
      }
      return k;
    };
    auto fits = [&](int64_t c, int mode) {
      const ChunkCounts k = counts(c, mode);
      return (r.max_items <= 0 || k.chunks <= r.max_items) &&
             (max_slots <= 0 || k.slots * per_row <= max_slots);
    };
    C = smallest(c_min, [&](int64_t c) { return counts(c, kChunkEqual).chunks * per_row <= slots; });
    if (!fits(C, kChunkEqual)) C = smallest(C, [&](int64_t c) { return fits(c, kChunkEqual); });
    if (C >= longest) C = 0;
    DecodeChunking best{C, kChunkEqual};
    int64_t best_cost = (C ? C : longest) + kDecodeTaskOverhead;
    if (longest > c_min && longest < (int64_t)1 << 30) {
      std::sort(len, len + rows, [](int32_t x, int32_t y) { return x > y; });
      for (int k = 8; k < 16; ++k) {
        const int64_t c = std::max(c_min, ((longest * k + 15) / 16 + ps - 1) / ps * ps);
        if (c >= longest || c + kDecodeTaskOverhead >= best_cost) break;  // span >= c + overhead
        if (2 * c < longest || !fits(c, kChunkHead)) continue;
        const int64_t cost =
            head_cut_makespan(len, rows, c, (int)per_row, (int)slots, pieces, buckets);
        if (cost < best_cost) {
          best_cost = cost;
          best = {c, kChunkHead};
        }
      }
    }
    return best;
  } else if ((int64_t)rows * per_row <= slots) {
    // one wave without the scored candidates (more slots than the score's storage holds)
    C = smallest(c_min, [&](int64_t c) {
      return count_chunks(r, c, kChunkEqual).chunks * per_row <= slots;
    });
  } else {
    // chunks of about the average load of a CTA slot
    C = std::max<int64_t>(c_min, (total * per_row + slots - 1) / slots);
    C = (C + ps - 1) / ps * ps;
  }
  if (C >= longest) return {0, kChunkEqual};
  if (!fits_caps(C, kChunkEqual))
    C = smallest(C, [&](int64_t c) { return fits_caps(c, kChunkEqual); });
  return {C >= longest ? 0 : C, kChunkEqual};
}

}  // namespace

int build_decode_schedule(const PlanRequest& r, int ctas, DecodeSchedule* s, const char** err) {
  int rc = decode_geometry(r, s, err);
  if (rc) return rc;
  s->n_tasks = s->n_merges = s->n_slots = s->n_chunks = 0;
  s->storage_short = false;
  const int rows = rows_of(r);
  const int ps = r.page_size;
  const int gsl = s->gslices;
  const int per_row = r.num_kv_heads * gsl;  // units of a row: one per (kv head, slice)
  auto too_small = [&](const char* what) {
    *err = what;
    return kErrWorkspaceD;
  };
  if (r.max_items > 0 && rows > r.max_items)
    return too_small("the batch has more query rows (requests x q_len_per_req) than the "
                     "work-list capacity");
  const DecodeChunking ch = choose_chunking(r, *s, std::max(1, ctas), s->max_slots);
  const int64_t C = ch.C;

  // 1. every row's chunks, its slots and merge entries (row order)
  int64_t n_chunks = 0, n_slots = 0, n_merges = 0;
  auto add_chunk = [&](int row, int64_t b, int64_t e, int64_t tile0, int64_t q, int64_t k,
                       int64_t slot_base, int64_t merge_base) {
    if (n_chunks < s->chunks_cap)
      s->chunks[n_chunks] = {row, (int32_t)b, (int32_t)e, (int32_t)tile0, (int32_t)q,
                             (int32_t)k, (int32_t)slot_base, (int32_t)merge_base};
    ++n_chunks;
  };
  for (int row = 0; row < rows; ++row) {
    const RowSpan sp = row_span(r, row);
    const int64_t k = chunks_of(sp, C, ch.mode);
    const int64_t slot_base = n_slots, merge_base = n_merges;
    if (k > 1) {
      for (int u = 0; u < per_row; ++u) {
        if (n_merges < s->merges_cap)
          s->merges[n_merges] = {row, (int32_t)(slot_base + u * k), (int32_t)k, u};
        ++n_merges;
      }
      n_slots += per_row * k;
    }
    if (sp.n == 0 || C == 0 || (k == 1 && ch.mode != kChunkFixed)) {
      add_chunk(row, sp.n == 0 ? 0 : sp.w, sp.n, sp.n == 0 ? 0 : sp.w / ps * ps, 0, 1, slot_base,
                merge_base);
    } else if (ch.mode == kChunkHead) {
      // the first C tokens (to a page boundary), then the rest
      const int64_t x = head_cut(sp, C, ps);
      add_chunk(row, sp.w, x, sp.w / ps * ps, 0, 2, slot_base, merge_base);
      add_chunk(row, x, sp.n, x, 1, 2, slot_base, merge_base);
    } else if (ch.mode == kChunkFixed) {
      // multiples of C counted from token 0
      int64_t q = 0;
      for (int64_t m = sp.w / C; m <= (sp.n - 1) / C; ++m, ++q)
        add_chunk(row, std::max(m * C, sp.w), std::min((m + 1) * C, sp.n), m * C, q, k,
                  slot_base, merge_base);
    } else {
      // k equal page-aligned parts, so no short remainder chunk launches last
      const int64_t a = sp.n - sp.w;
      int64_t b = sp.w, tile0 = sp.w / ps * ps, q = 0;
      for (int64_t m = 1; m <= k; ++m) {
        const int64_t e = m == k ? sp.n : (sp.w + a * m / k) / ps * ps;
        if (e <= b) continue;
        add_chunk(row, b, e, tile0, q++, k, slot_base, merge_base);
        b = e;
        tile0 = e;
      }
    }
  }
  const int64_t n_tasks = n_chunks * per_row;
  if (r.max_items > 0 && n_chunks > r.max_items)
    return too_small("fixed_split_size cuts this batch into more work items than the "
                     "work-list capacity");
  if (s->max_slots > 0 && n_slots > s->max_slots)
    return too_small("split partials exceed the workspace");
  if (n_chunks > s->chunks_cap || n_tasks > s->tasks_cap || n_merges > s->merges_cap) {
    s->storage_short = true;
    s->n_chunks = n_chunks;
    s->n_tasks = n_tasks;
    s->n_merges = n_merges;
    s->n_slots = n_slots;
    return too_small(n_merges > s->merges_cap ? "merge list full" : "work list full");
  }
  // 2. chunks longest first, ties in row and chunk order (a total order, so an in-place sort)
  std::sort(s->chunks, s->chunks + n_chunks, [](const DecodeChunk& x, const DecodeChunk& y) {
    const int32_t lx = x.e - x.b, ly = y.e - y.b;
    if (lx != ly) return lx > ly;
    return x.row != y.row ? x.row < y.row : x.q < y.q;
  });
  // 3. one task per unit of each chunk, the units of a chunk neighbours; task q runs on CTA q
  for (int64_t c = 0; c < n_chunks; ++c) {
    const DecodeChunk& ck = s->chunks[c];
    const RowSpan sp = row_span(r, ck.row);
    for (int u = 0; u < per_row; ++u) {
      DecodeTask& t = s->tasks[c * per_row + u];
      t.req = ck.row;
      t.page_base = sp.base;
      t.chunk_tok0 = ck.tile0;
      t.tok_begin = ck.b;
      t.tok_end = ck.e;
      t.out_slot = ck.k > 1 ? ck.slot_base + u * ck.k + ck.q : -1;
      t.merge_idx = ck.k > 1 ? ck.merge_base + u : -1;
      t.q_pos = sp.n > 0 ? (int32_t)(sp.n - 1) : 0;
      t.kvh = u / gsl;
      t.gs = u % gsl;
      t.cta = (int32_t)(c * per_row + u);
      t.pad = 0;
    }
  }
  s->n_chunks = n_chunks;
  s->n_tasks = n_tasks;
  s->n_merges = n_merges;
  s->n_slots = n_slots;
  *err = "";
  return 0;
}

}  // namespace pkd
