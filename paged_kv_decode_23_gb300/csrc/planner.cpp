// planner.cpp -- host planner: turns a CSR page table into the split-KV work list.
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
// chunk size.  The heuristic split cuts a long request into equal page-aligned chunks.
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
constexpr int kCtasPerSm = 2;        // every decode kernel is sized for two resident CTAs
constexpr int kWavesTarget = 1;      // heuristic: about one wave of CTAs (measured best on GB300)
constexpr int64_t kMinChunk = 256;   // never split below this many tokens

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int tile_tokens_for(int head_dim, int kv_dtype) {
  const int row_bytes = head_dim * (kv_dtype == kE4M3 ? 1 : 2);
  return 16384 / row_bytes;  // a K tile is 16 KiB; K + V make a 32 KiB stage
}

}  // namespace

int build_plan(const PlanRequest& r, Plan* plan, const char** err) {
  *plan = Plan();
  if (r.batch < 0 || (r.batch > 0 && (!r.indptr || (!r.last_page_len && !r.kv_len)))) {
    *err = "batch must be >= 0 and the page table pointers non-null";
    return kErrInvalid;
  }
  if (r.num_qo_heads <= 0 || r.num_kv_heads <= 0 || r.num_qo_heads % r.num_kv_heads != 0) {
    *err = "num_qo_heads must be a positive multiple of num_kv_heads";
    return kErrInvalid;
  }
  if (r.kv_dtype != kF16 && r.kv_dtype != kBF16 && r.kv_dtype != kE4M3) {
    *err = "kv_dtype must be F16, BF16 or E4M3";
    return kErrInvalid;
  }
  if (!r.mla && r.head_dim != 64 && r.head_dim != 128 && r.head_dim != 256) {
    *err = "head_dim must be 64, 128 or 256";
    return kErrUnsupported;
  }
  if (r.kv_dtype == kE4M3 && r.head_dim == 64) {
    *err = "e4m3 KV needs head_dim 128 or 256 (rows of whole 128-byte blocks)";
    return kErrUnsupported;
  }
  if (r.mla ? r.page_size < 1 : (!is_pow2(r.page_size) || r.page_size < 8 || r.page_size > 256)) {
    *err = r.mla ? "page_size must be >= 1" : "page_size must be a power of two in [8, 256]";
    return kErrUnsupported;
  }
  if (r.batch > 0 && r.indptr[0] < 0) {
    *err = "indptr[0] must be >= 0";
    return kErrInvalid;
  }
  const int ps = r.page_size;
  const int group = r.num_qo_heads / r.num_kv_heads;
  const int G = group;

  // kernel choice (use_tensor_cores): auto takes the tensor-core kernel
  plan->kind = r.use_tensor_cores == 0 ? kCudaCore : kTensorCore;
  if (plan->kind == kTensorCore) {
    plan->heads_per_cta = 8;
  } else {
    int gp = 2;
    while (gp < G && gp < 8) gp <<= 1;
    plan->heads_per_cta = gp;
  }
  if (r.mla) {
    plan->kind = kTensorCore;
    plan->heads_per_cta = r.mla_heads_per_cta;
  }
  plan->gslices = (G + plan->heads_per_cta - 1) / plan->heads_per_cta;
  if (r.mla) plan->gslices *= r.mla_ctas_per_head_tile;
  if (r.rope && plan->kind == kCudaCore) {
    *err = "pos_encoding_mode ROPE_LLAMA is built for the tensor-core kernel only";
    return kErrUnsupported;
  }
  plan->tile_tokens = r.mla ? r.mla_tile_tokens : tile_tokens_for(r.head_dim, r.kv_dtype);

  // per-request lengths
  std::vector<int64_t> n_req(r.batch);
  for (int i = 0; i < r.batch; ++i) {
    const int64_t pages = (int64_t)r.indptr[i + 1] - r.indptr[i];
    if (pages < 0) {
      *err = "indptr must be non-decreasing";
      return kErrInvalid;
    }
    if (r.kv_len) {  // lengths given directly (MLA's kv_len_arr); extra pages are ignored
      if (r.kv_len[i] < 0 || (int64_t)r.kv_len[i] > pages * ps) {
        *err = "kv_len must lie in [0, pages * page_size] for every request";
        return kErrInvalid;
      }
      n_req[i] = r.kv_len[i];
      continue;
    }
    if (pages == 0) {
      n_req[i] = 0;
      continue;
    }
    const int lpl = r.last_page_len[i];
    if (lpl < 1 || lpl > ps) {
      *err = "last_page_len must lie in [1, page_size] for every request with pages";
      return kErrInvalid;
    }
    n_req[i] = (int64_t)ps * (pages - 1) + lpl;
    if (n_req[i] > (int64_t)std::numeric_limits<int32_t>::max() - 4096) {
      *err = "a request is longer than 2^31 - 4096 tokens";
      return kErrInvalid;
    }
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
  if (r.disable_split_kv) {
    C = 0;
  } else if (r.fixed_split_size > 0) {
    C = (int64_t)r.fixed_split_size * ps;
  } else {
    const int sms = r.num_sms > 0 ? r.num_sms : 152;
    const int64_t slots = (int64_t)sms * (r.ctas_per_sm > 0 ? r.ctas_per_sm : kCtasPerSm);
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
    } else if (r.mla) {
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
    } else {
      // More requests than one wave: chunks of about the average load of a CTA slot over
      // kWavesTarget waves, so the longest requests stop bounding the tail.
      const int64_t per_cta = (total * ctas_per_item + slots * kWavesTarget - 1) /
                              (slots * kWavesTarget);
      int64_t c = std::max<int64_t>(c_min, per_cta);
      c = (c + ps - 1) / ps * ps;
      C = longest > c ? c : 0;
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
  const bool fixed = !r.disable_split_kv && r.fixed_split_size > 0;
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
    } else if (fixed) {
      // multiples of C counted from token 0: independent of the rest of the batch
      for (int64_t k = w[i] / C; k <= (n[i] - 1) / C; ++k) {
        bounds.push_back(std::max(k * C, w[i]));
        tile0.push_back(k * C);
      }
      bounds.push_back(n[i]);
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
  if (r.max_items > 0 && (int64_t)items.size() > r.max_items) {
    // only a fixed split can get here: the heuristic already fits the capacity
    *err = "fixed_split_size cuts this batch into more work items than the work-list capacity";
    return kErrWorkspace;
  }
  *err = "";
  return 0;
}

}  // namespace pkd
