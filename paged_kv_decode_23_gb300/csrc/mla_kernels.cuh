// mla_kernels.cuh -- MLA paged decode (FlashInfer attention API page, flashinfer.mla /
// BatchMLAPagedAttentionWrapper plan()/run()), sm_103a.
//
// With matrix absorption, every query head attends over one shared latent cache: the key of
// token t is [ckv_t (512), kpe_t (64)] and its value is ckv_t; logit = sm_scale * (<q_nope,
// ckv_t> + <q_pe, kpe_t>).  One CTA computes one work item (a chunk of one request's tokens)
// for a tile of 32 query heads.
//
// Structure (one CTA = 8 consumer warps + 4 producer warps):
//   producer  copies each 32-token tile's rows with 16-byte cp.async gathers (per token 1024
//             bytes of ckv and 128 bytes of kpe, so any page size works, 1 included; the warp
//             copies a row's ckv as two 512-byte halves, then its kpe on 8 lanes) into a
//             shared-memory stage of token rows 1168 bytes apart (1152 + 16: eight consecutive
//             rows fall in eight different 16-byte bank groups, so ldmatrix reads are
//             conflict-free without a swizzle).  A copy-only probe on GB300 gathered these rows
//             at 26.6 GB/s per SM with cp.async against 14.0 GB/s with two 1-D bulk copies per
//             row (the TMA unit's requests per second bound the latter).  Completion: each
//             lane's cp.async arrival, and lane 0's release arrival after it publishes the
//             stage's row mask.
//   consumers warp w owns latent dims [64w, 64w + 64): it forms the partial logits S_w^T
//             (32 tokens x 32 heads) over those dims with mma.m16n8k16 (warps 0-3 also add
//             one 16-dim k step of the kpe part each), the partials meet in shared memory,
//             all 256 consumer threads finish the logits and the online softmax (thread =
//             head x 4 tokens), write P and the per-head rescale factor, and warp w then adds
//             V^T P^T for its 64 dims (O^T accumulators: 64 dims x 32 heads per warp).
//   epilogue  O^T / l is staged through the (then idle) pipeline buffers and written with
//             16-byte stores, as the final o / lse or as an fp32 partial; the last CTA of a
//             split request merges the partials in chunk order (no CTA waits for another).
#pragma once

#include <type_traits>

#include "pkd_device.cuh"
#include "pkd_internal.h"

namespace pkd {

namespace mla {

constexpr int DC = 512;           // latent (ckv) dims
constexpr int DP = 64;            // rope (kpe) dims
constexpr int HT = 32;            // query heads per CTA
constexpr int TS = 32;            // tokens per stage
constexpr int NW = 8;             // consumer warps
constexpr int NCONS = NW * 32;
constexpr int NPW = 4;            // producer warps (rows 8 pw .. 8 pw + 7 of each tile)
constexpr int THREADS = NCONS + NPW * 32;
constexpr int NSTAGES = 3;
constexpr int ROW_BYTES = (DC + DP) * 2;        // 1152: ckv (1024) then kpe (128)
constexpr int ROW_STRIDE = ROW_BYTES + 16;       // 1168 bytes between token rows
constexpr int STAGE_BYTES = TS * ROW_STRIDE;     // 37376
constexpr int PIPE_BYTES = NSTAGES * STAGE_BYTES;
constexpr int SPART_STRIDE = 36;                // floats per head row of a partial-logit tile
constexpr int SPART_BYTES = NW * HT * SPART_STRIDE * 4;
constexpr int P_STRIDE = 80;                    // bytes per head row of P (32 tokens + pad)
constexpr int P_BYTES = HT * P_STRIDE;
constexpr int EPI_BYTES = HT * DC * 4;          // fp32 O staging in the epilogue
constexpr int SMEM_BYTES = PIPE_BYTES + SPART_BYTES + 2 * P_BYTES + 3 * HT * 4 + 1024;
static_assert(EPI_BYTES <= PIPE_BYTES, "the epilogue reuses the pipeline buffers");

}  // namespace mla

namespace mla_detail {

using namespace dev;

// 16-byte global -> shared copy through the load path (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "l"(policy)
               : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Byte offset of 16-byte chunk c (0..63 ckv, 64..71 kpe) of tile row r inside a stage.
__device__ __forceinline__ uint32_t row_chunk(int r, int c) {
  return (uint32_t)(r * mla::ROW_STRIDE + c * 16);
}

template <typename T>
__device__ __forceinline__ void produce(const MlaParams& p, const WorkItem& it, int j0, int ntiles,
                                        uint32_t smem, uint32_t full0, uint32_t empty0,
                                        volatile int* abort_flag, int lane, int pw,
                                        volatile uint32_t* bad_rows) {
  const int ps = p.page_size;
  const char* ckv = static_cast<const char*>(p.ckv);
  const char* kpe = static_cast<const char*>(p.kpe);
  const uint64_t pol = policy_evict_first();
  bool ok = true;
  // lane r: page id of tile row r of tile i (loaded one tile ahead, so its latency overlaps
  // the wait for a free stage); rows outside [tok_begin, tok_end) are not copied
  auto page_of = [&](int i) -> int64_t {
    const int t = it.chunk_tok0 + (j0 + i) * mla::TS + lane;
    return (i < ntiles && t >= it.tok_begin && t < it.tok_end)
               ? (int64_t)__ldg(p.indices + it.page_base + t / ps)
               : -1;
  };
  int64_t pid_next = page_of(0);
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % mla::NSTAGES;
    const int64_t pid = pid_next;
    pid_next = page_of(i + 1);
    if (i >= mla::NSTAGES) {  // lane 0 waits, so the whole warp takes one decision
      int freed = 1;
      if (lane == 0) freed = mbar_wait(empty0 + 8 * s, ((i / mla::NSTAGES) - 1) & 1, abort_flag);
      if (!__shfl_sync(~0u, freed, 0)) {
        ok = false;
        break;
      }
    }
    const int t = it.chunk_tok0 + (j0 + i) * mla::TS + lane;
    const bool ok_row = pid >= 0 && pid < p.num_pages;  // ids outside the caches: not copied
    const int64_t prow = ok_row ? pid * ps + t % ps : 0;
    const uint32_t stage = smem + s * mla::STAGE_BYTES;
    const unsigned m = __ballot_sync(~0u, ok_row);
    // tokens of the item whose page id lies outside the caches: zero rows (the consumers zero
    // them before use)
    const unsigned bad = __ballot_sync(~0u, !ok_row && t >= it.tok_begin && t < it.tok_end);
    // row by row, the whole warp: rows not copied keep stale data (their logits are masked,
    // their V zeroed)
    for (int r = 8 * pw; r < 8 * pw + 8; ++r) {
      if (!((m >> r) & 1u)) continue;  // the same for every lane
      const int64_t pr = __shfl_sync(~0u, prow, r);
      const char* src = ckv + pr * (mla::DC * 2) + lane * 16;
      const uint32_t dst = stage + r * mla::ROW_STRIDE + lane * 16;
      cp_async16(dst, src, pol);
      cp_async16(dst + 512, src + 512, pol);
      if (lane < 8) cp_async16(stage + r * mla::ROW_STRIDE + mla::DC * 2 + lane * 16,
                               kpe + pr * (mla::DP * 2) + lane * 16, pol);
    }
    if (pw == 0 && lane == 0) {
      bad_rows[s] = bad;
      mbar_arrive(full0 + 8 * s);  // release: the row mask before the consumers' acquire
    }
    cp_async_arrive(full0 + 8 * s);
  }
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(p.status, kStatusTimeout);
  }
  // every copy this lane issued lands before the CTA may exit
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// B fragments of Q^T for this warp: q_nope dims [64w, 64w + 64) (4 k steps) and, for warps
// 0-3, q_pe dims [16w, 16w + 16) (one k step), for heads g0 .. g0 + 31 (4 n tiles of 8).
template <typename T>
__device__ __forceinline__ void load_q(const MlaParams& p, int row, int g0, int gcnt, int warp,
                                       int lane, uint32_t (&qn)[4][4][2], uint32_t (&qp)[4][2]) {
  const int g = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int h = nt * 8 + g;
    const bool hl = h < gcnt;
    const T* qrow = static_cast<const T*>(p.q_nope) +
                    ((size_t)row * p.num_heads + g0 + (hl ? h : 0)) * mla::DC + warp * 64;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      qn[kk][nt][0] = hl ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + tig * 2) : 0u;
      qn[kk][nt][1] = hl ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + tig * 2 + 8) : 0u;
    }
    const T* prow = static_cast<const T*>(p.q_pe) +
                    ((size_t)row * p.num_heads + g0 + (hl ? h : 0)) * mla::DP + warp * 16;
    const bool pl = hl && warp < 4;
    qp[nt][0] = pl ? *reinterpret_cast<const uint32_t*>(prow + tig * 2) : 0u;
    qp[nt][1] = pl ? *reinterpret_cast<const uint32_t*>(prow + tig * 2 + 8) : 0u;
  }
}

}  // namespace mla_detail

// The consumer warps' part of mla_decode_kernel: attention over the item's tiles, the
// epilogue and the fused merge.
template <typename T>
__device__ __forceinline__ void consume(const MlaParams& p, const WorkItem& it, int j0, int ntiles,
                                        int gs, int g0, int gcnt, uint8_t* base, uint32_t smem,
                                        uint32_t full0, uint32_t empty0, volatile int* abort_flag,
                                        int* merge_last_s,
                                        const volatile uint32_t* bad_rows) {
  using namespace dev;
  using namespace mla_detail;
  constexpr float kNegInfF = -__builtin_huge_valf();
  float* spart = reinterpret_cast<float*>(base + mla::PIPE_BYTES);
  uint8_t* pbuf = base + mla::PIPE_BYTES + mla::SPART_BYTES;
  float* alpha_s = reinterpret_cast<float*>(pbuf + 2 * mla::P_BYTES);  // after P hi and P lo
  float* m_s = alpha_s + mla::HT;
  float* l_s = m_s + mla::HT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int g = lane >> 2, tig = lane & 3;
  uint32_t qn[4][4][2], qp[4][2];
  load_q<T>(p, it.req, g0, gcnt, warp, lane, qn, qp);
  float acc[4][4][4];  // O^T: [dims m tile][heads n tile][fragment]
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b][0] = acc[a][b][1] = acc[a][b][2] = acc[a][b][3] = 0.f;
  // softmax role: head sh = tid / 8, tokens 4 * (tid % 8) .. + 3 of each tile
  const int sh = tid >> 3, stg = tid & 7;
  float m2 = kNegInfF, lsum = 0.f;

  const int row_a = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix (A, K-major) row
  const int csel_a = lane >> 4;
  const int row_v = (lane & 7) + (lane >> 4) * 8;        // ldmatrix.trans (V^T) row
  const int csel_v = (lane >> 3) & 1;
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % mla::NSTAGES;
    if (!mbar_wait(full0 + 8 * s, (i / mla::NSTAGES) & 1, abort_flag)) {
      *abort_flag = 1;
      atomicOr(p.status, kStatusTimeout);
    }
    // after a timeout the loop runs on without waiting (every wait sees the abort flag), so
    // all consumer warps meet the same named barriers; the output is not written
    __syncwarp();
    uint32_t stage = stage_after_wait(smem + s * mla::STAGE_BYTES);
    const int tt0 = it.chunk_tok0 + (j0 + i) * mla::TS;  // first token of the tile
    bool wrote = false;
    const uint32_t bad = bad_rows[s];
    if (bad) {
      // rows with a page id outside the caches were not copied: zero the dims this warp reads
      // (ckv chunks 8w .. 8w + 7, kpe chunks 64 + 2w, 65 + 2w for w < 4)
      for (int u = lane; u < mla::TS * 10; u += 32) {
        const int r = u / 10, c = u - r * 10;
        const int chunk = c < 8 ? warp * 8 + c : (warp < 4 ? 64 + warp * 2 + (c - 8) : -1);
        if (((bad >> r) & 1u) && chunk >= 0)
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(stage + row_chunk(r, chunk)),
                       "r"(0)
                       : "memory");
      }
      wrote = true;
      __syncwarp();
      stage = stage_after_wait(stage);  // the MMA operand reads come after the zeroing
    }
    // ---- partial S^T over my dims: 2 token m tiles x 4 head n tiles
    float sa[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sa[mt][nt][0] = sa[mt][nt][1] = sa[mt][nt][2] = sa[mt][nt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4];
        ldsm_x4(stage + row_chunk(mt * 16 + row_a, warp * 8 + kk * 2 + csel_a), a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_16816<T>(sa[mt][nt], a, qn[kk][nt][0], qn[kk][nt][1]);
      }
      if (warp < 4) {
        uint32_t a[4];
        ldsm_x4(stage + row_chunk(mt * 16 + row_a, 64 + warp * 2 + csel_a), a);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_16816<T>(sa[mt][nt], a, qp[nt][0], qp[nt][1]);
      }
    }
    // C fragment (token row, head col) -> spart[warp][head][token]
    float* sp = spart + warp * mla::HT * mla::SPART_STRIDE;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int tk = mt * 16 + g, hd = nt * 8 + tig * 2;
        sp[hd * mla::SPART_STRIDE + tk] = sa[mt][nt][0];
        sp[(hd + 1) * mla::SPART_STRIDE + tk] = sa[mt][nt][1];
        sp[hd * mla::SPART_STRIDE + tk + 8] = sa[mt][nt][2];
        sp[(hd + 1) * mla::SPART_STRIDE + tk + 8] = sa[mt][nt][3];
      }
    named_bar_sync(1, mla::NCONS);
    // ---- logits, online softmax, P (thread: head sh, tokens 4 stg .. 4 stg + 3)
    {
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < mla::NW; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(
            spart + (w * mla::HT + sh) * mla::SPART_STRIDE + stg * 4);
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      const int t0 = tt0 + stg * 4;
      float sc[4] = {sum.x, sum.y, sum.z, sum.w};
      float mx = kNegInfF;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = t0 + e;
        sc[e] = (t >= it.tok_begin && t < it.tok_end) ? sc[e] * p.scale_log2 : kNegInfF;
        mx = fmaxf(mx, sc[e]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 4));
      const float mnew = fmaxf(m2, mx);
      const float ref = mnew == kNegInfF ? 0.f : mnew;
      const float alpha = fast_exp2(m2 - ref);
      float ps = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sc[e] = fast_exp2(sc[e] - ref);
        ps += sc[e];
      }
      ps += __shfl_xor_sync(~0u, ps, 1);
      ps += __shfl_xor_sync(~0u, ps, 2);
      ps += __shfl_xor_sync(~0u, ps, 4);
      lsum = lsum * alpha + ps;
      m2 = mnew;
      // P rounded to 16 bits, and the rounding remainder (P V = P_hi V + P_lo V to ~2^-17)
      uint2 pk, pl;
      pk.x = pack2<T>(sc[0], sc[1]);
      pk.y = pack2<T>(sc[2], sc[3]);
      const float2 r0 = unpack2<T>(pk.x), r1 = unpack2<T>(pk.y);
      pl.x = pack2<T>(sc[0] - r0.x, sc[1] - r0.y);
      pl.y = pack2<T>(sc[2] - r1.x, sc[3] - r1.y);
      *reinterpret_cast<uint2*>(pbuf + sh * mla::P_STRIDE + stg * 8) = pk;
      *reinterpret_cast<uint2*>(pbuf + mla::P_BYTES + sh * mla::P_STRIDE + stg * 8) = pl;
      if (stg == 0) alpha_s[sh] = alpha;
    }
    named_bar_sync(1, mla::NCONS);
    // ---- O^T += V^T P^T for my 64 dims (rescale by alpha of each head column first)
    uint32_t vst = stage;
    if (tt0 < it.tok_begin || tt0 + mla::TS > it.tok_end) {
      // rows outside [tok_begin, tok_end) were not copied: zero my 64 dims of them, so that
      // 0 * stale data cannot reach O (their logits are already -inf)
      for (int u = lane; u < mla::TS * 8; u += 32) {
        const int r = u >> 3, t = tt0 + r;
        if (t < it.tok_begin || t >= it.tok_end)
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                           stage + row_chunk(r, warp * 8 + (u & 7))),
                       "r"(0)
                       : "memory");
      }
      wrote = true;
      __syncwarp();
      vst = stage_after_wait(vst);  // V reads come after the zeroing stores
    }
    {
      float al[4][2];
      bool moved = false;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        al[nt][0] = alpha_s[nt * 8 + tig * 2];
        al[nt][1] = alpha_s[nt * 8 + tig * 2 + 1];
        moved |= al[nt][0] != 1.f || al[nt][1] != 1.f;
      }
      if (__any_sync(~0u, moved)) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            acc[mt][nt][0] *= al[nt][0];
            acc[mt][nt][1] *= al[nt][1];
            acc[mt][nt][2] *= al[nt][0];
            acc[mt][nt][3] *= al[nt][1];
          }
      }
      const uint32_t pb = smem_u32(pbuf);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        // P^T B fragments (hi and lo) for n tiles (2q, 2q+1): matrices (nt, tokens 0-7 /
        // 8-15 of the step)
        uint32_t bf[2][4][2];
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int mtx = lane >> 3;
            const int hd = (q2 * 2 + (mtx >> 1)) * 8 + (lane & 7);
            const uint32_t addr = pb + part * mla::P_BYTES + hd * mla::P_STRIDE +
                                  (ks * 16 + (mtx & 1) * 8) * 2;
            uint32_t r[4];
            ldsm_x4(addr, r);
            bf[part][q2 * 2][0] = r[0];
            bf[part][q2 * 2][1] = r[1];
            bf[part][q2 * 2 + 1][0] = r[2];
            bf[part][q2 * 2 + 1][1] = r[3];
          }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(vst + row_chunk(ks * 16 + row_v, warp * 8 + mt * 2 + csel_v), a);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
              mma_16816<T>(acc[mt][nt], a, bf[part][nt][0], bf[part][nt][1]);
        }
      }
    }
    if (wrote) fence_proxy_async_smem();  // the zeroing stores before the next TMA copies
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  if (stg == 0) {
    m_s[sh] = m2;
    l_s[sh] = lsum;
  }
  named_bar_sync(1, mla::NCONS);  // every consumer is done with the stages; m / l published
  const bool aborted = *abort_flag != 0;

  // ---- stage O^T / l as fp32 [head][dim] in the pipeline buffers
  float* ostage = reinterpret_cast<float*>(base);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int hd = nt * 8 + tig * 2;
    const float l0 = l_s[hd], l1 = l_s[hd + 1];
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int d = warp * 64 + mt * 16 + g;
      ostage[hd * mla::DC + d] = acc[mt][nt][0] * i0;
      ostage[(hd + 1) * mla::DC + d] = acc[mt][nt][1] * i1;
      ostage[hd * mla::DC + d + 8] = acc[mt][nt][2] * i0;
      ostage[(hd + 1) * mla::DC + d + 8] = acc[mt][nt][3] * i1;
    }
  }
  named_bar_sync(1, mla::NCONS);
  if (!aborted) {
    constexpr float kLn2f = 0.6931471805599453f;
    if (it.out_slot < 0) {
      for (int u = tid; u < gcnt * (mla::DC / 8); u += mla::NCONS) {
        const int hd = u / (mla::DC / 8), d0 = (u - hd * (mla::DC / 8)) * 8;
        const float4 x = *reinterpret_cast<const float4*>(ostage + hd * mla::DC + d0);
        const float4 y = *reinterpret_cast<const float4*>(ostage + hd * mla::DC + d0 + 4);
        uint4 v;
        v.x = pack2<T>(x.x, x.y);
        v.y = pack2<T>(x.z, x.w);
        v.z = pack2<T>(y.x, y.y);
        v.w = pack2<T>(y.z, y.w);
        *reinterpret_cast<uint4*>(static_cast<T*>(p.o) +
                                  ((size_t)it.req * p.num_heads + g0 + hd) * mla::DC + d0) = v;
      }
      if (tid < gcnt && p.lse) {
        const float l = l_s[tid];
        const float lse2 = l > 0.f ? m_s[tid] + log2f(l) : kNegInfF;
        p.lse[(size_t)it.req * p.num_heads + g0 + tid] = p.lse_base_e ? lse2 * kLn2f : lse2;
      }
    } else {
      for (int u = tid; u < gcnt * (mla::DC / 4); u += mla::NCONS) {
        const int hd = u / (mla::DC / 4), d0 = (u - hd * (mla::DC / 4)) * 4;
        *reinterpret_cast<float4*>(p.part_o + ((size_t)it.out_slot * p.num_heads + g0 + hd) *
                                                  mla::DC + d0) =
            *reinterpret_cast<const float4*>(ostage + hd * mla::DC + d0);
      }
      if (tid < gcnt) {
        const float l = l_s[tid];
        p.part_lse[(size_t)it.out_slot * p.num_heads + g0 + tid] =
            l > 0.f ? m_s[tid] + log2f(l) : kNegInfF;
      }
    }
  }

  // ---- fused merge: the CTA finishing a split request's last chunk (for its head slice)
  if (it.out_slot < 0) return;
  __threadfence();
  named_bar_sync(1, mla::NCONS);
  if (tid == 0) {
    int last = 0;
    if (!aborted) {
      uint32_t* ctr = p.counters + (size_t)it.merge_idx * p.gslices + gs;
      const uint32_t prev = atomicAdd(ctr, 1u);
      last = (prev + 1u == (uint32_t)p.merges[it.merge_idx].n_chunks) ? 1 : 0;
      if (last) *ctr = 0u;
    }
    *merge_last_s = last;
  }
  named_bar_sync(1, mla::NCONS);
  if (!*merge_last_s) return;
  __threadfence();
  const MergeEntry me = p.merges[it.merge_idx];
  constexpr float kLn2f = 0.6931471805599453f;
  for (int u = tid; u < gcnt * (mla::DC / 8); u += mla::NCONS) {
    const int hd = u / (mla::DC / 8), d0 = (u - hd * (mla::DC / 8)) * 8;
    const int h = g0 + hd;
    float M = kNegInfF;
    for (int c = 0; c < me.n_chunks; ++c)
      M = fmaxf(M, __ldcg(p.part_lse + (size_t)(me.first_slot + c) * p.num_heads + h));
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float W = 0.f;
    if (M != kNegInfF) {
      for (int c = 0; c < me.n_chunks; ++c) {
        const size_t slot = (size_t)(me.first_slot + c);
        const float w = fast_exp2(__ldcg(p.part_lse + slot * p.num_heads + h) - M);
        const float4* src =
            reinterpret_cast<const float4*>(p.part_o + (slot * p.num_heads + h) * mla::DC + d0);
        const float4 a = __ldcg(src), b = __ldcg(src + 1);
        W += w;
        o[0] += w * a.x; o[1] += w * a.y; o[2] += w * a.z; o[3] += w * a.w;
        o[4] += w * b.x; o[5] += w * b.y; o[6] += w * b.z; o[7] += w * b.w;
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint4 v;
    v.x = pack2<T>(o[0] * inv, o[1] * inv);
    v.y = pack2<T>(o[2] * inv, o[3] * inv);
    v.z = pack2<T>(o[4] * inv, o[5] * inv);
    v.w = pack2<T>(o[6] * inv, o[7] * inv);
    *reinterpret_cast<uint4*>(static_cast<T*>(p.o) + ((size_t)me.req * p.num_heads + h) * mla::DC +
                              d0) = v;
    if (d0 == 0 && p.lse) {
      const float lse2 = W > 0.f ? M + log2f(W) : kNegInfF;
      p.lse[(size_t)me.req * p.num_heads + h] = p.lse_base_e ? lse2 * kLn2f : lse2;
    }
  }
}


template <typename T>
__global__ void __launch_bounds__(mla::THREADS, 1) mla_decode_kernel(const MlaParams p) {
  using namespace dev;
  using namespace mla_detail;
  __shared__ __align__(8) uint64_t bars[2 * mla::NSTAGES];
  __shared__ int abort_flag_s;
  __shared__ int merge_last_s;
  __shared__ uint32_t bad_rows_s[mla::NSTAGES];
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t smem = smem_u32(base);
  const uint32_t full0 = smem_u32(&bars[0]);
  const uint32_t empty0 = smem_u32(&bars[mla::NSTAGES]);
  volatile int* abort_flag = &abort_flag_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int item = blockIdx.x / p.gslices;
  const int gs = blockIdx.x - item * p.gslices;
  const WorkItem it = p.items[item];  // within the capacity in CUDA-graph mode
  if (p.item_count && item >= *p.item_count) return;  // CUDA-graph mode: past the work list
  const int g0 = gs * mla::HT;
  const int gcnt = min(mla::HT, p.num_heads - g0);
  int j0 = 0, ntiles = 0;
  if (it.tok_end > it.tok_begin) {
    j0 = (it.tok_begin - it.chunk_tok0) / mla::TS;
    ntiles = (it.tok_end - it.chunk_tok0 + mla::TS - 1) / mla::TS - j0;
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < mla::NSTAGES; ++s) {
      mbar_init(full0 + 8 * s, mla::NPW * 32 + 1);  // the producers' cp.async arrivals + 1
      mbar_init(empty0 + 8 * s, mla::NW);  // one per consumer warp
    }
    abort_flag_s = ((*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  // peers' copies and arrivals reach this CTA's barriers only after their init
  __syncthreads();
  if (abort_flag_s) ntiles = 0;  // an earlier launch timed out: do nothing, write nothing

  if (warp >= mla::NW)
    produce<T>(p, it, j0, ntiles, smem, full0, empty0, abort_flag, lane, warp - mla::NW,
               bad_rows_s);
  else
    consume<T>(p, it, j0, ntiles, gs, g0, gcnt, base, smem, full0, empty0, abort_flag,
               &merge_last_s, bad_rows_s);
}

}  // namespace pkd
