// decode_kernels.cuh -- batch decode attention over a paged KV cache, sm_103a.
//
// What one CTA computes (FlashInfer attention API page, BatchDecodeWithPagedKVCacheWrapper,
// plan()/run()): one task -- a chunk of one output row's KV tokens for one kv head and one
// slice of its qo-head group -- that is, the attention of the slice's qo heads (GQA: qo head g
// reads kv head g / group) over the chunk's attended tokens: s_t = soft_cap(sm_scale * <q, k_t>),
// online softmax, o = sum p_t v_t.  Tasks are launched longest first; the hardware hands each
// free CTA slot the next one.
//
// Structure (one CTA = NW consumer warps + 1 producer warp):
//   producer  streams the chunk tile by tile (TS tokens per tile) with 4-D TMA tensor loads:
//             one box per (page, 128-byte column block, K|V), the page id read from the CSR
//             `indices`; the box lands 128-byte swizzled in a shared-memory stage; completion
//             is an mbarrier transaction count.  NSTAGES stages ring between producer and
//             consumers (full / empty mbarriers, every wait bounded).
//   consumers each own 16 tokens of every tile and keep their own online-softmax state.
//             Tensor-core variant: S^T = K_tile * Q^T with mma.m16n8k16 (16 tokens on M, 8
//             qo heads on N, head_dim on K), the P^T operand built in registers with
//             movmatrix, O^T += V_tile^T * P^T (ldmatrix.trans).  CUDA-core variant: lanes
//             own head_dim slices, dot products are finished with a 31-shuffle
//             reduce-scatter over 32 (token, head) pairs, P*V with fp32 FMAs.
//   epilogue  merges the warps' states in shared memory (the idle pipeline stages) and writes
//             either the final o / lse or an fp32 partial (normalised o, base-2 lse); the CTA
//             that finishes a split unit's last chunk merges the unit's partials.
// Slots past a request's last token and pages outside the chunk are loaded or left stale;
// their logits are replaced by -inf (a select, so NaN/Inf garbage cannot leak) and their V
// rows are zeroed or skipped before P*V.
#pragma once

#include <type_traits>

#include "pkd_device.cuh"
#include "pkd_internal.h"

namespace pkd {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
// Largest log2 headroom a running softmax reference may lag behind the scores (p <= 2^8).
constexpr float kLazyMax = 8.f;

template <typename TQ, bool KV_FP8, int D, int TS, int NSTAGES>
struct DecodeGeom {
  static constexpr int NW = TS / 16;  // consumer warps; each owns 16 tokens of a tile
  static constexpr int NCONS = NW * 32;
  static constexpr int THREADS = NCONS + 32;
  static constexpr int KV_ELT = KV_FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * KV_ELT;
  static constexpr int NBLK = ROW_BYTES / 128;  // 128-byte column blocks per K/V row
  static constexpr int BOX_ELEMS = 128 / KV_ELT;
  static constexpr int TILE_BYTES = TS * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  // the epilogue's image of every warp's state, in the stages once they are idle
  static constexpr int EPI_BYTES = NW * (kSlotHeads * D + 2 * kSlotHeads) * 4;
  static constexpr int PIPE_BYTES = NSTAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = PIPE_BYTES + 1024;
  static_assert(ROW_BYTES % 128 == 0, "K/V rows must be whole 128-byte blocks");
  static_assert(TS % 16 == 0 && NW >= 1 && NW <= 8, "tile of 16-token warp slices");
  static_assert(EPI_BYTES <= PIPE_BYTES, "the epilogue's image fits in the pipeline stages");
};

// Shared memory of the ROPE_LLAMA kernels, after the pipeline stages.  A "pair" is two
// consecutive rotation frequencies of one lane's MMA operand slots (D/4 pairs); an entry is
// their two phasors as {cos half2, sin half2} (8 bytes).
//   R: 16 rows j of D/4 entries: the rotation by tok(j) * rate, where tok(j) is the token (in
//      the warp's 16-token slice) that S^T row j holds.  Built once per CTA.
//   E: per consumer warp, two buffers of D/4 entries: the rotation by (q_pos - t_w) * rate
//      for the warp's current slice starting at token t_w.  Rebuilt every tile.
// RoPE's score depends only on the difference of the two positions, so q rotated by
// (q_pos - t_w) and the key of slice row j rotated by tok(j) give the logit of the key at
// t_w + tok(j): the per-tile angles are the warp's, not each token's.
template <int D, int NW>
struct RopeGeom {
  static constexpr int PAIRS = D / 4;
  static constexpr int ROW = PAIRS * 8;  // bytes of an R row or an E buffer
  static constexpr int R_BYTES = 16 * ROW;
  static constexpr int BYTES = R_BYTES + NW * 2 * ROW;
  static_assert(ROW >= 128, "the row swizzle flips bit 6 of an offset inside the row");
};

struct BlockCoords {
  DecodeTask it;
  int kvh;    // kv head
  int g0;     // first qo head of this task
  int gcnt;   // qo heads of this task
  int gs;     // which slice of the kv head's qo-head group
  int j0;     // first tile (relative to the chunk start)
  int ntiles;
};

template <int TS, int HEADS>
__device__ __forceinline__ BlockCoords task_coords(const DecodeParams& p) {
  BlockCoords b;
  b.it = p.tasks[blockIdx.x];
  b.kvh = b.it.kvh;
  b.gs = b.it.gs;
  b.g0 = b.kvh * p.group + b.gs * HEADS;
  b.gcnt = min(HEADS, p.group - b.gs * HEADS);
  if (b.it.tok_end > b.it.tok_begin) {
    b.j0 = (b.it.tok_begin - b.it.chunk_tok0) / TS;
    b.ntiles = (b.it.tok_end - b.it.chunk_tok0 + TS - 1) / TS - b.j0;
  } else {
    b.j0 = 0;
    b.ntiles = 0;
  }
  return b;
}

// ------------------------------------------------------------------------------ producer
template <class G, int TS, int NSTAGES>
__device__ __forceinline__ void produce(const DecodeParams& p, const BlockCoords& b, uint32_t smem,
                                        uint32_t full0, uint32_t empty0, volatile int* abort_flag,
                                        int lane) {
  using namespace dev;
  const int ps = p.page_size;
  const int br = ps < TS ? ps : TS;  // rows per box: a whole page, or a tile inside a page
  const int boxes = TS / br;
  const uint32_t tx_per_box = 2u * G::NBLK * br * 128u;
  const uint64_t pol = policy_evict_first();
  if (lane == 0) {
    prefetch_tmap(&p.tmap_k);
    prefetch_tmap(&p.tmap_v);
  }
  int issued = 0;
  bool ok = true, bad_page = false;
  for (int i = 0; i < b.ntiles; ++i) {
    const int s = i % NSTAGES;
    // one decision per warp: a lane that gave up takes the whole warp out of the loop
    if (i >= NSTAGES && !__all_sync(~0u, mbar_wait(empty0 + 8 * s, ((i / NSTAGES) - 1) & 1,
                                                   abort_flag, p.wait_ns))) {
      ok = false;
      break;
    }
    const int t0 = b.it.chunk_tok0 + (b.j0 + i) * TS;
    const int bt0 = t0 + lane * br;
    const bool need = lane < boxes && bt0 < b.it.tok_end && bt0 + br > b.it.tok_begin;
    int pid = 0;
    if (need) pid = __ldg(p.indices + b.it.page_base + bt0 / ps);
    bad_page |= need && (uint32_t)pid >= p.num_pages;
    const unsigned m = __ballot_sync(0xffffffffu, need);
    if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * s, __popc(m) * tx_per_box);
    __syncwarp();
    if (need) {
      const int slot0 = bt0 % ps;
      const int c1 = p.hnd ? slot0 : b.kvh;
      const int c2 = p.hnd ? b.kvh : slot0;
      const uint32_t kdst = smem + s * G::STAGE_BYTES + lane * br * 128;
#pragma unroll
      for (int blk = 0; blk < G::NBLK; ++blk) {
        tma_load_4d(kdst + blk * TS * 128, &p.tmap_k, blk * G::BOX_ELEMS, c1, c2, pid,
                    full0 + 8 * s, pol);
        tma_load_4d(kdst + G::TILE_BYTES + blk * TS * 128, &p.tmap_v, blk * G::BOX_ELEMS, c1, c2,
                    pid, full0 + 8 * s, pol);
      }
    }
    issued = i + 1;
  }
  // A page id outside the pool: reported, and its box read as zeros (the tensor map's bounds).
  if (__any_sync(~0u, bad_page) && lane == 0) atomicOr(p.status, kStatusBadPage);
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(p.status, kStatusTimeout);
  }
  // The producer warp stays until the copies of the last NSTAGES tiles it issued have landed
  // (an earlier tile's stage was reused only after its copies landed), so the CTA never exits
  // with a copy in flight into its shared memory -- also when the consumers gave up after the
  // last tile was issued.  These waits keep the full limit whatever the launch's wait_ns.
  if (lane == 0) {
    volatile int never = 0;
    for (int u = issued - NSTAGES < 0 ? 0 : issued - NSTAGES; u < issued; ++u)
      mbar_wait(full0 + 8 * (u % NSTAGES), (u / NSTAGES) & 1, &never);
  }
}

// ------------------------------------------------------------------------------ epilogue
// Shared-memory image of the consumer warps' states, in the idle pipeline stages: acc[w][g][d]
// (unnormalised, relative to m[w][g]), m[w][g] (base-2 running max), l[w][g] (sum of
// exp2(s - m)).
template <int D>
struct EpiView {
  float* acc;
  float* m;
  float* l;
  __device__ __forceinline__ EpiView(uint8_t* base, int nw) {
    acc = reinterpret_cast<float*>(base);
    m = acc + nw * kSlotHeads * D;
    l = m + nw * kSlotHeads;
  }
};

// Combines every warp's state and writes the task's final o / lse, or its fp32 partial.
template <typename TQ, int D, int NW>
__device__ __forceinline__ void store_task(const DecodeParams& p, const BlockCoords& b,
                                           const EpiView<D>& e, int tid) {
  using namespace dev;
  constexpr int NCONS = NW * 32;
  constexpr int D8 = D / 8;
  for (int u = tid; u < b.gcnt * D8; u += NCONS) {
    const int g = u / D8;
    const int d0 = (u - g * D8) * 8;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, e.m[w * kSlotHeads + g]);
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = 0.f;
    float L = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = fast_exp2(e.m[w * kSlotHeads + g] - M);
        L += f * e.l[w * kSlotHeads + g];
        const float4* a = reinterpret_cast<const float4*>(e.acc + (w * kSlotHeads + g) * D + d0);
        const float4 a0 = a[0], a1 = a[1];
        o[0] += f * a0.x; o[1] += f * a0.y; o[2] += f * a0.z; o[3] += f * a0.w;
        o[4] += f * a1.x; o[5] += f * a1.y; o[6] += f * a1.z; o[7] += f * a1.w;
      }
    }
    const float inv = L > 0.f ? p.v_scale / L : 0.f;
    const float lse2 = L > 0.f ? M + log2f(L) : kNegInf;
    const int qo = b.g0 + g;
    if (b.it.out_slot < 0) {
      uint4 v;
      v.x = pack2<TQ>(o[0] * inv, o[1] * inv);
      v.y = pack2<TQ>(o[2] * inv, o[3] * inv);
      v.z = pack2<TQ>(o[4] * inv, o[5] * inv);
      v.w = pack2<TQ>(o[6] * inv, o[7] * inv);
      TQ* dst = reinterpret_cast<TQ*>(p.o) + ((size_t)b.it.req * p.num_qo_heads + qo) * D + d0;
      *reinterpret_cast<uint4*>(dst) = v;
      if (d0 == 0 && p.lse) p.lse[(size_t)b.it.req * p.num_qo_heads + qo] = lse2 * kLn2;
    } else {
      float* dst = p.part_o + ((size_t)b.it.out_slot * kSlotHeads + g) * D + d0;
      reinterpret_cast<float4*>(dst)[0] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
      reinterpret_cast<float4*>(dst)[1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
      if (d0 == 0) p.part_lse[(size_t)b.it.out_slot * kSlotHeads + g] = lse2;
    }
  }
}

// merge_states, fused: the CTA that finishes the last chunk of a split (row, kv head, slice)
// unit combines all its chunks' partials, in chunk order: M = max lse_c, w_c = 2^(lse_c - M),
// o = sum w_c o_c / sum w_c, lse = M + log2 sum w_c.  Writers publish their partial with a
// fence before counting; the last one fences again, reads the partials from L2 and resets the
// counter for the next run of the plan.  No CTA waits for another.
template <typename TQ, int D, int NCONS>
__device__ __forceinline__ void merge_unit(const DecodeParams& p, const BlockCoords& b, int tid,
                                           volatile int* last_flag) {
  using namespace dev;
  constexpr int D8 = D / 8;
  // the CTA's partial stores are ordered before thread 0's fence by the barrier; one fence
  // then publishes them all before the count
  named_bar_sync(1, NCONS);
  if (tid == 0) {
    __threadfence();
    uint32_t* ctr = p.counters + b.it.merge_idx;
    const uint32_t prev = atomicAdd(ctr, 1u);
    const int last = (prev + 1u == (uint32_t)p.merges[b.it.merge_idx].n_chunks) ? 1 : 0;
    if (last) {
      *ctr = 0u;
      __threadfence();  // the other chunks' partials are visible to this CTA's reads below
    }
    *last_flag = last;
  }
  named_bar_sync(1, NCONS);
  if (!*last_flag) return;
  const MergeEntry me = p.merges[b.it.merge_idx];
  const int hq = p.num_qo_heads;
  for (int u = tid; u < b.gcnt * D8; u += NCONS) {
    const int g = u / D8;
    const int d0 = (u - g * D8) * 8;
    // Loads go four chunks at a time, independent of each other, so a merge costs about two
    // L2 round trips; the sums still run in chunk order.
    constexpr int U = 4;
    float M = kNegInf;
    for (int c0 = 0; c0 < me.n_chunks; c0 += U) {
      float l[U];
#pragma unroll
      for (int j = 0; j < U; ++j)
        l[j] = c0 + j < me.n_chunks
                   ? __ldcg(p.part_lse + (size_t)(me.first_slot + c0 + j) * kSlotHeads + g)
                   : kNegInf;
#pragma unroll
      for (int j = 0; j < U; ++j) M = fmaxf(M, l[j]);
    }
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = 0.f;
    float L = 0.f;
    if (M != kNegInf) {
      for (int c0 = 0; c0 < me.n_chunks; c0 += U) {
        float l[U];
        float4 a[U][2];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const bool in = c0 + j < me.n_chunks;
          const size_t row = (size_t)(me.first_slot + (in ? c0 + j : 0)) * kSlotHeads + g;
          const float4* src = reinterpret_cast<const float4*>(p.part_o + row * D + d0);
          l[j] = in ? __ldcg(p.part_lse + row) : kNegInf;
          a[j][0] = __ldcg(src);
          a[j][1] = __ldcg(src + 1);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
          if (c0 + j >= me.n_chunks) break;
          const float f = fast_exp2(l[j] - M);
          L += f;
          o[0] = fmaf(f, a[j][0].x, o[0]); o[1] = fmaf(f, a[j][0].y, o[1]);
          o[2] = fmaf(f, a[j][0].z, o[2]); o[3] = fmaf(f, a[j][0].w, o[3]);
          o[4] = fmaf(f, a[j][1].x, o[4]); o[5] = fmaf(f, a[j][1].y, o[5]);
          o[6] = fmaf(f, a[j][1].z, o[6]); o[7] = fmaf(f, a[j][1].w, o[7]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4 v;
    v.x = pack2<TQ>(o[0] * inv, o[1] * inv);
    v.y = pack2<TQ>(o[2] * inv, o[3] * inv);
    v.z = pack2<TQ>(o[4] * inv, o[5] * inv);
    v.w = pack2<TQ>(o[6] * inv, o[7] * inv);
    const int qo = b.g0 + g;
    TQ* dst = reinterpret_cast<TQ*>(p.o) + ((size_t)me.req * hq + qo) * D + d0;
    *reinterpret_cast<uint4*>(dst) = v;
    if (d0 == 0 && p.lse)
      p.lse[(size_t)me.req * hq + qo] = L > 0.f ? (M + log2f(L)) * kLn2 : kNegInf;
  }
}

// ------------------------------------------------------------------------------ score
// tanh(x) = 1 - 2 / (e^(2x) + 1): one ex2.approx and one reciprocal.  Saturates to +-1 for
// large |x| (e^(2x) overflows to inf, or underflows to 0); near 0 its absolute error is a few
// 1e-7, far below what the soft-capped logits need.
__device__ __forceinline__ float tanh_via_exp2(float x) {
  const float e = dev::fast_exp2(x * 2.8853900817779268f);  // 2 * log2(e)
  return 1.f - __fdividef(2.f, e + 1.f);
}

// The logit in base-2 units: dot * scale_qk (sm_scale and the calibration scales, times
// log2 e, or divided by the cap) plus the ALiBi bias in the same units, then the soft cap.
__device__ __forceinline__ float score_log2(float dot, float scale_qk, float bias, float cap_log2) {
  const float x = fmaf(dot, scale_qk, bias);
  return cap_log2 > 0.f ? cap_log2 * tanh_via_exp2(x) : x;
}

// ALiBi slope of a qo head, in score units (0 without ALiBi).
template <int D>
__device__ __forceinline__ float alibi_slope(const DecodeParams& p, int qo_head) {
  return p.alibi ? __ldg(p.pos_table + 2 * D + qo_head) : 0.f;
}

// ROPE_LLAMA rotation pairs.  Pair P (of D/4) is slot pair P % 2 of k-step block P / 2 =
// kk * 4 + tig: lane tig's MMA k slots {2tig, 2tig+1} (pair 0) or {2tig+8, 2tig+9} (pair 1) of
// k step kk < D/32, which hold dims f, f + 1, and in k step kk + D/32 their rotation partners
// f + D/2, f + D/2 + 1.  PERM: the e4m3 slot order (four consecutive dims per lane).
template <bool PERM>
__device__ __forceinline__ int rope_pair_freq(int P) {
  const int blk = P >> 1, h = P & 1, kk = blk >> 2, tig = blk & 3;
  return PERM ? kk * 16 + tig * 4 + 2 * h : kk * 16 + tig * 2 + 8 * h;
}

// Table entry of the rotation by t * rate for dims f and f + 1: {cos of both, sin of both} as
// fp16 pairs.  rates[f] = {rate hi, rate lo}.
__device__ __forceinline__ uint2 rope_entry(float t, const float2* rates, int f) {
  using namespace dev;
  const float2 r0 = __ldg(rates + f), r1 = __ldg(rates + f + 1);
  float s0, c0, s1, c1;
  rope_sincos(t, r0.x, r0.y, s0, c0);
  rope_sincos(t, r1.x, r1.y, s1, c1);
  return make_uint2(pack2<__half>(c0, c1), pack2<__half>(s0, s1));
}

// Byte offset of pair P's entry in R row j.  The lanes of one shared-memory phase read rows
// j and j + 1 (g_row 2m and 2m + 1) at the same pairs, so odd rows swap the 64-byte halves of
// every 128 bytes.
template <int D>
__device__ __forceinline__ uint32_t rope_r_off(int j, int P) {
  return (uint32_t)(j * (D / 4) * 8 + (((P >> 1) * 16) ^ ((j & 1) << 6)) + (P & 1) * 8);
}

__device__ __forceinline__ void sts_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

// A warp's E buffer for its slice starting at token t_w: the rotation by (q_pos - t_w) * rate,
// entry P at byte 8P.  Followed by __syncwarp: every lane reads every lane's entries.
template <int D, bool PERM>
__device__ __forceinline__ void rope_build_e(uint32_t ebuf, const float2* rates, float dt, int lane) {
#pragma unroll
  for (int P = lane; P < D / 4; P += 32) sts_v2(ebuf + P * 8, rope_entry(dt, rates, rope_pair_freq<PERM>(P)));
  __syncwarp();
}

// ROPE_LLAMA on a K fragment register pair: x holds two dims of a token, y their partners
// (+ D/2), both fp16 after the widening; (c, s) the phasors of the two dims.
template <typename TIN>
__device__ __forceinline__ void rope_k(uint32_t& x, uint32_t& y, uint32_t c, uint32_t s) {
  using namespace dev;
  if constexpr (std::is_same<TIN, __nv_bfloat16>::value) {
    const float2 fx = unpack2<__nv_bfloat16>(x), fy = unpack2<__nv_bfloat16>(y);
    x = pack2<__half>(fx.x, fx.y);
    y = pack2<__half>(fy.x, fy.y);
  }
  rot_h2(x, y, c, s);
}

// ------------------------------------------------------------------------------ tensor core
// Loads the B fragments of Q^T (mma k = head_dim, n = 8 qo heads) for this lane.  For e4m3
// KV the MMA runs in fp16: q is scaled by 2^-qexp (exact) so it fits fp16's range; the
// caller multiplies the scores back by 2^qexp.
// With PERM (the e4m3 path), the 16 head_dim values of k-step kk are assigned to the MMA's k
// slots so that lane tig's four slots {2tig, 2tig+1, 2tig+8, 2tig+9} hold d = kk*16 + 4tig ..
// kk*16 + 4tig + 3: the matching K bytes are then one 32-bit load.  A dot product does not
// depend on the order of its terms, so K and Q only have to agree.
// With ROPE the fragments hold q unrotated, in fp16: the consumers rotate them tile by tile
// (the two halves of a rotation pair sit in k steps kk and kk + D/32 of the same lane).  The
// scaling keeps |q| * 2^-qexp below 2^15, so a rotated component stays below 2^15.5.
template <typename TQ, typename T, int D, bool PERM = false, bool ROPE = false>
__device__ __forceinline__ void load_q_frags(const DecodeParams& p, const BlockCoords& b, int lane,
                                             uint32_t (&qb)[D / 16][2], float& qmul) {
  using namespace dev;
  const int g = lane >> 2, tig = lane & 3;
  const int off0 = PERM ? tig * 4 : tig * 2;      // d of slot pair 0 within the k-step
  const int off1 = PERM ? tig * 4 + 2 : tig * 2 + 8;  // d of slot pair 1
  const bool live = g < b.gcnt;
  const TQ* qrow = reinterpret_cast<const TQ*>(p.q) +
                   ((size_t)b.it.req * p.num_qo_heads + b.g0 + (live ? g : 0)) * D;
  qmul = 1.f;
  if constexpr (!ROPE && std::is_same<TQ, T>::value) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qb[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + off0) : 0u;
      qb[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + off1) : 0u;
    }
  } else {
    float2 f[D / 16][2];
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t raw =
            live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + (h ? off1 : off0)) : 0u;
        f[kk][h] = unpack2<TQ>(raw);
      }
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        amax = fmaxf(amax, fmaxf(fabsf(f[kk][h].x), fabsf(f[kk][h].y)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, off));
    int qexp = 0;
    if (amax > 16384.f) qexp = ilogbf(amax) - 13;  // keeps |q| * 2^-qexp below 2^15
    const float down = exp2f(static_cast<float>(-qexp));
    qmul = exp2f(static_cast<float>(qexp));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) qb[kk][h] = pack2<T>(f[kk][h].x * down, f[kk][h].y * down);
  }
}

// The e4m3 tensor-core path never widens a tile in shared memory.  Instead it reorders the
// MMA operands so that every lane's operand bytes are contiguous:
//   * tokens: row j of S^T (= k slot j of P^T) holds token perm_tok(j) of the warp's slice,
//     chosen so that lane tig's k slots {2tig, 2tig+1, 2tig+8, 2tig+9} are tokens
//     tig, tig+4, tig+8, tig+12 (and the eight S^T rows a K load touches fall in eight
//     different swizzle phases, so those loads are free of bank conflicts);
//   * head_dim: rows r and r+8 of O^T block mb = 4q + jj hold d = d0(r, q) + 2jj and
//     d0(r, q) + 2jj + 1, where d0(r, q) = 128(q/2) + 16 vchunk(r, q%2) + 8(r%2) and
//     vchunk(r, p) = 4((r/2)%2) + r/4 + 2p.  So lane r reads bytes d0 .. d0 + 7 of each of its
//     four tokens (one 64-bit load) and builds the V^T fragments with two byte permutes per
//     block.  The chunk order puts the four rows a half-warp reads (tokens tig + 4t4, whose
//     swizzle phases are 0..3 or 4..7) on eight distinct 16-byte positions of the 128-byte
//     swizzle pattern, so the V loads are free of bank conflicts too.
// Every e4m3 value is an fp16 value, so the widening (cvt.f16x2.e4m3x2) is exact.
__device__ __forceinline__ int perm_tok(int j) {
  return ((j & 7) >> 1) + 4 * (j & 1) + 8 * (j >> 3);
}

// Fills the CTA's R table (see RopeGeom) with the consumer threads; the caller synchronises
// them before the first read.
template <int D, bool PERM>
__device__ __forceinline__ void rope_build_r(uint32_t rtab, const float2* rates, int tid, int nthreads) {
  constexpr int PAIRS = D / 4;
  for (int idx = tid; idx < 16 * PAIRS; idx += nthreads) {
    const int j = idx / PAIRS, P = idx - j * PAIRS;
    const int tok = PERM ? perm_tok(j) : j;
    sts_v2(rtab + rope_r_off<D>(j, P), rope_entry((float)tok, rates, rope_pair_freq<PERM>(P)));
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// d index held by accumulator row `row` (0..15) of O^T block mb.
template <bool KV_FP8>
__device__ __forceinline__ int acc_dim(int mb, int row) {
  if constexpr (KV_FP8) {
    const int r = row & 7, q = mb >> 2;
    return 128 * (q >> 1) + 16 * (4 * ((r >> 1) & 1) + (r >> 2) + 2 * (q & 1)) + 8 * (r & 1) +
           2 * (mb & 3) + (row >> 3);
  } else {
    return mb * 16 + row;
  }
}

// One k-step pair of S^T = K * Q^T under ROPE_LLAMA: a / h are the K fragments of k steps kk
// and kk + D/32 (dims f and their partners f + D/2), qx / qy the raw q fragments of the same
// steps.  q is rotated by the slice's E entries (at address e), the K rows a and b by their R
// entries (row a at address r, row b eight rows further); then the two MMAs in fp16.
template <typename TIN, int D>
__device__ __forceinline__ void rope_qk_step(float (&c)[4], float (&c2)[4], uint32_t (&a)[4],
                                             uint32_t (&h)[4], const uint32_t (&qx)[2],
                                             const uint32_t (&qy)[2], uint32_t e, uint32_t r) {
  using namespace dev;
  const uint4 ev = lds_v4(e);
  const uint4 ra = lds_v4(r), rb = lds_v4(r + 8 * (D / 4) * 8);
  uint32_t q0 = qx[0], q1 = qx[1], p0 = qy[0], p1 = qy[1];
  rot_h2(q0, p0, ev.x, ev.y);  // slot pair 0 (dims f, f + 1)
  rot_h2(q1, p1, ev.z, ev.w);  // slot pair 1
  rope_k<TIN>(a[0], h[0], ra.x, ra.y);
  rope_k<TIN>(a[1], h[1], rb.x, rb.y);
  rope_k<TIN>(a[2], h[2], ra.z, ra.w);
  rope_k<TIN>(a[3], h[3], rb.z, rb.w);
  mma_16816<__half>(c, a, q0, q1);
  mma_16816<__half>(c2, h, p0, p1);
}

// ROPE: per tile, q is rotated by the warp slice's E entries and each K row by its R entries
// (the two halves of a rotation pair are k steps kk and kk + D/32 of the same lane), in fp16
// arithmetic, so QK runs in fp16; P*V keeps V's type.
template <typename TQ, bool KV_FP8, int D, int TS, int NSTAGES, bool ROPE = false>
__device__ __forceinline__ void consume_tc(const DecodeParams& p, const BlockCoords& b, uint32_t smem,
                                           uint32_t full0, uint32_t empty0, volatile int* abort_flag,
                                           int warp, int lane, float (&m2)[2], float (&lsum)[2],
                                           float (&acc)[D / 16][4]) {
  using namespace dev;
  using T = typename std::conditional<KV_FP8, __half, TQ>::type;      // P*V operand type
  using TQK = typename std::conditional<KV_FP8 || ROPE, __half, TQ>::type;  // QK operand type
  using G = DecodeGeom<TQ, KV_FP8, D, TS, NSTAGES>;
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;  // P as bf16 hi + lo
  uint32_t qb[D / 16][2];
  float qmul;
  load_q_frags<TQ, TQK, D, KV_FP8, ROPE>(p, b, lane, qb, qmul);
  const float scale_qk = p.scale_qk * qmul;
  const float cap_log2 = p.cap_log2;
  const int g_row = lane >> 2, tig = lane & 3;
  // tokens (within the warp's 16-token slice) of this lane's two S^T rows
  const int tok_a = KV_FP8 ? perm_tok(g_row) : g_row;
  const int tok_b = KV_FP8 ? perm_tok(g_row + 8) : g_row + 8;
  // ALiBi slopes of this lane's two C columns (qo heads g0 + 2tig, + 1; dead columns of a
  // partial head slice read the last live head's slope, their results are discarded)
  const float slope0 = alibi_slope<D>(p, b.g0 + min(2 * tig, b.gcnt - 1));
  const float slope1 = alibi_slope<D>(p, b.g0 + min(2 * tig + 1, b.gcnt - 1));
  // ROPE: this warp's E buffers and the lane's R entries (rows g_row and g_row + 8; odd rows
  // swap 64-byte halves, so an even k step kk reads at base + swz + 64kk, an odd one at
  // base - swz + 64kk)
  using RG = RopeGeom<D, G::NW>;
  const float2* rope_rates = reinterpret_cast<const float2*>(p.pos_table);
  const uint32_t rope_r = smem + G::PIPE_BYTES;
  const uint32_t rope_e = rope_r + RG::R_BYTES + warp * 2 * RG::ROW;
  const uint32_t rope_swz = (uint32_t)(g_row & 1) << 6;
  const uint32_t rope_ra = rope_r + g_row * RG::ROW + tig * 16;
  // e4m3 path: this lane's byte offsets inside a stage tile, with the 128-byte swizzle of the
  // row already folded in (a chunk index is then applied with one XOR).  K: rows tok_a, tok_b,
  // bytes 4tig.. of each 16-byte chunk.  V: rows tig + 4*t4, bytes 8*(g_row&1).. of chunk
  // vchunk(g_row, q4 % 2) of each 128-byte block (odd q4: chunk ^ 2, i.e. offset bit 5 flips).
  uint32_t koff_a = 0, koff_b = 0, voff[4] = {0, 0, 0, 0};
  if constexpr (KV_FP8) {
    const int ra = warp * 16 + tok_a, rb = warp * 16 + tok_b;
    koff_a = (uint32_t)(ra * 128 + tig * 4) ^ (uint32_t)((ra & 7) << 4);
    koff_b = (uint32_t)(rb * 128 + tig * 4) ^ (uint32_t)((rb & 7) << 4);
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
      const int row = warp * 16 + tig + 4 * t4;
      const int vchunk = 4 * ((g_row >> 1) & 1) + (g_row >> 2);  // vchunk(g_row, 0)
      voff[t4] = (uint32_t)(row * 128 + ((vchunk ^ (row & 7)) << 4) + (g_row & 1) * 8);
    }
  }

  for (int i = 0; i < b.ntiles; ++i) {
    const int s = i % NSTAGES;
    const int t_w = b.it.chunk_tok0 + (b.j0 + i) * TS + warp * 16;  // first token of my slice
    // ROPE: the slice's q rotation, while the stage may still be loading
    if constexpr (ROPE)
      rope_build_e<D, KV_FP8>(rope_e + (i & 1) * RG::ROW, rope_rates, (float)(b.it.q_pos - t_w), lane);
    if (!__all_sync(~0u, mbar_wait(full0 + 8 * s, (i / NSTAGES) & 1, abort_flag, p.wait_ns))) {
      *abort_flag = 1;  // warp-uniform: the warp leaves the loop together
      atomicOr(p.status, kStatusTimeout);
      break;
    }
    const int vlo = max(0, b.it.tok_begin - t_w);
    const int vhi = min(16, b.it.tok_end - t_w);
    const uint32_t ktile = stage_after_wait(smem + s * G::STAGE_BYTES);
    uint32_t vtile = ktile + G::TILE_BYTES;
    const int r0 = warp * 16;  // first tile row of my slice
    bool wrote_stage = false;
    if (vhi > vlo) {
      const bool partial = vlo > 0 || vhi < 16;
      if constexpr (!KV_FP8) {
        if (partial) {
          // Zero the V rows this slice does not attend, so 0 * garbage cannot reach O.
          constexpr int CPR = D / 8;  // 16-byte chunks per 16-bit row
          for (int idx = lane; idx < 16 * CPR; idx += 32) {
            const int r = idx / CPR;
            if (r < vlo || r >= vhi) {
              const uint32_t a = vtile + swz_off(r0 + r, idx - r * CPR, TS);
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
            }
          }
          wrote_stage = true;
          __syncwarp();
          vtile = stage_after_wait(vtile);  // V reads come after the zeroing stores
        }
      }
      // ---- S^T = K * Q^T : rows = 16 tokens, cols = 8 qo heads.  Even and odd k steps go to
      // two accumulators, halving the chain of dependent MMAs.
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV_FP8) {
        // rows tok_a / tok_b; k slots as in load_q_frags<PERM>: four consecutive e4m3 bytes
        const uint32_t ka = ktile + koff_a, kb = ktile + koff_b;
        auto load_k = [&](int kk, uint32_t (&a)[4]) {
          const uint32_t blk = (kk >> 3) * TS * 128;  // 128-byte column block of the chunk
          const uint32_t wa = lds_u32((ka ^ ((kk & 7) << 4)) + blk);
          const uint32_t wb = lds_u32((kb ^ ((kk & 7) << 4)) + blk);
          e4m3x4_to_half2x2(wa, a[0], a[2]);
          e4m3x4_to_half2x2(wb, a[1], a[3]);
        };
        if constexpr (ROPE) {
          const uint32_t eb = rope_e + (i & 1) * RG::ROW + tig * 16;
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t a[4], h[4];  // k steps kk and kk + D/32: dims f and f + D/2
            load_k(kk, a);
            load_k(kk + D / 32, h);
            rope_qk_step<__half, D>(c, c2, a, h, qb[kk], qb[kk + D / 32], eb + kk * 64,
                                    rope_ra + ((kk & 1) ? -rope_swz : rope_swz) + kk * 64);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            load_k(kk, a);
            mma_16816<TQK>((kk & 1) ? c2 : c, a, qb[kk][0], qb[kk][1]);
          }
        }
      } else {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int csel = lane >> 4;
        if constexpr (ROPE) {
          // ldmatrix: a[0] / a[2] are row g_row (token tok_a), dims 16kk + 2tig (+1) and
          // 16kk + 8 + 2tig (+1); a[1] / a[3] the same dims of row g_row + 8 (tok_b)
          const uint32_t eb = rope_e + (i & 1) * RG::ROW + tig * 16;
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t a[4], h[4];
            ldsm_x4(ktile + swz_off(r0 + row, kk * 2 + csel, TS), a);
            ldsm_x4(ktile + swz_off(r0 + row, (kk + D / 32) * 2 + csel, TS), h);
            rope_qk_step<TQ, D>(c, c2, a, h, qb[kk], qb[kk + D / 32], eb + kk * 64,
                                rope_ra + ((kk & 1) ? -rope_swz : rope_swz) + kk * 64);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(ktile + swz_off(r0 + row, kk * 2 + csel, TS), a);
            mma_16816<TQK>((kk & 1) ? c2 : c, a, qb[kk][0], qb[kk][1]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] += c2[e];
      // ---- online softmax over the 16 tokens, per qo-head column
      float sc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = e >= 2 ? tok_b : tok_a;
        const float bias = ((e & 1) ? slope1 : slope0) * (float)(t_w + t - b.it.q_pos);
        const float sv = score_log2(c[e], scale_qk, bias, cap_log2);
        sc[e] = (t >= vlo && t < vhi) ? sv : kNegInf;
      }
      // The reference m2 of a column only moves when one of its scores exceeds it by more
      // than kLazyMax: until then p = 2^(s - m2) <= 2^kLazyMax, far inside the 16-bit P
      // operand's range, and o = acc / l and lse = m2 + log2(l) are unchanged by the choice
      // of m2.  Most tiles thus skip the cross-lane max and the rescale of O.
      const bool grow = sc[0] > m2[0] + kLazyMax || sc[2] > m2[0] + kLazyMax ||
                        sc[1] > m2[1] + kLazyMax || sc[3] > m2[1] + kLazyMax;
      if (__any_sync(~0u, grow)) {
        float alpha[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = fmaxf(sc[j], sc[j + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 16));
          const float mnew = fmaxf(m2[j], mx);
          const float ref = mnew == kNegInf ? 0.f : mnew;
          alpha[j] = fast_exp2(m2[j] - ref);
          sc[j] = fast_exp2(sc[j] - ref);
          sc[j + 2] = fast_exp2(sc[j + 2] - ref);
          lsum[j] = lsum[j] * alpha[j] + sc[j] + sc[j + 2];
          m2[j] = mnew;
        }
        // rescale O only when some column's reference moved (alpha is exactly 1 otherwise)
        if (__any_sync(~0u, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int mb = 0; mb < D / 16; ++mb) {
            acc[mb][0] *= alpha[0];
            acc[mb][1] *= alpha[1];
            acc[mb][2] *= alpha[0];
            acc[mb][3] *= alpha[1];
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float ref = m2[j] == kNegInf ? 0.f : m2[j];
          sc[j] = fast_exp2(sc[j] - ref);
          sc[j + 2] = fast_exp2(sc[j + 2] - ref);
          lsum[j] += sc[j] + sc[j + 2];
        }
      }
      // ---- P^T as the B operand (k = token, n = qo head): transpose the C fragment.  A
      // bf16 P keeps only 8 significant bits: its rounding error, 2^-9 of each weight, can
      // exceed the output tolerance where a few large weights cancel.  So with bf16 V the
      // weights go in as P_hi + P_lo (the bf16 value and its bf16 rounding remainder, one more
      // MMA per block), which carries ~16 bits; fp16 P (11 bits) goes in alone.
      const uint32_t h01 = pack2<T>(sc[0], sc[1]), h23 = pack2<T>(sc[2], sc[3]);
      const uint32_t b0 = movmatrix_trans(h01);
      const uint32_t b1 = movmatrix_trans(h23);
      uint32_t b0_lo = 0u, b1_lo = 0u;
      if constexpr (kSplitP) {
        const float2 r01 = unpack2<T>(h01), r23 = unpack2<T>(h23);
        b0_lo = movmatrix_trans(pack2<T>(sc[0] - r01.x, sc[1] - r01.y));
        b1_lo = movmatrix_trans(pack2<T>(sc[2] - r23.x, sc[3] - r23.y));
      }
      // ---- O^T += V^T * P^T : rows = head_dim (16 per block), cols = 8 qo heads
      if constexpr (KV_FP8) {
        uint32_t va[4], vb[4];  // even / odd q4
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          va[t4] = vtile + voff[t4];
          vb[t4] = va[t4] ^ 32u;  // vchunk(g_row, 1) = vchunk(g_row, 0) ^ 2
        }
#pragma unroll
        for (int q4 = 0; q4 < D / 64; ++q4) {
          // bytes d0(g_row, q4) .. +7 of tokens tig + 4*t4 (zero if not attended)
          uint2 w[4];
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4)
            w[t4] = lds_v2(((q4 & 1) ? vb[t4] : va[t4]) + (q4 >> 1) * TS * 128);
          if (partial) {
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              const int tok = tig + 4 * t4;
              if (tok < vlo || tok >= vhi) w[t4] = make_uint2(0u, 0u);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t sel = (jj & 1) ? 0x7362u : 0x5140u;  // bytes (b, b') of two words
            const uint32_t x01 = prmt(jj >> 1 ? w[0].y : w[0].x, jj >> 1 ? w[1].y : w[1].x, sel);
            const uint32_t x23 = prmt(jj >> 1 ? w[2].y : w[2].x, jj >> 1 ? w[3].y : w[3].x, sel);
            uint32_t a[4];
            e4m3x4_to_half2x2(x01, a[0], a[1]);  // d = c0 / c0 + 1, tokens tig, tig+4
            e4m3x4_to_half2x2(x23, a[2], a[3]);  // d = c0 / c0 + 1, tokens tig+8, tig+12
            mma_16816<T>(acc[4 * q4 + jj], a, b0, b1);
          }
        }
      } else {
        const int row = (lane & 7) + (lane >> 4) * 8;
        const int csel = (lane >> 3) & 1;
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) {
          uint32_t a[4];
          ldsm_x4_trans(vtile + swz_off(r0 + row, mb * 2 + csel, TS), a);
          mma_16816<T>(acc[mb], a, b0, b1);
          if constexpr (kSplitP) mma_16816<T>(acc[mb], a, b0_lo, b1_lo);
        }
      }
    }
    if (wrote_stage) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

// A tensor-core warp's state into its own slot of the epilogue image.  Lane (row r = lane / 4,
// tig = lane % 4) holds columns 2 tig, 2 tig + 1 (qo heads) of every O^T block; m2 is the same
// on the 8 lanes of a column, lsum their partial sums.
template <int D, bool KV_FP8>
__device__ __forceinline__ void stash_tc(const EpiView<D>& e, int warp, int lane,
                                             float (&m2)[2], float (&lsum)[2],
                                             float (&acc)[D / 16][4]) {
  const int gr = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = lsum[j];
    l += __shfl_xor_sync(~0u, l, 4);
    l += __shfl_xor_sync(~0u, l, 8);
    l += __shfl_xor_sync(~0u, l, 16);
    if (gr == 0) {
      e.m[warp * kSlotHeads + tig * 2 + j] = m2[j];
      e.l[warp * kSlotHeads + tig * 2 + j] = l;
    }
  }
  float* a = e.acc + warp * kSlotHeads * D;
#pragma unroll
  for (int mb = 0; mb < D / 16; ++mb) {
    const int da = acc_dim<KV_FP8>(mb, gr), db = acc_dim<KV_FP8>(mb, gr + 8);
    a[(tig * 2) * D + da] = acc[mb][0];
    a[(tig * 2 + 1) * D + da] = acc[mb][1];
    a[(tig * 2) * D + db] = acc[mb][2];
    a[(tig * 2 + 1) * D + db] = acc[mb][3];
  }
}

// ------------------------------------------------------------------------------ CUDA core
// Geometry of the CUDA-core consumers.  A K/V row is split over L lanes: lane sub-index
// h = lane / R owns dims [h*DL, (h+1)*DL), LB bytes of the row read as NU loads ("units") of
// UB = 16 bytes (chunks h*NU .. h*NU + NU - 1) or, when a lane's share is 8 bytes, one
// 8-byte half of chunk h / 2.  One warp instruction covers R = 32 / L rows of the warp's
// 16-token slice and the slice takes NP = 16 / R passes.  L grows with the head group so that
// a lane's accumulators (GP heads x DL dims, V floats) stay at VMAX.  Scores need a reduction
// over only the L lanes of a row; the P*V products stay in the lane that read the row, and
// the lanes of a column are summed once per task.
template <bool KV_FP8, int D, int GP, int NW, bool ROPE>
struct CcGeom {
  static constexpr int ELT = KV_FP8 ? 1 : 2;
  static constexpr int CH = D * ELT / 16;  // 16-byte chunks of a K/V row
  static constexpr int VMAX = 64;          // accumulators per lane the split aims for
  static constexpr int L0 = GP * D / VMAX < 2 ? 2 : GP * D / VMAX;
  static constexpr int L1 = L0 > 32 ? 32 : L0;
  static constexpr int L = L1 > 2 * CH ? 2 * CH : L1;
  static constexpr int R = 32 / L;
  static constexpr int NP = 16 / R;
  static constexpr int LB = D * ELT / L;        // bytes of a row per lane
  static constexpr int UB = LB >= 16 ? 16 : 8;  // bytes per load
  static constexpr int NU = LB / UB;            // loads per lane and row
  static constexpr int EPU = UB / ELT;          // elements per load
  static constexpr int DL = D / L;
  static constexpr int V = GP * DL;
  // Rows of a pass.  The swizzled tile puts chunk c of row r in bank group (c ^ r) & 7.  A
  // shared-memory phase serves 8 lanes' 16-byte loads (or 16 lanes' 8-byte loads, two per
  // chunk), which must hit eight groups.  With R >= 8 they read one chunk of eight
  // consecutive rows.  With R < 8 they hold 8 / R chunk indices, differing in bits HBITS, so
  // their rows take the other bits of r & 7 (RR_MASK) and the passes take HBITS and bit 3
  // (P_MASK).
  static constexpr int HBITS = R >= 8 ? 0 : (8 / R - 1) * (UB == 16 ? NU : 1);
  static constexpr int RR_MASK = R >= 8 ? R - 1 : (7 & ~HBITS);
  static constexpr int P_MASK = R >= 8 ? (15 & ~(R - 1)) : (8 | HBITS);
  // q as fp32 [GP][L][DL]: each lane's DL dims of a head in a block of DL / 4 16-byte chunks.
  // A phase reads chunk k of the blocks of up to 8 / R values of h at once; chunk k of block h
  // sits at k ^ QSWZ(h), which puts those reads in different bank groups.
  static constexpr int QB = DL / 4;  // chunks per block
  __host__ __device__ static constexpr int qswz(int h) { return ((h * QB) >> 3) & (QB - 1); }
  // float index of element d of head g
  __host__ __device__ static constexpr int qidx(int g, int d) {
    return (g * L + d / DL) * DL + (((d % DL) / 4) ^ qswz(d / DL)) * 4 + d % 4;
  }
  static constexpr int Q_BYTES = GP * D * 4;
  // Without ROPE: the task's q rows.  With ROPE: each warp's q rotated for its current slice
  // (same layout), then the K rotations by |m| = 0..8 positions (a negative m flips the
  // sine): row |m| holds, per frequency pair (f, f+1), {cos f, cos f+1, sin f, sin f+1} at
  // entry jl * L/2 + hp for f = 2 * (hp * DL/2 + jl), i.e. the lanes' dims blocks hp
  // interleaved so that a phase reads consecutive entries; rows are padded by 16 bytes so
  // that eight rows fall in eight bank groups.
  static constexpr int RT_ROW = D / 2 * 8 + 16;
  static constexpr int RT_OFF = ROPE ? NW * Q_BYTES : 0;
  static constexpr int BYTES = ROPE ? RT_OFF + 9 * RT_ROW : Q_BYTES;
  // Registers per thread, capped so that CTAs of `threads` threads can share an SM: each of
  // its four sub-partitions holds 16384 registers and a CTA's warps are spread over them.
  // Two CTAs per SM where that leaves at least 160 registers and the accumulators fit in
  // VMAX, else one.
  static constexpr int regs_for(int warps_per_sm) {
    return (16384 / ((warps_per_sm + 3) / 4 * 32)) / 8 * 8 > 255
               ? 255
               : (16384 / ((warps_per_sm + 3) / 4 * 32)) / 8 * 8;
  }
  static constexpr int max_regs(int threads) {
    return V <= VMAX && regs_for(2 * threads / 32) >= 160 ? regs_for(2 * threads / 32)
                                                         : regs_for(threads / 32);
  }
  static_assert(NU >= 1 && (NU & (NU - 1)) == 0 && HBITS <= 7 && EPU % 4 == 0, "lane loads");
  static_assert(2 * R * L == 64 && V % (2 * R) == 0, "lane split");
};

// The bits of x placed, in order, at the set bits of a 4-bit mask.
__device__ __forceinline__ int deposit4(int x, int mask) {
  int out = 0, b = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if ((mask >> i) & 1) out |= ((x >> b++) & 1) << i;
  return out;
}

// Byte offset of chunk c of tile row r (128-byte column blocks of TS rows, 128-byte swizzle).
template <int TS>
__device__ __forceinline__ uint32_t cc_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * TS * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// NWD words of K/V widened to fp32 pairs (element 2j, 2j + 1 in pair j).
template <typename TQ, bool KV_FP8, int NWD>
__device__ __forceinline__ void cc_widen(const uint32_t (&v)[NWD],
                                         float2 (&x)[NWD * (KV_FP8 ? 2 : 1)]) {
  using namespace dev;
#pragma unroll
  for (int k = 0; k < NWD; ++k) {
    if constexpr (KV_FP8) {
      x[2 * k] = unpack2<__half>(e4m3x2_to_half2((uint16_t)(v[k] & 0xffffu)));
      x[2 * k + 1] = unpack2<__half>(e4m3x2_to_half2((uint16_t)(v[k] >> 16)));
    } else if constexpr (std::is_same<TQ, __nv_bfloat16>::value) {
      x[k] = make_float2(__uint_as_float(v[k] << 16), __uint_as_float(v[k] & 0xffff0000u));
    } else {
      x[k] = unpack2<__half>(v[k]);
    }
  }
}

// Load u (of NU) of this lane's share of tile row r: UB bytes widened to fp32 pairs (element
// 2j, 2j + 1 in pair j), or zeros if `zero`.  The load is volatile: its values feed plain
// FMAs, so only this keeps it ahead of the stage's release.
template <typename TQ, bool KV_FP8, int TS, int UB, int NU>
__device__ __forceinline__ void cc_load(uint32_t tile, int r, int h, int u, bool zero,
                                        float2 (&x)[UB / (KV_FP8 ? 1 : 2) / 2]) {
  using namespace dev;
  constexpr int NWD = UB / 4;
  uint32_t v[NWD];
  if constexpr (UB == 16) {
    const uint32_t a = tile + cc_chunk<TS>(r, h * NU + u);
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(a));
  } else {
    const uint32_t a = tile + cc_chunk<TS>(r, h >> 1) + (h & 1) * 8;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(a));
  }
#pragma unroll
  for (int k = 0; k < NWD; ++k) v[k] = zero ? 0u : v[k];
  cc_widen<TQ, KV_FP8, NWD>(v, x);
}

__device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// a[i] for a runtime i < N, by selects (no local-memory indexing).
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float v = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) v = i == k ? a[k] : v;
  return v;
}

// The dims block h (as h bits of the lane) of the lane that finishes score x of a batch after
// a reduce-scatter over LOG_LR lane bits 16, 8, ...: level k keeps the upper half (bit
// LOG_X - 1 - k of x) on lanes with bit 4 - k set.
template <int LOG_X, int LOG_LR, int LOG_R>
__device__ __forceinline__ constexpr int hsrc(int x) {
  int h = 0;
  for (int k = 0; k < LOG_LR; ++k) h |= ((x >> (LOG_X - 1 - k)) & 1) << (4 - k - LOG_R);
  return h;
}

__device__ __forceinline__ uint4 lds_v4_vol(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Set-up of a CUDA-core CTA by its consumer threads (tid of nthreads), at `base` as CcGeom
// lays it out: the task's GP q rows in fp32 (rows of heads past the group are zero), or with
// ROPE the K rotation table.
template <typename TQ, bool KV_FP8, int D, int GP, int NW, bool ROPE>
__device__ __forceinline__ void cc_setup(const DecodeParams& p, const BlockCoords& b,
                                         uint8_t* base, int tid, int nthreads) {
  using namespace dev;
  using C = CcGeom<KV_FP8, D, GP, NW, ROPE>;
  if constexpr (!ROPE) {
    float* q = reinterpret_cast<float*>(base);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q);
    for (int idx = tid; idx < GP * D / 2; idx += nthreads) {
      const int g = idx / (D / 2), d = (idx - g * (D / 2)) * 2;
      float2 v = make_float2(0.f, 0.f);
      if (g < b.gcnt)
        v = unpack2<TQ>(__ldg(src + (((size_t)b.it.req * p.num_qo_heads + b.g0 + g) * D + d) / 2));
      q[C::qidx(g, d)] = v.x;
      q[C::qidx(g, d + 1)] = v.y;
    }
  } else {
    const float2* rates = reinterpret_cast<const float2*>(p.pos_table);
    for (int idx = tid; idx < 9 * (D / 4); idx += nthreads) {
      const int k = idx / (D / 4), fp = idx - k * (D / 4);  // row |m| = k; pair 2fp, 2fp+1
      const int hp = fp / (C::DL / 2), jl = fp % (C::DL / 2);
      const float2 r0 = __ldg(rates + 2 * fp), r1 = __ldg(rates + 2 * fp + 1);
      float s0, c0, s1, c1;
      rope_sincos((float)k, r0.x, r0.y, s0, c0);
      rope_sincos((float)k, r1.x, r1.y, s1, c1);
      *reinterpret_cast<float4*>(base + C::RT_OFF + k * C::RT_ROW + (jl * (C::L / 2) + hp) * 16) =
          make_float4(c0, c1, s0, s1);
    }
  }
}

// ROPE: the task's q rows rotated by dt * rate (dt = q_pos minus the middle of the warp's
// slice) into the warp's buffer, in the layout of the q rows (heads past the group are zero).
// Lane handles frequencies f = lane + 32k; q is read from global memory (it stays in L1).
template <typename TQ, bool KV_FP8, int D, int GP, int NW>
__device__ __forceinline__ void cc_rotate_q(const DecodeParams& p, const BlockCoords& b,
                                            float* qr, float dt, int lane) {
  using namespace dev;
  using C = CcGeom<KV_FP8, D, GP, NW, true>;
  const float2* rates = reinterpret_cast<const float2*>(p.pos_table);
  const TQ* q = reinterpret_cast<const TQ*>(p.q) + ((size_t)b.it.req * p.num_qo_heads + b.g0) * D;
  __syncwarp();  // every lane is done reading the previous slice's rotation
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    const int f = lane + 32 * k;
    const float2 r = __ldg(rates + f);
    float s, c;
    rope_sincos(dt, r.x, r.y, s, c);
    const int ox = C::qidx(0, f), oy = C::qidx(0, f + D / 2);
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const bool live = g < b.gcnt;
      const float x = live ? to_float(__ldg(q + g * D + f)) : 0.f;
      const float y = live ? to_float(__ldg(q + g * D + f + D / 2)) : 0.f;
      qr[g * D + ox] = x * c - y * s;
      qr[g * D + oy] = y * c + x * s;
    }
  }
  __syncwarp();
  asm volatile("" ::: "memory");  // the q reads that follow see this slice's rotation
}

// The CUDA-core consumer warp.  For each tile its 16-token slice is taken in NP passes of R
// rows (lane: row rr = lane % R of the pass, dims block h = lane / R), NB passes at a time:
//  - the partial dot products of the lane's rows with its q dims (fp32 pair FMAs), one
//    independent chain per pass and head;
//  - the batch's NB x GP partial sums reduce-scattered over the row's L lanes, so each lane
//    finishes XH scores (no two lanes repeat the softmax work of a score);
//  - the online softmax in base 2 with a lazy reference: m2 moves only when a score exceeds
//    it by more than kLazyMax, so p <= 2^kLazyMax and most batches skip the cross-lane max;
//  - every lane fetches p of its own rows and adds p * V into its own accumulators (rows of a
//    window or chunk edge that are not attended have p = 0 and their V zeroed, so stale
//    values in the stage cannot leak).
// At the end the accumulators are reduce-scattered over the R row lanes of each dims block
// and stored, with m2 and l, into the warp's slot of the epilogue image.
// ROPE: q is rotated per slice to the slice's middle t_w + 8 and each K row by its offset
// row - 8 from there (the partner dims of a rotation pair are on lane ^ 16): the logit
// depends only on the difference of the two positions.
// Returns false when a pipeline wait gave up (the CTA's consumers then leave together).
template <typename TQ, bool KV_FP8, int D, int TS, int NSTAGES, int GP, bool ROPE>
__device__ __forceinline__ bool consume_cc(const DecodeParams& p, const BlockCoords& b,
                                           uint32_t smem, uint8_t* smem_p, uint32_t full0,
                                           uint32_t empty0, volatile int* abort_flag, int warp,
                                           int lane, const EpiView<D>& epi) {
  using namespace dev;
  using G = DecodeGeom<TQ, KV_FP8, D, TS, NSTAGES>;
  using C = CcGeom<KV_FP8, D, GP, G::NW, ROPE>;
  constexpr int L = C::L, R = C::R, NP = C::NP, NU = C::NU, EPU = C::EPU, DL = C::DL;
  constexpr int V2 = C::V / 2;  // fp32 pairs of accumulators
  // passes taken together (independent chains in flight), as many as registers allow
  constexpr int NB0 = (ROPE ? 8 : 16) / GP < 1 ? 1 : (ROPE ? 8 : 16) / GP;
  constexpr int NB = NB0 < NP ? NB0 : NP;
  constexpr int X = NB * GP;            // scores a lane holds partial sums of, per batch
  constexpr int LR = X < L ? X : L;     // lanes a row's scores are scattered over
  constexpr int XH = X / LR;            // scores a lane finishes
  constexpr int LOG_X = ilog2(X), LOG_LR = ilog2(LR), LOG_R = ilog2(R);
  static_assert((X & (X - 1)) == 0 && (1 << LOG_R) == R, "powers of two");
  const int rr = lane % R, h = lane / R;
  const int rowbase = deposit4(rr, C::RR_MASK);
  float* qs = reinterpret_cast<float*>(smem_p + G::PIPE_BYTES);
  float* qr = reinterpret_cast<float*>(smem_p + G::PIPE_BYTES) + warp * (C::Q_BYTES / 4);
  const uint32_t qlane_s = smem_u32((ROPE ? qr : qs) + h * DL);
  const int qswz_h = C::qswz(h);
  const uint8_t* rt = smem_p + G::PIPE_BYTES + C::RT_OFF + (h % (L / 2)) * 16;
  const float send_sign = h >= L / 2 ? -1.f : 1.f;
  const float scale_qk = p.scale_qk;
  const float cap_log2 = p.cap_log2;

  float m2[GP];
  float2 acc[GP][DL / 2];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m2[g] = kNegInf;
#pragma unroll
    for (int k = 0; k < DL / 2; ++k) acc[g][k] = make_float2(0.f, 0.f);
  }
  // the scores this lane finishes: batch entries x = xb + j (pass x / GP, head x % GP), the
  // same for every batch; their running sums of p
  int xb = 0;
#pragma unroll
  for (int k = 0; k < LOG_LR; ++k) xb |= ((lane >> (4 - k)) & 1) << (LOG_X - 1 - k);
  int hg[XH], hdep[XH];
  float hslope[XH], lsum_h[XH];
#pragma unroll
  for (int j = 0; j < XH; ++j) {
    hg[j] = (xb + j) % GP;
    hdep[j] = deposit4((xb + j) / GP, C::P_MASK);
    hslope[j] = alibi_slope<D>(p, b.g0 + min(hg[j], b.gcnt - 1));
    lsum_h[j] = 0.f;
  }

  for (int i = 0; i < b.ntiles; ++i) {
    const int s = i % NSTAGES;
    const int t_w = b.it.chunk_tok0 + (b.j0 + i) * TS + warp * 16;  // first token of my slice
    if constexpr (ROPE)
      cc_rotate_q<TQ, KV_FP8, D, GP, G::NW>(p, b, qr, (float)(b.it.q_pos - t_w - 8), lane);
    if (!__all_sync(~0u, mbar_wait(full0 + 8 * s, (i / NSTAGES) & 1, abort_flag, p.wait_ns))) {
      *abort_flag = 1;  // warp-uniform: the warp leaves the loop together
      atomicOr(p.status, kStatusTimeout);
      break;
    }
    const int vlo = max(0, b.it.tok_begin - t_w);
    const int vhi = min(16, b.it.tok_end - t_w);
    const uint32_t ktile = stage_after_wait(smem + s * G::STAGE_BYTES);
    const uint32_t vtile = ktile + G::TILE_BYTES;
    if (vlo < vhi) {  // warp-uniform
      const bool partial = vlo > 0 || vhi < 16;
#pragma unroll 1
      for (int pb = 0; pb < NP; pb += NB) {  // a batch of NB passes
        int row[NB];
        bool valid[NB];
#pragma unroll
        for (int pp = 0; pp < NB; ++pp) {
          row[pp] = rowbase | deposit4(pb + pp, C::P_MASK);
          valid[pp] = row[pp] >= vlo && row[pp] < vhi;
        }
        // ---- the lane's partial dot products for every pass (independent chains), with each
        // q chunk read once and used by all passes
        float2 s2[NB][GP];
#pragma unroll
        for (int pp = 0; pp < NB; ++pp)
#pragma unroll
          for (int g = 0; g < GP; ++g) s2[pp][g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < NU; ++c) {
          float2 kf[NB][EPU / 2];
#pragma unroll
          for (int pp = 0; pp < NB; ++pp) {
            cc_load<TQ, KV_FP8, TS, C::UB, NU>(ktile, warp * 16 + row[pp], h, c, false, kf[pp]);
            if constexpr (ROPE) {
              // offset m = row - 8 from the slice's middle: table row |m|; a negative m flips
              // the sine, folded into the value the partner sends
              const int am = row[pp] < 8 ? 8 - row[pp] : row[pp] - 8;
              const float sf = row[pp] < 8 ? -send_sign : send_sign;
              const uint8_t* tr = rt + am * C::RT_ROW + c * EPU / 2 * (L / 2) * 16;
#pragma unroll
              for (int j = 0; j < EPU / 2; ++j) {
                const float4 t = *reinterpret_cast<const float4*>(tr + j * (L / 2) * 16);
                const float2 ks = __fmul2_rn(kf[pp][j], make_float2(sf, sf));
                float2 kp;
                kp.x = __shfl_xor_sync(~0u, ks.x, 16);
                kp.y = __shfl_xor_sync(~0u, ks.y, 16);
                kf[pp][j] = __ffma2_rn(kp, make_float2(t.z, t.w),
                                       __fmul2_rn(kf[pp][j], make_float2(t.x, t.y)));
              }
            }
          }
#pragma unroll
          for (int g = 0; g < GP; ++g) {
#pragma unroll
            for (int j = 0; j < EPU / 4; ++j) {
              const uint4 t = lds_v4_vol(qlane_s + (g * D + ((c * EPU / 4 + j) ^ qswz_h) * 4) * 4);
              const float2 q01 = make_float2(__uint_as_float(t.x), __uint_as_float(t.y));
              const float2 q23 = make_float2(__uint_as_float(t.z), __uint_as_float(t.w));
#pragma unroll
              for (int pp = 0; pp < NB; ++pp) {
                s2[pp][g] = __ffma2_rn(kf[pp][2 * j], q01, s2[pp][g]);
                s2[pp][g] = __ffma2_rn(kf[pp][2 * j + 1], q23, s2[pp][g]);
              }
            }
          }
        }
        // ---- scores: the batch's NB x GP partial sums reduce-scattered over the row's L
        // lanes (lane bits 16, 8, ... first), so each lane finishes XH of them; the online
        // softmax runs on those, and every lane then fetches the p of its own rows
        float d[X];
#pragma unroll
        for (int pp = 0; pp < NB; ++pp)
#pragma unroll
          for (int g = 0; g < GP; ++g) d[pp * GP + g] = s2[pp][g].x + s2[pp][g].y;
#pragma unroll
        for (int k = 0; k < LOG_LR; ++k) {
          const int o = 16 >> k, n = X >> k;
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < n / 2; ++i) {
            const float send = up ? d[i] : d[i + n / 2];
            const float keep = up ? d[i + n / 2] : d[i];
            d[i] = keep + __shfl_xor_sync(~0u, send, o);
          }
        }
#pragma unroll
        for (int o = R; o < 32 / LR; o <<= 1)
#pragma unroll
          for (int j = 0; j < XH; ++j) d[j] += __shfl_xor_sync(~0u, d[j], o);
        const int pbdep = deposit4(pb, C::P_MASK);
        float sc[XH], m2h[XH];
        bool grow = false;
#pragma unroll
        for (int j = 0; j < XH; ++j) {
          const int hrow = rowbase | pbdep | hdep[j];
          const float bias = hslope[j] * (float)(t_w + hrow - b.it.q_pos);
          sc[j] = hrow >= vlo && hrow < vhi ? score_log2(d[j], scale_qk, bias, cap_log2) : kNegInf;
          m2h[j] = pick<GP>(m2, hg[j]);
          grow |= sc[j] > m2h[j] + kLazyMax;
        }
        if (__any_sync(~0u, grow)) {
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            float mx = kNegInf;
#pragma unroll
            for (int j = 0; j < XH; ++j) mx = hg[j] == g ? fmaxf(mx, sc[j]) : mx;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, o));
            if (mx > m2[g]) {  // warp-uniform: every lane holds the same maximum
              const float alpha = fast_exp2(m2[g] - mx);
#pragma unroll
              for (int j = 0; j < XH; ++j) lsum_h[j] = hg[j] == g ? lsum_h[j] * alpha : lsum_h[j];
              const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
              for (int k = 0; k < DL / 2; ++k) acc[g][k] = __fmul2_rn(acc[g][k], a2);
              m2[g] = mx;
            }
          }
#pragma unroll
          for (int j = 0; j < XH; ++j) m2h[j] = pick<GP>(m2, hg[j]);
        }
        float prh[XH];
#pragma unroll
        for (int j = 0; j < XH; ++j) {
          prh[j] = fast_exp2(sc[j] - (m2h[j] == kNegInf ? 0.f : m2h[j]));
          lsum_h[j] += prh[j];
        }
        float pr[NB][GP];
#pragma unroll
        for (int pp = 0; pp < NB; ++pp)
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const int x = pp * GP + g;
            pr[pp][g] = __shfl_sync(~0u, prh[x % XH], rr | (hsrc<LOG_X, LOG_LR, LOG_R>(x) << LOG_R));
          }
        // ---- p * V
#pragma unroll
        for (int c = 0; c < NU; ++c) {
#pragma unroll
          for (int pp = 0; pp < NB; ++pp) {
            float2 vf[EPU / 2];
            cc_load<TQ, KV_FP8, TS, C::UB, NU>(vtile, warp * 16 + row[pp], h, c,
                                               partial && !valid[pp], vf);
#pragma unroll
            for (int g = 0; g < GP; ++g) {
              const float2 p2 = make_float2(pr[pp][g], pr[pp][g]);
#pragma unroll
              for (int j = 0; j < EPU / 2; ++j)
                acc[g][c * EPU / 2 + j] = __ffma2_rn(p2, vf[j], acc[g][c * EPU / 2 + j]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  // every consumer is done with the stages; one shared decision whether any wait gave up
  if (named_bar_or(1, G::NCONS, *abort_flag != 0)) return false;

  // ---- into the epilogue image: l summed over the rows (every dims block holds the same
  // sums); the accumulators reduce-scattered over the row lanes, after which lane rr holds
  // pairs rr * SEG .. rr * SEG + SEG - 1 of its block's flattened [GP][DL / 2] array
  // each score was finished by L / LR lanes (the ones differing in the lane bits below the
  // scatter); count the copy with those bits zero
  const bool counted = ((lane >> LOG_R) & (L / LR - 1)) == 0;
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    float l = 0.f;
#pragma unroll
    for (int j = 0; j < XH; ++j) l += counted && hg[j] == g ? lsum_h[j] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(~0u, l, o);
    if (lane == 0) {
      epi.m[warp * kSlotHeads + g] = m2[g];
      epi.l[warp * kSlotHeads + g] = l;
    }
  }
  float2 a[V2];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int k = 0; k < DL / 2; ++k) a[g * (DL / 2) + k] = acc[g][k];
#pragma unroll
  for (int o = R / 2, n = V2; o >= 1; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float2 send = up ? a[k] : a[k + n / 2];
      const float2 keep = up ? a[k + n / 2] : a[k];
      a[k].x = keep.x + __shfl_xor_sync(~0u, send.x, o);
      a[k].y = keep.y + __shfl_xor_sync(~0u, send.y, o);
    }
  }
  constexpr int SEG = V2 / R;
#pragma unroll
  for (int k = 0; k < SEG; ++k) {
    const int n = rr * SEG + k;
    const int g = n / (DL / 2), j = (n % (DL / 2)) * 2;
    *reinterpret_cast<float2*>(epi.acc + (warp * kSlotHeads + g) * D + h * DL + j) = a[k];
  }
  return true;
}

// ------------------------------------------------------------------------------ kernel
// KIND: kTensorCore (HEADS = 8 qo heads per task) or kCudaCore (HEADS = GP).  ROPE: ROPE_LLAMA
// applied to q and K.  CTA blockIdx.x runs task blockIdx.x.
template <typename TQ, bool KV_FP8, int D, int TS, int NSTAGES, int KIND, int GP, bool ROPE = false>
__global__ void __launch_bounds__(DecodeGeom<TQ, KV_FP8, D, TS, NSTAGES>::THREADS,
                                  KIND == kTensorCore ? 2 : 1)
    __maxnreg__((KIND == kTensorCore ? 255
                                     : CcGeom<KV_FP8, D, GP, TS / 16, ROPE>::max_regs(TS / 16 * 32 + 32)))
    decode_paged_kernel(const __grid_constant__ DecodeParams p) {
  using namespace dev;
  using G = DecodeGeom<TQ, KV_FP8, D, TS, NSTAGES>;
  constexpr int HEADS = KIND == kTensorCore ? 8 : GP;
  __shared__ __align__(8) uint64_t bars[2 * NSTAGES];
  __shared__ int abort_flag_s;
  __shared__ int merge_last_s;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem_p =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t smem = smem_u32(smem_p);
  const uint32_t full0 = smem_u32(&bars[0]);
  const uint32_t empty0 = smem_u32(&bars[NSTAGES]);
  volatile int* abort_flag = &abort_flag_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Programmatic dependent launch: this grid may have been started while the previous kernel
  // in the stream was still running.  The next kernel may start its own launch as soon as
  // every CTA of this one is running.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The work list (and its count) came with the plan's upload, a copy that the stream orders
  // before this launch, so the CTA reads its task and sets up its barriers while the previous
  // kernel may still run.  CUDA-graph mode: the grid is cut for a fixed work-list capacity;
  // CTAs past this plan's tasks have nothing to do (the whole CTA leaves at once).
  if (p.task_count != nullptr && (int)blockIdx.x >= *p.task_count) return;
  const BlockCoords b = task_coords<TS, HEADS>(p);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, G::NW);
    }
    fence_mbar_init();
  }
  // Everything else (q, the page table, the pools, the status word and the shared partial
  // slots and counters) is read or written only after the previous kernel has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0)
    abort_flag_s = (*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) ? 1 : 0;
  __syncthreads();
  if (abort_flag_s) return;  // an earlier launch timed out: touch nothing

  if (warp == G::NW) {
    produce<G, TS, NSTAGES>(p, b, smem, full0, empty0, abort_flag, lane);
    return;
  }
  const EpiView<D> epi(smem_p, G::NW);
  if constexpr (KIND == kTensorCore) {
    if constexpr (ROPE) {
      rope_build_r<D, KV_FP8>(smem + G::PIPE_BYTES, reinterpret_cast<const float2*>(p.pos_table),
                              threadIdx.x, G::NCONS);
      named_bar_sync(2, G::NCONS);
    }
    float m2[2] = {kNegInf, kNegInf}, lsum[2] = {0.f, 0.f};
    float acc[D / 16][4];
#pragma unroll
    for (int mb = 0; mb < D / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
    consume_tc<TQ, KV_FP8, D, TS, NSTAGES, ROPE>(p, b, smem, full0, empty0, abort_flag, warp,
                                                 lane, m2, lsum, acc);
    // every consumer is done with the stages; one shared decision whether any wait gave up
    if (named_bar_or(1, G::NCONS, *abort_flag != 0)) return;
    stash_tc<D, KV_FP8>(epi, warp, lane, m2, lsum, acc);
  } else {
    cc_setup<TQ, KV_FP8, D, GP, G::NW, ROPE>(p, b, smem_p + G::PIPE_BYTES, threadIdx.x, G::NCONS);
    named_bar_sync(2, G::NCONS);
    if (!consume_cc<TQ, KV_FP8, D, TS, NSTAGES, GP, ROPE>(p, b, smem, smem_p, full0, empty0,
                                                          abort_flag, warp, lane, epi))
      return;
  }
  named_bar_sync(1, G::NCONS);
  store_task<TQ, D, G::NW>(p, b, epi, threadIdx.x);
  if (b.it.out_slot >= 0) merge_unit<TQ, D, G::NCONS>(p, b, threadIdx.x, &merge_last_s);
}

// ------------------------------------------------------------------------------ registry
template <typename TQ, bool KV_FP8, int D, int TS, int NSTAGES, int KIND, int GP, bool ROPE = false>
DecodeKernel make_decode_kernel(int q_dtype, int kv_dtype) {
  using G = DecodeGeom<TQ, KV_FP8, D, TS, NSTAGES>;
  DecodeKernel k;
  k.kind = KIND;
  k.q_dtype = q_dtype;
  k.kv_dtype = kv_dtype;
  k.head_dim = D;
  k.heads_per_cta = KIND == kTensorCore ? 8 : GP;
  k.fn = reinterpret_cast<const void*>(
      &decode_paged_kernel<TQ, KV_FP8, D, TS, NSTAGES, KIND, GP, ROPE>);
  k.rope = ROPE ? 1 : 0;
  k.nstages = NSTAGES;
  k.threads = G::THREADS;
  k.smem_bytes = G::SMEM_BYTES + (KIND == kTensorCore
                                      ? (ROPE ? RopeGeom<D, G::NW>::BYTES : 0)
                                      : CcGeom<KV_FP8, D, GP, G::NW, ROPE>::BYTES);
  k.tile_tokens = TS;
  return k;
}

}  // namespace pkd
