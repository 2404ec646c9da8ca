// mla_tc_kernels.cuh -- MLA paged decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// sm_103a.  Same operation as mla_kernels.cuh (FlashInfer attention API page, flashinfer.mla /
// BatchMLAPagedAttentionWrapper): logit = sm_scale * (<q_nope, ckv_t> + <q_pe, kpe_t>), value
// ckv_t, for 128 query heads per CTA pair.
//
// Why a CTA pair: one SM's tensor memory (512 columns x 128 lanes of fp32) holds O for 128
// heads x 512 dims and nothing else, so the two CTAs of a cluster split the work by feature:
//   CTA 0 holds q_nope[:, 0:256], loads ckv[t, 0:256] and owns O[:, 0:256];
//   CTA 1 holds q_nope[:, 256:512] and q_pe, loads ckv[t, 256:512] and kpe[t], owns O[:, 256:512].
// Each CTA's logit MMA gives a partial S over its features; the two partials are exchanged
// through distributed shared memory (one bulk shared-to-shared copy per tile) and added
// (a + b == b + a exactly, so both CTAs hold the same S, the same softmax and the same P), and
// each CTA multiplies P by the value columns it loaded itself.  Every byte of the caches is
// read once, by one CTA.
//
// Roles (416 threads):
//   warps 0-3  softmax: thread h owns head h (TMEM lane h).  The exchange runs two tiles
//              ahead of the softmax (S is triple-buffered in TMEM), so its latency hides behind
//              the softmax of the tiles in between.  Online softmax with a lazy reference (O in
//              TMEM is rescaled only when the running maximum grows by more than 2^8); P goes to
//              TMEM as a 16-bit value and its rounding remainder (P_hi + P_lo), so the 16-bit
//              rounding of P costs no accuracy.  Epilogue through shared memory (coalesced
//              stores) and the fused merge of split requests.
//   warps 4-7, 9-12  producer: 16-byte cp.async gathers of the token rows (any page size; a TMA
//              request per row is rate-bound for rows this small), zero-filled for tokens
//              outside the item and for page ids outside the caches, into NST stages laid out
//              as the MMA's 128-byte-swizzled K-major blocks (8 rows x 128 bytes per atom).  It
//              starts before Q is loaded.
//   warp 8     MMA issuer (one thread) and TMEM owner: S = Q K^T as M=128 x N=32 MMAs over
//              16-feature steps, issued two tiles ahead of O += P V (four M=128 x N=256 MMAs,
//              A = P_hi / P_lo from TMEM, V read MN-major from the same stage blocks).
//              tcgen05.commit signals the softmax (S ready, PV done) and the producer (stage
//              free).
// Every wait is bounded; a timeout sets the status word and the kernel runs on without waiting
// (the output is then not written).  No CTA leaves before its peer (cluster barrier).
#pragma once

#include <type_traits>

#include "pkd_device.cuh"
#include "pkd_internal.h"

namespace pkd {

namespace mlatc {

constexpr int DC = 512;
constexpr int DP = 64;
constexpr int HT = 128;                       // heads per CTA: the MMA's M
constexpr int TS = 32;                        // tokens per tile: the logit MMA's N
constexpr int NST = 4;                        // pipeline stages
constexpr int QBLK = 5;                       // 64-feature blocks held by CTA 1 (CTA 0: 4)
constexpr int QBLK_BYTES = HT * 128;          // 16384
constexpr int BLK_BYTES = TS * 128;           // 4096: one 64-feature block of a tile
constexpr int STAGE_BYTES = QBLK * BLK_BYTES;  // 20480
constexpr int XBUF_BYTES = HT * TS * 4;      // 16384: a partial S tile, 128-byte rows, chunk
                                              // q of head h at chunk q ^ (h & 7)
constexpr int OFF_Q = 0;
constexpr int OFF_STAGE = OFF_Q + QBLK * QBLK_BYTES;         // 81920
constexpr int OFF_XOUT = OFF_STAGE + NST * STAGE_BYTES;      // 143360: my partial, 2 buffers
constexpr int OFF_XIN = OFF_XOUT + 2 * XBUF_BYTES;           // the peer's partials, 2 buffers
constexpr int SMEM_BYTES = OFF_XIN + 2 * XBUF_BYTES + 1024;  // + alignment slack
// epilogue staging (rows of 256 outputs) reuses [OFF_STAGE, ...): stages, then the exchange
constexpr int STAGE_OUT_BYTES = HT * 256 * 4;
constexpr int NSOFT = 128;
constexpr int NPW = 8;                        // producer warps: 4-7 and 9-12 (row pw + 8 k)
constexpr int NPROD = NPW * 32;
constexpr int THREADS = NSOFT + NPROD + 32;
constexpr int TMEM_COLS = 512;
constexpr int TM_S = 0;      // three S buffers: columns [0, 96)
constexpr int TM_PHI = 96;   // P, 16-bit pairs: columns [96, 112)
constexpr int TM_PLO = 112;  // its rounding remainder: columns [112, 128)
constexpr int TM_O = 256;    // O: columns [256, 512)
constexpr float kLazyMax = 8.f;  // log2 growth of the running maximum that forces a rescale
constexpr int kIdTiles = 8;  // the producer loads page ids this many tiles ahead
static_assert(OFF_STAGE % 1024 == 0 && STAGE_BYTES % 1024 == 0 && OFF_XOUT % 1024 == 0 &&
                  OFF_XIN % 1024 == 0,
              "align");
static_assert(OFF_STAGE + STAGE_OUT_BYTES <= OFF_XIN + XBUF_BYTES, "epilogue staging fits");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

// mbarriers
enum {
  B_FULL = 0,                 // [NST] producer -> MMA: stage filled (128 cp.async arrivals)
  B_EMPTY = B_FULL + NST,     // [NST] MMA -> producer: stage read (tcgen05.commit)
  B_SFULL = B_EMPTY + NST,    // [3]   MMA -> softmax: S buffer ready (tcgen05.commit)
  B_PFULL = B_SFULL + 3,      //       softmax -> MMA: P written (128 arrivals)
  B_PVDONE = B_PFULL + 1,     //       MMA -> softmax: P V done (tcgen05.commit)
  B_XFULL = B_PVDONE + 1,     // [2]   the peer's partial S landed (own expect_tx + the
                              //       peer's bulk copy bytes)
  B_XEMPTY = B_XFULL + 2,     // [2]   the peer read the partial I sent (one remote arrival
                              //       per softmax warp)
  B_FINAL = B_XEMPTY + 2,     //       every MMA of the CTA complete
  B_MERGE = B_FINAL + 1,      //       a block of another chunk's partials loaded (merge)
  NBARS = B_MERGE + 1
};

}  // namespace mlatc

namespace mlatc_detail {

using namespace dev;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Relaxed: no cluster-scope fence.  Used only to say "I have read buffer b", after the values
// read have been consumed (so the loads are complete when this issues).
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Wait with cluster-scope acquire (the barrier's arrivals come from the peer CTA).
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) return false;
  }
}

// Bulk copy of `bytes` from this CTA's shared memory into the peer's (cluster addresses for
// the destination and its mbarrier), completing as transaction bytes on that mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src,
                                                  uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// 16-byte global -> shared copy, zero-filled when src_bytes == 0 (nothing is read then).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
      "r"(src_bytes), "l"(policy)
      : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading / stride byte offsets, swizzle
// (2 = 128-byte, 4 = 64-byte), fixed version bits 46-47 = 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)swizzle << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A / B both bf16 (ab = 1) or both
// fp16 (ab = 0), B MN-major when b_mn, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t instr_desc(int m, int n, uint32_t ab, uint32_t b_mn) {
  return (1u << 4) | (ab << 7) | (ab << 10) | (b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with A (M=128 rows x 16 values, two 16-bit values per column) read from TMEM.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace mlatc_detail

template <typename T>
__global__ void __launch_bounds__(mlatc::THREADS, 1) mla_tc_kernel(const MlaParams p) {
  using namespace dev;
  using namespace mlatc;
  using namespace mlatc_detail;
  constexpr float kNegInfF = -__builtin_huge_valf();
  constexpr float kLn2f = 0.6931471805599453f;
  constexpr uint32_t kAB = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  __shared__ __align__(8) uint64_t bars[NBARS];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag_s;
  __shared__ int merge_last_s;
  __shared__ float wself_s[HT], wchunk_s[HT];  // merge weights per head
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(base);
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = &abort_flag_s;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, kStatusTimeout);
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();  // 0: features [0, 256); 1: [256, 512) and the rope part
  const int nblk = rank ? QBLK : QBLK - 1;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int item = blockIdx.x / p.gslices;
  const int gs = blockIdx.x - item * p.gslices;  // head tile * 2 + rank
  const WorkItem it = p.items[item];  // within the capacity in CUDA-graph mode
  // CUDA-graph mode: the grid covers the work list's capacity; both CTAs of a pair hold the
  // same item, so both leave here, before any barrier or tensor-memory use
  if (p.item_count && item >= *p.item_count) return;
  const int H = p.num_heads;
  const int g0 = (gs >> 1) * HT;
  const int gcnt = min(HT, H - g0);
  int j0 = 0, ntiles = 0;
  if (it.tok_end > it.tok_begin) {
    j0 = (it.tok_begin - it.chunk_tok0) / TS;
    ntiles = (it.tok_end - it.chunk_tok0 + TS - 1) / TS - j0;
  }

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_FULL + s), NPROD);
      mbar_init(bar(B_EMPTY + s), 1);
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) mbar_init(bar(B_SFULL + s), 1);
    mbar_init(bar(B_PFULL), NSOFT);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_XFULL), 1);
    mbar_init(bar(B_XFULL + 1), 1);
    mbar_init(bar(B_XEMPTY), NSOFT / 32);
    mbar_init(bar(B_XEMPTY + 1), NSOFT / 32);
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_MERGE), 1);
    abort_flag_s = ((*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (abort_flag_s) ntiles = 0;  // an earlier launch timed out: do nothing, write nothing

  if ((warp >= 4 && warp < 8) || warp >= 9) {
    // ================================================================ producer
    cluster_arrive();  // nothing here depends on the peer: start at once
    const int pw = warp < 8 ? warp - 4 : warp - 5;  // rows pw, pw + NPW, ... of each tile
    const int ps = p.page_size;
    const char* ckv = static_cast<const char*>(p.ckv) + rank * 512;
    const char* kpe = static_cast<const char*>(p.kpe);
    const uint64_t pol = policy_evict_first();
    // Eight warps, not four: the gathers are bound by the copies in flight, and more issuing
    // warps keep more in flight (114.4 us with six warps, 110.2 with eight, 120.6 with four on
    // the batch-114 example).
    // lane r (< 8; lanes 8-31 repeat lanes 0-7): page id of tile row pw + NPW r of tile i, or -1
    // for a row that is not a token of the item (zero-filled).  ids[k] holds tile i + k: the
    // ids of a tile are loaded kIdTiles iterations before its copies.  (An L2 prefetch of the
    // rows a few tiles ahead measured 3 % slower: the gathers are rate-bound per SM, not by
    // DRAM latency.)
    auto page_of = [&](int i) -> int {
      const int r = pw + NPW * (lane & 7);
      const int t = it.chunk_tok0 + (j0 + i) * TS + r;
      return (i < ntiles && r < TS && t >= it.tok_begin && t < it.tok_end)
                 ? __ldg(p.indices + it.page_base + t / ps)
                 : -1;
    };
    int ids[kIdTiles];
#pragma unroll
    for (int k = 0; k < kIdTiles; ++k) ids[k] = page_of(k);
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NST;
      const int64_t pid_mine = ids[0];
#pragma unroll
      for (int k = 0; k + 1 < kIdTiles; ++k) ids[k] = ids[k + 1];
      ids[kIdTiles - 1] = page_of(i + kIdTiles);
      if (i >= NST) {
        int freed = 1;
        if (lane == 0)
          freed = mbar_wait(bar(B_EMPTY + s), (uint32_t)(((i / NST) - 1) & 1), abort_flag) ? 1 : 0;
        if (!__shfl_sync(~0u, freed, 0) && lane == 0) fail();
      }
      const uint32_t stage = sb + OFF_STAGE + s * STAGE_BYTES;
      const int tt0 = it.chunk_tok0 + (j0 + i) * TS;
#pragma unroll
      for (int rr = 0; rr < (TS + NPW - 1) / NPW; ++rr) {
        const int row = pw + NPW * rr;
        if (row >= TS) break;  // the same for every lane
        const int64_t pid = __shfl_sync(~0u, pid_mine, rr);
        const bool ok = pid >= 0 && pid < p.num_pages;
        const int64_t prow = ok ? pid * ps + (tt0 + row) % ps : 0;
        const uint32_t sw = (uint32_t)(row & 7);
        // ckv: lane = 16-byte chunk c of this CTA's 512 bytes (block c / 8)
        cp_async16(stage + (lane >> 3) * BLK_BYTES + row * 128 + (((uint32_t)(lane & 7) ^ sw) << 4),
                   ckv + prow * (DC * 2) + lane * 16, ok ? 16u : 0u, pol);
        if (rank && lane < 8)
          cp_async16(stage + 4 * BLK_BYTES + row * 128 + (((uint32_t)lane ^ sw) << 4),
                     kpe + prow * (DP * 2) + lane * 16, ok ? 16u : 0u, pol);
      }
      cp_async_arrive(bar(B_FULL + s));
    }
    cp_async_wait_all();
    cluster_wait();
  } else {
    // Q part of this CTA -> 128-byte-swizzled K-major blocks (heads past H are zero rows), by
    // the softmax and MMA warps while the producer already streams K; loads are issued in
    // batches of 16 before their stores so their latencies overlap
    {
      constexpr int kQT = NSOFT + 32;
      constexpr int kBatch = 16;
      const int nch = nblk * 8;
      const int tq = warp == 8 ? NSOFT + lane : (int)threadIdx.x;
      for (int k0 = 0; k0 * kQT < HT * QBLK * 8; k0 += kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int u = tq + (k0 + k) * kQT;
          const int h = u / nch, c = u - h * nch;
          const int b = c >> 3, ch = c & 7;
          v[k] = make_uint4(0u, 0u, 0u, 0u);
          if (u < HT * nch && h < gcnt) {
            const size_t row = (size_t)it.req * H + g0 + h;
            const T* src = b < 4 ? static_cast<const T*>(p.q_nope) + row * DC + rank * 256 + b * 64 +
                                       ch * 8
                                 : static_cast<const T*>(p.q_pe) + row * DP + ch * 8;
            v[k] = __ldg(reinterpret_cast<const uint4*>(src));
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int u = tq + (k0 + k) * kQT;
          const int h = u / nch, c = u - h * nch;
          const int b = c >> 3, ch = c & 7;
          if (u < HT * nch)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             sb + OFF_Q + b * QBLK_BYTES + h * 128 + ((ch ^ (h & 7)) << 4)),
                         "r"(v[k].x), "r"(v[k].y), "r"(v[k].z), "r"(v[k].w)
                         : "memory");
        }
      }
    }
    fence_proxy_async_smem();  // Q (generic stores) before the MMAs read it
    cluster_arrive();          // also: both CTAs' barriers initialised before any remote use
    cluster_wait();

    if (warp == 8) {
      // ============================================================== MMA issuer
      if (lane == 0) {
        const uint32_t id_qk = instr_desc(HT, TS, kAB, 0u);
        const uint32_t id_pv = instr_desc(HT, 256, kAB, 1u);
        const uint64_t qdesc0 = smem_desc(sb + OFF_Q, 16, 1024, 2);
        auto qk = [&](int i) {
          const int s = i % NST;
          if (!mbar_wait(bar(B_FULL + s), (uint32_t)((i / NST) & 1), abort_flag)) fail();
          fence_proxy_async_smem();  // the cp.async (generic) writes before the tensor core reads
          tc_fence_after();
          const uint64_t kdesc0 = smem_desc(sb + OFF_STAGE + s * STAGE_BYTES, 16, 1024, 2);
          const uint32_t d = tmem + TM_S + 32 * (i % 3);
          for (int b = 0; b < nblk; ++b)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma(d, qdesc0 + (uint64_t)((b * QBLK_BYTES + kk * 32) >> 4),
                     kdesc0 + (uint64_t)((b * BLK_BYTES + kk * 32) >> 4), id_qk,
                     (b | kk) ? 1u : 0u);
          tc_commit(bar(B_SFULL + i % 3));
        };
        auto pv = [&](int i) {
          if (!mbar_wait(bar(B_PFULL), (uint32_t)(i & 1), abort_flag)) fail();
          tc_fence_after();
          const uint64_t vdesc0 =
              smem_desc(sb + OFF_STAGE + (i % NST) * STAGE_BYTES, 4096, 1024, 2);  // MN-major
          // O += P_hi V + P_lo V: P = P_hi + P_lo to about 2^-17
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
              tc_mma_ts(tmem + TM_O, tmem + (part ? TM_PLO : TM_PHI) + ks * 8,
                        vdesc0 + (uint64_t)(ks * 2048 >> 4), id_pv,
                        (i > 0 || part > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar(B_PVDONE));
          tc_commit(bar(B_EMPTY + i % NST));
        };
        // logits run two tiles ahead of P V (three S buffers)
        if (ntiles > 0) qk(0);
        if (ntiles > 1) qk(1);
        for (int i = 0; i < ntiles; ++i) {
          if (i + 2 < ntiles) qk(i + 2);
          pv(i);
        }
        tc_commit(bar(B_FINAL));
        volatile int never = 0;
        mbar_wait(bar(B_FINAL), 0u, &never);  // every MMA done before TMEM is freed
      }
      __syncwarp();
    } else {
      // ============================================================== softmax (thread = head)
      const int h = threadIdx.x;
      const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
      const uint32_t peer = (uint32_t)(rank ^ 1);
      const uint32_t xrow = (uint32_t)h * 128u, xsw = (uint32_t)(h & 7);
      const uint32_t xin_peer = map_peer(sb + OFF_XIN, peer);
      const uint32_t xfull_peer = map_peer(bar(B_XFULL), peer);
      const uint32_t xempty_peer = map_peer(bar(B_XEMPTY), peer);
      bool ok = true;
      // My partial S of tile j: into v, and into the peer's exchange buffer j % 2, each warp
      // its 32 rows by one bulk copy, once the peer has read what I sent there two tiles ago
      // (which also means those copies have finished reading my buffer j % 2).
      auto send = [&](int j, float (&v)[32]) {
        const uint32_t b = (uint32_t)(j & 1);
        ok &= mbar_wait(bar(B_SFULL + j % 3), (uint32_t)((j / 3) & 1), abort_flag);
        tc_fence_after();
        tmem_ld32(tmem + lane_off + TM_S + 32 * (j % 3), v);
        if (lane == 0 && j >= 2)
          ok &= wait_cluster(bar(B_XEMPTY + b), (uint32_t)(((j >> 1) - 1) & 1), abort_flag);
        __syncwarp();
        const uint32_t xo = sb + OFF_XOUT + b * XBUF_BYTES + xrow;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                           xo + ((((uint32_t)q) ^ xsw) << 4)),
                       "f"(v[4 * q]), "f"(v[4 * q + 1]), "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                       : "memory");
        fence_proxy_async_smem();  // generic stores before the bulk copy reads them
        __syncwarp();
        if (lane == 0) {
          if (h == 0)  // the peer's four copies to me, 16 KB in all
            mbar_arrive_expect_tx(bar(B_XFULL + b), (uint32_t)XBUF_BYTES);
          const uint32_t off = b * XBUF_BYTES + (uint32_t)warp * 32u * 128u;
          bulk_copy_to_peer(xin_peer + off, sb + OFF_XOUT + off, 32u * 128u, xfull_peer + 8 * b);
        }
      };
      float m_ref = kNegInfF, lsum = 0.f;
      float va[32], vb[32];  // my partials of tiles j and j + 1
      if (ntiles > 0) send(0, va);
      if (ntiles > 1) send(1, vb);
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t b = (uint32_t)(j & 1);
        // ---- the peer's partial of tile j
        ok &= mbar_wait(bar(B_XFULL + b), (uint32_t)((j >> 1) & 1), abort_flag);
        const uint32_t xi = sb + OFF_XIN + b * XBUF_BYTES + xrow;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = lds_v4(xi + ((((uint32_t)q) ^ xsw) << 4));
          va[4 * q] += __uint_as_float(w.x);
          va[4 * q + 1] += __uint_as_float(w.y);
          va[4 * q + 2] += __uint_as_float(w.z);
          va[4 * q + 3] += __uint_as_float(w.w);
        }
        // ---- logits, lazy online softmax.  The maximum is taken on the unscaled partial sums
        // (sm_scale > 0 keeps their order, and rounding is monotone, so max(s)·c = max(s·c)), and
        // the scale is folded into the exponent's FMA; only a tile cut by the item's bounds
        // needs the per-token mask.
        const int t0 = it.chunk_tok0 + (j0 + j) * TS;
        if (t0 < it.tok_begin || t0 + TS > it.tok_end) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int t = t0 + e;
            if (t < it.tok_begin || t >= it.tok_end) va[e] = kNegInfF;
          }
        }
        float mq[4] = {va[0], va[1], va[2], va[3]};
#pragma unroll
        for (int e = 4; e < 32; ++e) mq[e & 3] = fmaxf(mq[e & 3], va[e]);
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
        // buffer b read (the values are consumed above): the peer may refill it
        __syncwarp();
        if (lane == 0) arrive_remote_relaxed(xempty_peer + 8 * b);
        float alpha = 1.f;
        bool resc = false;
        if (mx > m_ref + kLazyMax) {  // also the first tile (m_ref = -inf)
          if (m_ref != kNegInfF) {
            alpha = fast_exp2(m_ref - mx);
            resc = true;
          }
          m_ref = mx;
        }
        const float nref = m_ref == kNegInfF ? 0.f : -m_ref;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[16], pl[16];  // P rounded to 16 bits, and the rounding remainder
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float a = fast_exp2(fmaf(va[e], p.scale_log2, nref));
          const float c = fast_exp2(fmaf(va[e + 1], p.scale_log2, nref));
          ps[(e >> 1) & 3] += a + c;
          pk[e >> 1] = pack2<T>(a, c);
          const float2 r = unpack2<T>(pk[e >> 1]);
          pl[e >> 1] = pack2<T>(a - r.x, c - r.y);
        }
        lsum = lsum * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        // ---- P V of the previous tile done: P columns free, O stable
        if (j > 0) ok &= mbar_wait(bar(B_PVDONE), (uint32_t)((j - 1) & 1), abort_flag);
        if (!ok) {
          fail();
          ok = true;
        }
        tc_fence_after();
        if (__any_sync(~0u, resc)) {
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + TM_O + 32 * c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tmem + lane_off + TM_O + 32 * c, o);
          }
        }
        tmem_st16(tmem + lane_off + TM_PHI, pk);
        tmem_st16(tmem + lane_off + TM_PLO, pl);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
        // ---- the exchange two tiles ahead
#pragma unroll
        for (int e = 0; e < 32; ++e) va[e] = vb[e];
        if (j + 2 < ntiles) send(j + 2, vb);
      }

      // ---- epilogue: O / l through shared memory (stages and exchange buffers, now idle)
      if (ntiles > 0) {
        ok &= mbar_wait(bar(B_PVDONE), (uint32_t)((ntiles - 1) & 1), abort_flag);
        tc_fence_after();
      }
      if (h == 0)  // my last copies have landed and been read (their sources are reused here)
        for (int jj = ntiles - 2; jj < ntiles; ++jj)
          if (jj >= 0)
            ok &= wait_cluster(bar(B_XEMPTY + (jj & 1)), (uint32_t)((jj >> 1) & 1), abort_flag);
      if (!ok) fail();
      named_bar_sync(1, NSOFT);
      const bool aborted = *abort_flag != 0;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float lse2 = lsum > 0.f ? m_ref + log2f(lsum) : kNegInfF;
      const bool split = it.out_slot >= 0;
      auto prow_of = [&](int slot, int row) -> size_t {  // [slots, 2 (rank), H] partial rows
        return ((size_t)slot * 2 + rank) * H + g0 + row;
      };
      // row r in 16-byte chunks q at (q & ~7) | ((q ^ r) & 7): conflict-free per warp
      auto swz = [](int q, int r) -> uint32_t { return (uint32_t)((q & ~7) | ((q ^ r) & 7)) << 4; };
      const uint32_t stg = sb + OFF_STAGE;
      const int row_bytes = split ? 1024 : 512;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float o[32];
        if (ntiles > 0) {
          tmem_ld32(tmem + lane_off + TM_O + 32 * c, o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (split) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                             stg + h * row_bytes + swz(c * 8 + k, h)),
                         "f"(o[4 * k] * inv), "f"(o[4 * k + 1] * inv), "f"(o[4 * k + 2] * inv),
                         "f"(o[4 * k + 3] * inv)
                         : "memory");
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             stg + h * row_bytes + swz(c * 4 + k, h)),
                         "r"(pack2<T>(o[8 * k] * inv, o[8 * k + 1] * inv)),
                         "r"(pack2<T>(o[8 * k + 2] * inv, o[8 * k + 3] * inv)),
                         "r"(pack2<T>(o[8 * k + 4] * inv, o[8 * k + 5] * inv)),
                         "r"(pack2<T>(o[8 * k + 6] * inv, o[8 * k + 7] * inv))
                         : "memory");
        }
      }
      named_bar_sync(1, NSOFT);
      const int qrow = row_bytes / 16;
      if (!aborted) {
#pragma unroll 4
        for (int u = h; u < gcnt * qrow; u += NSOFT) {
          const int r = u / qrow, q = u - r * qrow;
          const uint4 v = lds_v4(stg + r * row_bytes + swz(q, r));
          if (split)
            *reinterpret_cast<uint4*>(p.part_o + prow_of(it.out_slot, r) * 256 + q * 4) = v;
          else
            *reinterpret_cast<uint4*>(static_cast<T*>(p.o) + ((size_t)it.req * H + g0 + r) * DC +
                                      rank * 256 + q * 8) = v;
        }
        if (h < gcnt) {
          if (split)
            p.part_lse[prow_of(it.out_slot, h)] = lse2;
          else if (rank == 0 && p.lse)
            p.lse[(size_t)it.req * H + g0 + h] = p.lse_base_e ? lse2 * kLn2f : lse2;
        }
      }
      // ---- fused merge: the CTA finishing a split request's last chunk for its (tile, half)
      if (split) {
        __threadfence();
        named_bar_sync(1, NSOFT);
        if (h == 0) {
          int last = 0;
          if (!aborted) {
            uint32_t* ctr = p.counters + (size_t)it.merge_idx * p.gslices + gs;
            const uint32_t prev = atomicAdd(ctr, 1u);
            last = (prev + 1u == (uint32_t)p.merges[it.merge_idx].n_chunks) ? 1 : 0;
            if (last) *ctr = 0u;
          }
          merge_last_s = last;
        }
        named_bar_sync(1, NSOFT);
        if (merge_last_s) {
          // This CTA's own partial is still in the staging rows (fp32, 1 KB per head).  The
          // other chunks' partials of this (head tile, half) are contiguous rows in global
          // memory: each is brought in 64 heads at a time by one bulk copy into the (now idle)
          // Q area and folded into the staging rows with coalesced shared-memory passes.
          // Every element is summed in slot order, whichever chunk finished last, so repeated
          // launches agree bit for bit: with two chunks, w0 x0 is rounded first and w1 x1
          // added by one fma (the own partial taken from the staging rows); with more, every
          // chunk, the own one included, comes from global memory in slot order.
          __threadfence();
          const MergeEntry me = p.merges[it.merge_idx];
          float M = lse2;
          if (h < gcnt)
            for (int c = 0; c < me.n_chunks; ++c)
              if (me.first_slot + c != it.out_slot)
                M = fmaxf(M, __ldcg(p.part_lse + prow_of(me.first_slot + c, h)));
          float W = 0.f;
          if (h < gcnt && M != kNegInfF)
            for (int c = 0; c < me.n_chunks; ++c)
              W += fast_exp2((me.first_slot + c == it.out_slot
                                  ? lse2
                                  : __ldcg(p.part_lse + prow_of(me.first_slot + c, h))) -
                             M);
          const float iw = W > 0.f ? 1.f / W : 0.f;
          wself_s[h] = (M != kNegInfF) ? fast_exp2(lse2 - M) * iw : 0.f;
          asm volatile("fence.proxy.async.global;" ::: "memory");  // partials: generic -> TMA
          uint32_t mphase = 0;
          const bool two = me.n_chunks == 2;
          const bool own_first = it.out_slot == me.first_slot;
          for (int c = 0; c < me.n_chunks; ++c) {
            const int slot = me.first_slot + c;
            if (two && slot == it.out_slot) continue;
            named_bar_sync(1, NSOFT);  // the previous chunk's passes are done with wchunk_s
            wchunk_s[h] = (h < gcnt && M != kNegInfF)
                              ? fast_exp2((slot == it.out_slot
                                               ? lse2
                                               : __ldcg(p.part_lse + prow_of(slot, h))) -
                                          M) *
                                    iw
                              : 0.f;
            const bool swap = two && !own_first;  // two chunks, the own one second
            const bool zero_b = !two && c == 0;
            for (int r0 = 0; r0 < gcnt; r0 += 64) {
              const int rows = min(64, gcnt - r0);
              named_bar_sync(1, NSOFT);  // the buffer and the weights are ready for reuse
              if (h == 0) {
                mbar_arrive_expect_tx(bar(B_MERGE), (uint32_t)rows * 1024u);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                    "%2, [%3];" ::"r"(sb + OFF_Q),
                    "l"(p.part_o + prow_of(slot, r0) * 256), "r"((uint32_t)rows * 1024u),
                    "r"(bar(B_MERGE))
                    : "memory");
              }
              if (!mbar_wait(bar(B_MERGE), mphase, abort_flag)) fail();
              mphase ^= 1u;
#pragma unroll 4
              for (int u = h; u < rows * 64; u += NSOFT) {
                const int r = u >> 6, q = u & 63, row = r0 + r;
                const uint32_t oa = stg + row * 1024 + swz(q, row);
                float4 o = *reinterpret_cast<const float4*>(base + (oa - sb));
                const float4 x =
                    *reinterpret_cast<const float4*>(base + OFF_Q + r * 1024 + q * 16);
                // o = fma(a, wa, b * wb): with two chunks, (a, b) = (chunk 1, chunk 0); with
                // more, a = this chunk and b the running sum (zero for chunk 0)
                const float wc = wchunk_s[row], ws = wself_s[row];
                const float wa = swap ? ws : wc, wb = swap ? wc : (two ? ws : 1.f);
                const float4 a = swap ? o : x;
                const float4 b = swap ? x : (zero_b ? make_float4(0.f, 0.f, 0.f, 0.f) : o);
                o.x = fmaf(a.x, wa, __fmul_rn(b.x, wb));
                o.y = fmaf(a.y, wa, __fmul_rn(b.y, wb));
                o.z = fmaf(a.z, wa, __fmul_rn(b.z, wb));
                o.w = fmaf(a.w, wa, __fmul_rn(b.w, wb));
                *reinterpret_cast<float4*>(base + (oa - sb)) = o;
              }
            }
          }
          named_bar_sync(1, NSOFT);
#pragma unroll 4
          for (int u = h; u < gcnt * 32; u += NSOFT) {
            const int r = u >> 5, q = u & 31;
            const float4 a = *reinterpret_cast<const float4*>(base + (stg - sb) + r * 1024 + swz(2 * q, r));
            const float4 c2 =
                *reinterpret_cast<const float4*>(base + (stg - sb) + r * 1024 + swz(2 * q + 1, r));
            uint4 v;
            v.x = pack2<T>(a.x, a.y);
            v.y = pack2<T>(a.z, a.w);
            v.z = pack2<T>(c2.x, c2.y);
            v.w = pack2<T>(c2.z, c2.w);
            *reinterpret_cast<uint4*>(static_cast<T*>(p.o) + ((size_t)me.req * H + g0 + r) * DC +
                                      rank * 256 + q * 8) = v;
          }
          if (h < gcnt && rank == 0 && p.lse) {
            const float l2 = W > 0.f ? M + log2f(W) : kNegInfF;
            p.lse[(size_t)me.req * H + g0 + h] = p.lse_base_e ? l2 * kLn2f : l2;
          }
        }
      }
    }
  }
  // ---- teardown: no CTA leaves while its peer may still write to it; TMEM freed last
  tc_fence_before();
  __syncwarp();
  cluster_sync();
  if (warp == 8) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace pkd
