// merge_kernel.cuh -- merge_states: combine split-KV partials of a request by their
// log-sum-exp.
//
// FlashInfer attention API page, BatchDecodeWithPagedKVCacheWrapper.plan(fixed_split_size):
// split-KV partial results are reduced by a merge_states step, deterministically when the
// split size is fixed.  For partials (o_c, lse_c) over disjoint key sets:
//   M = max_c lse_c, w_c = 2^(lse_c - M), o = sum_c w_c o_c / sum_c w_c,
//   lse = M + log2(sum_c w_c)   (kept base 2 in the workspace, written as natural log).
// One warp per (request, qo head); chunks are summed in chunk order, so the result does not
// depend on timing or on the rest of the batch.
#pragma once

#include "pkd_device.cuh"
#include "pkd_internal.h"

namespace pkd {

template <typename TO, int D>
__global__ void __launch_bounds__(128) merge_states_kernel(const MergeParams p) {
  using namespace dev;
  constexpr int EPL = D / 32;
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int entry = wid / p.num_qo_heads;
  const int qo = wid - entry * p.num_qo_heads;
  if (entry >= p.num_merges) return;
  if ((*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) != 0u) return;
  const MergeEntry me = p.merges[entry];
  const float neg_inf = -__int_as_float(0x7f800000);
  float M = neg_inf;
  for (int c = 0; c < me.n_chunks; ++c)
    M = fmaxf(M, p.part_lse[(size_t)(me.first_slot + c) * p.num_qo_heads + qo]);
  float o[EPL];
#pragma unroll
  for (int k = 0; k < EPL; ++k) o[k] = 0.f;
  float L = 0.f;
  if (M != neg_inf) {
    for (int c = 0; c < me.n_chunks; ++c) {
      const size_t row = (size_t)(me.first_slot + c) * p.num_qo_heads + qo;
      const float f = fast_exp2(p.part_lse[row] - M);
      L += f;
      const float* src = p.part_o + row * D + lane * EPL;
#pragma unroll
      for (int k = 0; k < EPL; k += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + k);
        o[k] = fmaf(f, v.x, o[k]);
        o[k + 1] = fmaf(f, v.y, o[k + 1]);
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  TO* dst = reinterpret_cast<TO*>(p.o) + ((size_t)me.req * p.num_qo_heads + qo) * D + lane * EPL;
#pragma unroll
  for (int k = 0; k < EPL; k += 2)
    *reinterpret_cast<uint32_t*>(dst + k) = pack2<TO>(o[k] * inv, o[k + 1] * inv);
  if (lane == 0 && p.lse)
    p.lse[(size_t)me.req * p.num_qo_heads + qo] =
        L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : neg_inf;
}

}  // namespace pkd
