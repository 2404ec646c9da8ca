// merge.cu -- registry of the merge_states kernels (the kernel is in merge_kernel.cuh).
#include "merge_kernel.cuh"

namespace pkd {

template <typename TO, int D>
static MergeKernel make_merge(int o_dtype) {
  MergeKernel k;
  k.o_dtype = o_dtype;
  k.head_dim = D;
  k.fn = reinterpret_cast<const void*>(&merge_states_kernel<TO, D>);
  k.threads = 128;
  k.heads_per_block = 4;
  return k;
}

void register_merge(std::vector<MergeKernel>& out) {
  out.push_back(make_merge<__half, 64>(kF16));
  out.push_back(make_merge<__half, 128>(kF16));
  out.push_back(make_merge<__half, 256>(kF16));
  out.push_back(make_merge<__nv_bfloat16, 64>(kBF16));
  out.push_back(make_merge<__nv_bfloat16, 128>(kBF16));
  out.push_back(make_merge<__nv_bfloat16, 256>(kBF16));
}

}  // namespace pkd
