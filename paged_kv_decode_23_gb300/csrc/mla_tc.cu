// mla_tc.cu -- instantiations of the tcgen05 MLA paged decode kernel (bf16 and fp16).
#include "mla_tc_kernels.cuh"

namespace pkd {

void register_mla_tc(std::vector<MlaKernel>& out) {
  MlaKernel k;
  k.variant = kMlaTcgen05;
  k.threads = mlatc::THREADS;
  k.smem_bytes = mlatc::SMEM_BYTES;
  k.heads_per_cta = mlatc::HT;
  k.tile_tokens = mlatc::TS;
  k.ctas_per_head_tile = 2;
  k.dtype = kBF16;
  k.fn = reinterpret_cast<const void*>(&mla_tc_kernel<__nv_bfloat16>);
  out.push_back(k);
  k.dtype = kF16;
  k.fn = reinterpret_cast<const void*>(&mla_tc_kernel<__half>);
  out.push_back(k);
}

}  // namespace pkd
