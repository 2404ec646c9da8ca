// mla.cu -- instantiations of the MLA paged decode kernel (bf16 and fp16, latent 512 + rope 64).
#include "mla_kernels.cuh"

namespace pkd {

void register_mla(std::vector<MlaKernel>& out) {
  MlaKernel k;
  k.variant = kMlaMmaSync;
  k.ctas_per_head_tile = 1;
  k.threads = mla::THREADS;
  k.smem_bytes = mla::SMEM_BYTES;
  k.heads_per_cta = mla::HT;
  k.tile_tokens = mla::TS;
  k.dtype = kBF16;
  k.fn = reinterpret_cast<const void*>(&mla_decode_kernel<__nv_bfloat16>);
  out.push_back(k);
  k.dtype = kF16;
  k.fn = reinterpret_cast<const void*>(&mla_decode_kernel<__half>);
  out.push_back(k);
}

}  // namespace pkd
