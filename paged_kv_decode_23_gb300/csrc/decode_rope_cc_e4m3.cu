// decode_rope_cc_e4m3.cu -- the CUDA-core decode kernels with ROPE_LLAMA for e4m3 KV (f16 or
// bf16 q): each K row is widened to fp32 and rotated in registers.  Same tiles and head
// groups as the plain CUDA-core e4m3 kernels; where the rotated q buffers would leave room
// for only one CTA per SM, two pipeline stages instead of three.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_rope_cc_e4m3(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 1, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 2, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 4, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 8, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kCudaCore, 1, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 2, kCudaCore, 2, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 2, kCudaCore, 4, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 2, kCudaCore, 8, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 1, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 2, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 4, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 8, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kCudaCore, 1, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 2, kCudaCore, 2, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 2, kCudaCore, 4, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 2, kCudaCore, 8, true>(kBF16, kE4M3));
}

}  // namespace pkd
