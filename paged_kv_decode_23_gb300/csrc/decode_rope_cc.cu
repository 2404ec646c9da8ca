// decode_rope_cc.cu -- the CUDA-core decode kernels with ROPE_LLAMA (plan's pos_encoding_mode
// with use_tensor_cores off), 16-bit KV: q rotated per tile, every K row in fp32 registers.
// Same tiles and head groups as the plain CUDA-core kernels; where the rotated q buffers
// would leave room for only one CTA per SM, two pipeline stages instead of three.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_rope_cc(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 1, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 2, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 4, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 1, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 2, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 4, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 2, kCudaCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 1, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 2, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 2, kCudaCore, 4, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 2, kCudaCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 1, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 2, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 4, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 8, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 1, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 2, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 4, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 2, kCudaCore, 8, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 1, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 2, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 2, kCudaCore, 4, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 2, kCudaCore, 8, true>(kBF16, kBF16));
}

}  // namespace pkd
