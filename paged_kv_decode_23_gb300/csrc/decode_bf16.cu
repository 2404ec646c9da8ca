// decode_bf16.cu -- instantiations of the paged decode kernels for bf16 q / K / V / o.
// Tiles are sized so one pipeline stage (K + V) is 32 KiB: head_dim 64 -> 128 tokens,
// 128 -> 64 tokens, 256 -> 32 tokens; three stages per CTA, two CTAs per SM.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_bf16(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kTensorCore, 8>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kTensorCore, 8>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kTensorCore, 8>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 1>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 2>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 4>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kCudaCore, 8>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 1>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 2>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 4>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kCudaCore, 8>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 1>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 2>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 4>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kCudaCore, 8>(kBF16, kBF16));
}

}  // namespace pkd
