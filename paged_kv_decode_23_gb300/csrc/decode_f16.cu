// decode_f16.cu -- instantiations of the paged decode kernels for f16 q / K / V / o.
// Tiles are sized so one pipeline stage (K + V) is 32 KiB: head_dim 64 -> 128 tokens,
// 128 -> 64 tokens, 256 -> 32 tokens; three stages per CTA, two CTAs per SM.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_f16(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kTensorCore, 8>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kTensorCore, 8>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kTensorCore, 8>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 1>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 2>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 4>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kCudaCore, 8>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 1>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 2>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 4>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kCudaCore, 8>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 1>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 2>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 4>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kCudaCore, 8>(kF16, kF16));
}

}  // namespace pkd
