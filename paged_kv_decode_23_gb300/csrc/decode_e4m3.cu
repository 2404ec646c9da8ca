// decode_e4m3.cu -- instantiations of the paged decode kernels for fp8 e4m3 K/V with fp16 or
// bf16 q / o.  A stage holds 32 KiB of fp8 K + V (head_dim 128 -> 128 tokens, 256 -> 64).
// Both variants widen e4m3 to fp16 in registers (exact: every e4m3 value is an fp16 value);
// the tensor-core variant runs fp16 MMAs on operands built straight from the fp8 bytes.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_e4m3(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kTensorCore, 8>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kTensorCore, 8>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kTensorCore, 8>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kTensorCore, 8>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 1>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 2>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 4>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kCudaCore, 8>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kCudaCore, 1>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kCudaCore, 2>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kCudaCore, 4>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kCudaCore, 8>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 1>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 2>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 4>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kCudaCore, 8>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kCudaCore, 1>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kCudaCore, 2>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kCudaCore, 4>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kCudaCore, 8>(kBF16, kE4M3));
}

}  // namespace pkd
