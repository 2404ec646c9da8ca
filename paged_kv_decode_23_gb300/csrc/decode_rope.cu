// decode_rope.cu -- the tensor-core decode kernels with ROPE_LLAMA (plan's pos_encoding_mode):
// q and every K row are rotated in registers before the QK MMAs (in fp16), for each q / KV
// dtype pair and head_dim the plain kernels are built for.  Same tiles as the plain kernels.
#include "decode_kernels.cuh"

namespace pkd {

void register_decode_rope(std::vector<DecodeKernel>& out) {
  out.push_back(make_decode_kernel<__half, false, 64, 128, 3, kTensorCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 128, 64, 3, kTensorCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__half, false, 256, 32, 3, kTensorCore, 8, true>(kF16, kF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 64, 128, 3, kTensorCore, 8, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 128, 64, 3, kTensorCore, 8, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__nv_bfloat16, false, 256, 32, 3, kTensorCore, 8, true>(kBF16, kBF16));
  out.push_back(make_decode_kernel<__half, true, 128, 128, 3, kTensorCore, 8, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__half, true, 256, 64, 3, kTensorCore, 8, true>(kF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 128, 128, 3, kTensorCore, 8, true>(kBF16, kE4M3));
  out.push_back(make_decode_kernel<__nv_bfloat16, true, 256, 64, 3, kTensorCore, 8, true>(kBF16, kE4M3));
}

}  // namespace pkd
