// Instantiations of the attention kernel: tensor math, bf16 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_tensor_bf16(int head_size, int group) { return select_tensor<__nv_bfloat16>(head_size, group); }

}  // namespace pa
