// Instantiations of the attention kernel: tensor math, f16 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_tensor_f16(int head_size, int group) { return select_tensor<__half>(head_size, group); }

}  // namespace pa
