// Instantiations of the attention kernel: simt math, bf16 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_simt_bf16(int head_size, int group) { return select_simt<__nv_bfloat16>(head_size, group); }

}  // namespace pa
