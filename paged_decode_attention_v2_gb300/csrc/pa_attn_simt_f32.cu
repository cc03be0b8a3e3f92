// Instantiations of the attention kernel: simt math, f32 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_simt_f32(int head_size, int group) { return select_simt<float>(head_size, group); }

}  // namespace pa
