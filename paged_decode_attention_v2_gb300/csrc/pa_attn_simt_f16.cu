// Instantiations of the attention kernel: simt math, f16 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_simt_f16(int head_size, int group) { return select_simt<__half>(head_size, group); }

}  // namespace pa
