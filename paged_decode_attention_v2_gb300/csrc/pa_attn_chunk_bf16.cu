// Instantiations of the attention kernel for query chunks: tensor math, bf16 elements.
#include "pa_attn.cuh"

namespace pa {

AttnKernelInfo attn_kernel_chunk_bf16(int head_size, int group, int max_rows) {
  return select_chunk<__nv_bfloat16>(head_size, group, max_rows);
}

}  // namespace pa
