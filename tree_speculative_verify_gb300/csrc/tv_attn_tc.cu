// tcgen05 tensor-core tree-verify attention: placeholder until the kernel lands.
#include "tv_attn_tc.cuh"

bool tv_tc_available() { return false; }
size_t tv_tc_workspace_size(const tv_shape*) { return 0; }
int tv_launch_attn_tc(const tv_shape*, const tv::AttnParams<__nv_bfloat16>&, void*, cudaStream_t) {
  return tv_set_error(TV_ERR_DTYPE, "tv_tree_verify_attn: tcgen05 kernel not built");
}
