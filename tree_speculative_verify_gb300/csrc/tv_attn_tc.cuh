// tcgen05 tensor-core tree-verify attention (bf16, d = 512): host-side interface.
#pragma once

#include "tv_attn_common.cuh"

// True when the tensor-core kernel takes this shape (bf16, d = 512, D <= 8, B <= 12288; a C4
// selection list is gathered into the workspace first).
bool tv_tc_shape_ok(const tv_shape* s);
// True when the tensor-core kernel is compiled in and the current device can run it.
bool tv_tc_available();
// Workspace bytes the tensor-core kernel needs for this shape.
size_t tv_tc_workspace_size(const tv_shape* s);
// Enqueue the tensor-core kernel (and its merge) on `stream`.
int tv_launch_attn_tc(const tv_shape* s, const tv::AttnParams<__nv_bfloat16>& p, void* workspace,
                      cudaStream_t stream);
