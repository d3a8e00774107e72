// Shared device helpers of libtreeverify (status words, element loads/stores, launch checks).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "treeverify.h"

namespace tv {

constexpr int kMaxD = 64;          // tree nodes per request (one 64-bit ancestor mask)
constexpr int kMaxHeadDim = 512;   // largest head dimension

// First-error-wins device status: the word only ever moves from 0 to a negative code.
__device__ __forceinline__ void record_error(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Lowest raw position visible from a query at position p.
__device__ __forceinline__ int raw_lo_of(int p, int tail_mode, int W, int m_min) {
  if (tail_mode == TV_TAIL_WINDOW) return p - W > 0 ? p - W : 0;
  return m_min * (p / m_min);
}

__host__ __device__ __forceinline__ int m_min_of(int comp_mask) {
  return (comp_mask & TV_COMP_C4) ? 4 : 128;
}

}  // namespace tv

// Host-side helpers shared by the entry points (defined in tv_api.cu).
int tv_set_error(int code, const char* fmt, ...);
int tv_check_launch(const char* what);
