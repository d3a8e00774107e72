// Shared device helpers of libtreeverify (status words, element loads/stores, launch checks).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdio.h>

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
// Four consecutive values in one store (p aligned to 4 elements).
__device__ __forceinline__ void store_f4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store_f4(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = w;
}

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

// Range checks of the bounds-checked build (compiled with -DTV_CHECK_BOUNDS, see build.py): a global
// index computed on the device must satisfy lo <= i < hi before the access it addresses.  A
// violation records TV_ERR_BOUNDS in the status word, prints the site number and the index (from
// the thread that recorded it), and the caller skips the access.  In the normal build the check
// is the constant true and costs nothing.  Sites:
//   1 attention producer, first row of a prefix tile inside its map
//   2 attention producer, the request's tree / scratch rows
//   3 attention epilogue, O rows                  4 attention epilogue, split-KV partial rows
//   5 a persistent row (raw, C4, C128) inside its request's capacity (layer_row, contiguous
//     layout: prefill, scratch pad, refresh, selection gather); the paged layout checks its page
//     ids against the pool and reports TV_ERR_ARG in every build
#ifdef TV_CHECK_BOUNDS
__device__ __forceinline__ bool tv_in_range(int64_t i, int64_t lo, int64_t hi, int32_t* status,
                                            int site) {
  if (i >= lo && i < hi) return true;
  if (status != nullptr && atomicCAS(status, 0, TV_ERR_BOUNDS) == 0)
    printf("treeverify bounds check: site %d index %lld not in [%lld, %lld) (block %d, thread %d)\n",
           site, (long long)i, (long long)lo, (long long)hi, (int)blockIdx.x, (int)threadIdx.x);
  return false;
}
#else
__device__ __forceinline__ constexpr bool tv_in_range(int64_t, int64_t, int64_t, int32_t*, int) {
  return true;
}
#endif

// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the kernel
// before it in the stream still runs, once every CTA of that kernel has called
// pdl_launch_dependents (or finished).  It must call pdl_wait before it reads anything that
// kernel writes and before it writes anything that kernel reads, and before it exits, so that
// its own completion still implies the completion of everything before it in the stream.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the kernel this one depends on programmatically has completed and its memory
// operations are visible (returns at once for a kernel launched without such a dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Lowest raw position visible from a query at position p.
__device__ __forceinline__ int raw_lo_of(int p, int tail_mode, int W, int m_min) {
  if (tail_mode == TV_TAIL_WINDOW) return p - W > 0 ? p - W : 0;
  return m_min * (p / m_min);
}

__host__ __device__ __forceinline__ int m_min_of(int comp_mask) {
  return (comp_mask & TV_COMP_C4) ? 4 : 128;
}

// Persistent-row addressing, contiguous or paged (see tv_shape).  A layer whose rows each cover
// `tokens_per_row` positions (raw 1, C4 4, C128 128) has page_tokens / tokens_per_row rows per page.
struct Paging {
  int32_t page_tokens;   // 0: contiguous [B][cap] rows
  int32_t max_pages;
  int32_t n_pool_pages;
  const int32_t* table;  // [B][max_pages]
};

inline Paging paging_of(const tv_shape* s) {
  Paging p;
  p.page_tokens = s->page_tokens;
  p.max_pages = s->max_pages;
  p.n_pool_pages = s->n_pool_pages;
  p.table = s->page_table;
  return p;
}

// Row of row `idx` of request b in a layer with `cap` rows per request.  A page id outside the
// pool records TV_ERR_ARG and addresses page 0 (so no access leaves the pool).  With pages, an
// index past the request's capacity (the padding rows of a partial tile, never used unmasked) is
// clamped to its last row, so the page-table read stays inside the request's row of the table.
__device__ __forceinline__ int64_t layer_row(const Paging& pg, int b, int64_t idx, int64_t cap,
                                             int tokens_per_row, int32_t* status) {
  if (pg.page_tokens == 0)
    return (int64_t)b * cap + (tv_in_range(idx, 0, cap, status, 5) ? idx : 0);
  if (idx >= cap) idx = cap - 1;
  if (idx < 0) idx = 0;
  const int64_t rpp = pg.page_tokens / tokens_per_row;
  int32_t page = pg.table[(int64_t)b * pg.max_pages + idx / rpp];
  if (page < 0 || page >= pg.n_pool_pages) {
    record_error(status, TV_ERR_ARG);
    page = 0;
  }
  return (int64_t)page * rpp + idx % rpp;
}

}  // namespace tv

// Host-side helpers shared by the entry points (defined in tv_api.cu).
int tv_set_error(int code, const char* fmt, ...);
// tv_tree_verify_attn's body; fn names the public entry point in error messages.
int tv_attn_entry(const char* fn, const tv_shape* s, const void* Q, const void* c4K,
                  const void* c4V, const int32_t* sel, const void* c128K, const void* c128V,
                  const void* rawK, const void* rawV, const int32_t* L, const void* treeK,
                  const void* treeV, const uint64_t* anc, const int32_t* raw_lo,
                  const uint64_t* scr_vis4, const uint64_t* scr_vis128, const void* scrK4,
                  const void* scrV4, const void* scrK128, const void* scrV128, float scale,
                  void* O, float* lse, void* workspace, size_t ws_bytes, int32_t* status,
                  tv_stream_t stream);
int tv_check_launch(const char* what);
