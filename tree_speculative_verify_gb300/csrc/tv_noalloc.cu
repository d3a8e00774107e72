// tv_tree_verify_attn_noalloc: the tree-verify attention for callers that cannot allocate device
// memory.
//
// Some callers of this library have no way to obtain a device workspace: a serving engine that
// reserves all free device memory for its own KV page pool at start-up (a later cudaMalloc fails
// or fragments that pool), a decode loop that must not pay cudaMalloc's implicit device
// synchronisation on its critical path, or a plug-in host that hands a library streams and
// tensors but no allocator.  This entry point takes the same inputs and outputs as
// tv_tree_verify_attn but keeps the split-KV partial results in a scratch array that is part of
// the library image itself, so it never allocates.
//
// The scratch array is a file-scope __device__ array of kNoAllocScratchBytes (32 MiB): every GPU
// that loads the library's device code holds it until the process exits.  With CUDA's lazy module
// loading (the default) that happens at the first call on each device that resolves the array --
// tv_noalloc_prepare or the first tv_tree_verify_attn_noalloc -- so a caller that hands all free
// memory to its own pool makes one of those calls first.  Calls whose shape needs more scratch
// than that (see tv_workspace_size) are rejected with TV_ERR_WORKSPACE.  All calls share the
// array, so calls that overlap on the GPU (different streams, or different threads without
// ordering) race on it; the kernels write every partial result they later read, so nothing in it
// needs to start at zero and the contents left by the previous call are never used.  The array's
// address is looked up on every call, in the caller's current context, so it stays right across a
// device reset or a change of context.
#include "tv_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context (host code cannot use the array's
// name as a device address: it is a host-side stand-in for the symbol).
int scratch_address(const char* fn, void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return tv_set_error(TV_ERR_CUDA, "%s: the built-in scratch is not available: %s", fn,
                        cudaGetErrorString(e));
  }
  *out = p;
  return TV_OK;
}

}  // namespace

extern "C" int tv_noalloc_prepare(void) {
  void* p = nullptr;
  return scratch_address("tv_noalloc_prepare", &p);
}

extern "C" int tv_tree_verify_attn_noalloc(
    const tv_shape* s, const void* Q, const void* c4K, const void* c4V, const int32_t* sel,
    const void* c128K, const void* c128V, const void* rawK, const void* rawV, const int32_t* L,
    const void* treeK, const void* treeV, const uint64_t* anc, const int32_t* raw_lo,
    const uint64_t* scr_vis4, const uint64_t* scr_vis128, const void* scrK4, const void* scrV4,
    const void* scrK128, const void* scrV128, float scale, void* O, float* lse, int32_t* status,
    tv_stream_t stream) {
  const char* fn = "tv_tree_verify_attn_noalloc";
  if (s == nullptr) return tv_set_error(TV_ERR_ARG, "%s: shape is null", fn);
  const size_t need = tv_workspace_size(s);
  if (need > kNoAllocScratchBytes)
    return tv_set_error(TV_ERR_WORKSPACE,
                        "%s: this shape needs %zu bytes of scratch; the built-in scratch holds "
                        "%zu (use tv_tree_verify_attn with a workspace)",
                        fn, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if (int rc = scratch_address(fn, &scratch)) return rc;
  return tv_attn_entry(fn, s, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK, treeV, anc,
                       raw_lo, scr_vis4, scr_vis128, scrK4, scrV4, scrK128, scrV128, scale, O,
                       lse, scratch, kNoAllocScratchBytes, status, stream);
}
