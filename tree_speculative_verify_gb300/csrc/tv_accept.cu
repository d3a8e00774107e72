// Accepted-path selection: the greedy acceptance walk ("Adapting Tree-Structured Speculative
// Decoding to DeepSeek-V4 for Efficient Inference", §3.2 and §4.1: after verification one
// specific root-to-node path is selected and only its results are kept).
//
// One warp per request.  Lane l holds nodes l and l + 32; each step of the walk is two ballots
// over "is a child of the current node and drafted the current node's target token", and the
// lowest set bit is the next node.  At most D - 1 steps.
#include "tv_common.cuh"

namespace tv {

__global__ void accept_kernel(int B, int D, const int32_t* __restrict__ parents,
                              const int32_t* __restrict__ draft,
                              const int32_t* __restrict__ target, int32_t* __restrict__ accept_len,
                              int32_t* __restrict__ path, int32_t* __restrict__ bonus,
                              int32_t* status) {
  pdl_launch_dependents();   // the refresh may launch now; it waits for this kernel's results
  const int warps_per_block = blockDim.x / 32;
  const int b = blockIdx.x * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (b >= B) {
    pdl_wait();
    return;
  }
  const int64_t base = (int64_t)b * D;
  const int v0 = lane, v1 = lane + 32;
  const int p0 = v0 < D ? parents[base + v0] : -2;
  const int p1 = v1 < D ? parents[base + v1] : -2;
  const int d0 = v0 < D ? draft[base + v0] : 0;
  const int d1 = v1 < D ? draft[base + v1] : 0;
  const int t0 = v0 < D ? target[base + v0] : 0;   // the walk reads targets from registers
  const int t1 = v1 < D ? target[base + v1] : 0;
  bool ok = true;
  if (v0 < D) ok &= (v0 == 0) ? (p0 == -1) : (p0 >= 0 && p0 < v0);
  if (v1 < D) ok &= (p1 >= 0 && p1 < v1);
  // launched as a programmatic dependent of the attention: the inputs above are not written by
  // it, and the walk runs in registers; the stores below wait for the kernel before this one to
  // complete
  if (!__all_sync(0xffffffffu, ok)) {
    pdl_wait();
    if (lane == 0) {
      record_error(status, TV_ERR_BAD_TREE);
      accept_len[b] = 1;
      bonus[b] = -1;
    }
    if (v0 < D) path[base + v0] = v0 == 0 ? 0 : -1;
    if (v1 < D) path[base + v1] = -1;
    return;
  }
  int cur = 0, n = 1;
  int my0 = v0 == 0 ? 0 : -1;  // path entry held by this lane (index lane / lane + 32)
  int my1 = -1;
  for (int step = 1; step < D; ++step) {
    const int tgt = __shfl_sync(0xffffffffu, cur < 32 ? t0 : t1, cur & 31);
    const unsigned b0 = __ballot_sync(0xffffffffu, v0 > 0 && v0 < D && p0 == cur && d0 == tgt);
    const unsigned b1 = __ballot_sync(0xffffffffu, v1 < D && p1 == cur && d1 == tgt);
    if (b0 == 0u && b1 == 0u) break;
    const int nxt = b0 ? (__ffs(b0) - 1) : (32 + __ffs(b1) - 1);
    if (n == lane) my0 = nxt;
    if (n == lane + 32) my1 = nxt;
    ++n;
    cur = nxt;
  }
  const int bonus_tok = __shfl_sync(0xffffffffu, cur < 32 ? t0 : t1, cur & 31);
  pdl_wait();
  if (v0 < D) path[base + v0] = my0;
  if (v1 < D) path[base + v1] = my1;
  if (lane == 0) {
    accept_len[b] = n;
    bonus[b] = bonus_tok;
  }
}

}  // namespace tv

int tv_launch_accept(const tv_shape* s, const int32_t* parents, const int32_t* draft,
                     const int32_t* target, int32_t* accept_len, int32_t* path, int32_t* bonus,
                     int32_t* status, cudaStream_t stream) {
  const int warps = 4;
  const int grid = (s->B + warps - 1) / warps;
  // a programmatic dependent: its launch and its loads overlap the kernel before it
  const cudaError_t e = tv::launch_pdl(tv::accept_kernel, dim3(grid), dim3(warps * 32), 0, stream,
                                       s->B, s->D, parents, draft, target, accept_len, path,
                                       bonus, status);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return tv_set_error(TV_ERR_CUDA, "tv_accept_walk: launch failed: %s", cudaGetErrorString(e));
  }
  return tv_check_launch("tv_accept_walk");
}
