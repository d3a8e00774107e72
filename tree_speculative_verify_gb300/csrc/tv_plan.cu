// Verify preprocess: parent array -> ancestor masks, depths, raw window bounds and scratch-pad
// visibility ("Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient
// Inference", §4.1 verification plan, §4.3 device-side metadata).
//
// One warp per request; lane l owns nodes l and l + 32.  Each node walks up its own parent chain
// (at most D - 1 steps, since parents[v] < v strictly), so the kernel needs no inter-thread
// ordering and every loop is bounded by D.
#include "tv_common.cuh"

namespace tv {

__global__ void plan_kernel(int B, int D, int W, int tail_mode, int comp_mask,
                            const int32_t* __restrict__ parents, const int32_t* __restrict__ L,
                            uint64_t* __restrict__ anc, int32_t* __restrict__ depth,
                            int32_t* __restrict__ raw_lo, uint64_t* __restrict__ scr_vis4,
                            uint64_t* __restrict__ scr_vis128, int32_t* status) {
  pdl_launch_dependents();   // the scratch-pad kernel reads nothing this one writes
  const int warps_per_block = blockDim.x / 32;
  const int b = blockIdx.x * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (b >= B) return;
  // the request's parents in shared memory (warp-private), so the walks below cost no round trips
  __shared__ int s_par[4][kMaxD];
  int* par = s_par[(threadIdx.x / 32) & 3];
  const int Lb = L[b];
  for (int v = lane; v < D; v += 32) par[v] = parents[(int64_t)b * D + v];
  __syncwarp();

  // validate the tree: every node must name an earlier node (root: -1)
  bool ok = Lb >= 0;
  for (int v = lane; v < D; v += 32) {
    const int p = par[v];
    if (v == 0 ? (p != -1) : (p < 0 || p >= v)) ok = false;
  }
  const bool all_ok = __all_sync(0xffffffffu, ok);
  if (!all_ok) {
    if (lane == 0) record_error(status, Lb < 0 ? TV_ERR_ARG : TV_ERR_BAD_TREE);
    for (int v = lane; v < D; v += 32) {
      const int64_t i = (int64_t)b * D + v;
      anc[i] = 0;
      depth[i] = 0;
      raw_lo[i] = 0;
      if (scr_vis4) scr_vis4[i] = 0;
      if (scr_vis128) scr_vis128[i] = 0;
    }
    return;
  }

  const int m_min = m_min_of(comp_mask);
  for (int v = lane; v < D; v += 32) {
    // first pass: ancestor mask and depth
    uint64_t mask = 0;
    int dep = 0;
    int u = v;
    for (int step = 0; step < D; ++step) {
      mask |= 1ull << u;
      if (u == 0) break;
      u = par[u];
      ++dep;
    }
    // second pass: proper ancestors whose token closes a block (position L + their depth)
    uint64_t vis4 = 0, vis128 = 0;
    u = v;
    int du = dep;
    for (int step = 0; step < D && u != 0; ++step) {
      u = par[u];
      --du;
      const int pos_u = Lb + du;
      if (((pos_u + 1) & 3) == 0) vis4 |= 1ull << u;
      if (((pos_u + 1) & 127) == 0) vis128 |= 1ull << u;
    }
    const int64_t i = (int64_t)b * D + v;
    anc[i] = mask;
    depth[i] = dep;
    raw_lo[i] = raw_lo_of(Lb + dep, tail_mode, W, m_min);
    if (scr_vis4) scr_vis4[i] = (comp_mask & TV_COMP_C4) ? vis4 : 0;
    if (scr_vis128) scr_vis128[i] = (comp_mask & TV_COMP_C128) ? vis128 : 0;
  }
}

}  // namespace tv

int tv_launch_plan(const tv_shape* s, const int32_t* parents, const int32_t* L, uint64_t* anc,
                   int32_t* depth, int32_t* raw_lo, uint64_t* scr_vis4, uint64_t* scr_vis128,
                   int32_t* status, cudaStream_t stream) {
  const int warps = 4;
  const int grid = (s->B + warps - 1) / warps;
  tv::plan_kernel<<<grid, warps * 32, 0, stream>>>(s->B, s->D, s->W, s->tail_mode, s->comp_mask,
                                                   parents, L, anc, depth, raw_lo, scr_vis4,
                                                   scr_vis128, status);
  return tv_check_launch("tv_build_ancestor_mask");
}
