// Branch-aware causal tree-verify attention on CUDA cores (fp32 arithmetic), split-KV.
//
// "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference",
// §3.1: each candidate sees the accepted context and its own ancestors only; §3.2 / §4.2: the
// blocks a branch closes are seen through that branch's scratch-pad entries only.
//
// This kernel serves every supported shape and both storage dtypes; it is the production path
// for fp32 caches and for shapes the tcgen05 kernel does not take.  Work decomposition:
//   CTA = (chunk of the request's entry list, group of 8 query rows, request); warp = one row
//   (node v = row / H, head h = row % H); the CTA stages 8 K/V entries at a time in shared memory
//   (converted to fp32) and every warp runs an online softmax over them.  Each (row, chunk) pair
//   leaves (m, l, o[d]) in the workspace; merge_kernel combines the chunks into O and LSE.
// Logits are kept in base-2 units (scaled by scale * log2 e) so that exp2f is the only
// transcendental on the hot loop.
#include <math.h>

#include "tv_attn_common.cuh"

namespace tv {

constexpr int kSimtRows = 8;      // rows (warps) per CTA
constexpr int kSimtTile = 8;      // entries staged per step
constexpr int kSimtThreads = kSimtRows * 32;

template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
simt_attn_kernel(AttnParams<T> p) {
  extern __shared__ float smem[];
  float* sK = smem;                                // [kSimtTile][d]
  float* sV = sK + kSimtTile * p.d;                // [kSimtTile][d]
  __shared__ EntryRef ent[kSimtTile];

  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int DH = p.D * p.H;
  const int row = blockIdx.y * kSimtRows + warp;
  const bool row_ok = row < DH;
  const int v = row_ok ? row / p.H : 0;
  const int d = p.d;
  const int per_lane = d / 32 + (lane < d % 32 ? 1 : 0);

  const EntryLayout lay = entry_layout(p, b);
  const int c = blockIdx.x;
  const int e_begin = c * p.chunk;
  int e_end = e_begin + p.chunk;
  if (e_end > lay.total) e_end = lay.total;

  NodeVis nv = node_vis(p, b, v);

  float q[kMaxHeadDim / 32];
  float o[kMaxHeadDim / 32];
#pragma unroll
  for (int k = 0; k < kMaxHeadDim / 32; ++k) {
    q[k] = 0.f;
    o[k] = 0.f;
  }
  if (row_ok) {
    const T* qrow = p.Q + ((int64_t)b * DH + row) * d;
#pragma unroll
    for (int k = 0; k < kMaxHeadDim / 32; ++k)
      if (k < per_lane) q[k] = load_f(qrow + lane + 32 * k) * p.scale_log2;
  }
  float m_run = -INFINITY, l_run = 0.f;

  for (int e0 = e_begin; e0 < e_end; e0 += kSimtTile) {
    const int ne = (e_end - e0) < kSimtTile ? (e_end - e0) : kSimtTile;
    __syncthreads();
    if (threadIdx.x < kSimtTile) {
      EntryRef r;
      if ((int)threadIdx.x < ne) r = resolve_entry(p, lay, b, e0 + threadIdx.x);
      else r.kind = kEntryNone;
      ent[threadIdx.x] = r;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < ne * d; idx += blockDim.x) {
      const int t = idx / d, i = idx - t * d;
      const EntryRef r = ent[t];
      float kx = 0.f, vx = 0.f;
      if (r.kind != kEntryNone) {
        kx = load_f(static_cast<const T*>(r.k) + i);
        vx = load_f(static_cast<const T*>(r.v) + i);
      }
      sK[t * d + i] = kx;
      sV[t * d + i] = vx;
    }
    __syncthreads();
    if (!row_ok) continue;
    float s[kSimtTile];
    float tile_max = -INFINITY;
#pragma unroll
    for (int t = 0; t < kSimtTile; ++t) {
      float acc = 0.f;
      if (t < ne) {
#pragma unroll
        for (int k = 0; k < kMaxHeadDim / 32; ++k)
          if (k < per_lane) acc = fmaf(q[k], sK[t * d + lane + 32 * k], acc);
      }
      acc = warp_sum(acc);
      const bool vis = t < ne && entry_visible(ent[t], nv);
      s[t] = vis ? acc : -INFINITY;
      tile_max = fmaxf(tile_max, s[t]);
    }
    if (tile_max == -INFINITY) continue;
    const float m_new = fmaxf(m_run, tile_max);
    const float alpha = exp2f(m_run - m_new);   // 0 when m_run = -inf
    l_run *= alpha;
#pragma unroll
    for (int k = 0; k < kMaxHeadDim / 32; ++k) o[k] *= alpha;
#pragma unroll
    for (int t = 0; t < kSimtTile; ++t) {
      if (s[t] == -INFINITY) continue;
      const float pt = exp2f(s[t] - m_new);
      l_run += pt;
#pragma unroll
      for (int k = 0; k < kMaxHeadDim / 32; ++k)
        if (k < per_lane) o[k] = fmaf(pt, sV[t * d + lane + 32 * k], o[k]);
    }
    m_run = m_new;
  }
  if (!row_ok) return;
  float* part = p.part + (((int64_t)b * DH + row) * p.n_chunks + c) * (d + 4);
#pragma unroll
  for (int k = 0; k < kMaxHeadDim / 32; ++k)
    if (k < per_lane) part[lane + 32 * k] = o[k];
  if (lane == 0) {
    part[d] = m_run;
    part[d + 1] = l_run;
  }
}

}  // namespace tv

template <typename T>
static int launch_simt_t(const tv::AttnParams<T>& p, cudaStream_t stream) {
  const int DH = p.D * p.H;
  const dim3 grid(p.n_chunks, (DH + tv::kSimtRows - 1) / tv::kSimtRows, p.B);
  const size_t smem = 2 * tv::kSimtTile * p.d * sizeof(float);
  tv::simt_attn_kernel<T><<<grid, tv::kSimtThreads, smem, stream>>>(p);
  if (int rc = tv_check_launch("tv_tree_verify_attn (SIMT partials)")) return rc;
  return tv_launch_merge<T>(p.B, DH, p.d, p.n_chunks, p.part, p.O, p.lse, stream);
}

int tv_launch_attn_simt_bf16(const tv::AttnParams<__nv_bfloat16>& p, cudaStream_t stream) {
  return launch_simt_t(p, stream);
}
int tv_launch_attn_simt_f32(const tv::AttnParams<float>& p, cudaStream_t stream) {
  return launch_simt_t(p, stream);
}
