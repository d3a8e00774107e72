// Entry list, visibility rule and split-KV merge shared by the attention kernels.
//
// The entries a request's tree rows may attend to are laid out in one index space:
//   [C4 (all L/4, or the n_sel selected) | C128 (L/128) | raw tail t0 .. L-1 | tree nodes 0..D-1
//    | C4 scratch rows 0..D-1 | C128 scratch rows 0..D-1]
// The first two segments are visible to every row; the tail segments are filtered per node by
// the plan (raw_lo, ancestor mask, scratch visibility masks).  This is the branch-aware causal
// visibility of "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient
// Inference" §3.1 with the scratch-pad isolation of §3.2 / §4.2.
#pragma once

#include <math.h>

#include "tv_common.cuh"

namespace tv {

template <typename T>
struct AttnParams {
  int B, D, H, d, W, tail_mode, comp_mask, n_sel;
  int64_t raw_cap, c4_cap, c128_cap;
  Paging pg;
  const T* Q;
  const T* c4K;
  const T* c4V;
  const T* c128K;
  const T* c128V;
  const T* rawK;
  const T* rawV;
  const T* treeK;
  const T* treeV;
  const T* scrK4;
  const T* scrV4;
  const T* scrK128;
  const T* scrV128;
  const int32_t* sel;
  const int32_t* L;
  const int32_t* raw_lo;
  const uint64_t* anc;
  const uint64_t* scr_vis4;
  const uint64_t* scr_vis128;
  float scale_log2;   // logit scale times log2(e)
  int n_chunks;       // split-KV chunks per request
  int chunk;          // entries per chunk
  float* part;        // [B][D*H][n_chunks][d + 4] partial (o[d], m, l, 2 pad)
  T* O;
  float* lse;
  int32_t* status;
};

enum EntryKind { kEntryNone = 0, kEntryShared, kEntryRaw, kEntryTree, kEntryScr4, kEntryScr128 };

struct EntryLayout {
  int L;
  int n4, n128, t0, nraw, nscr4, nscr128;
  int base128, baseraw, basetree, basescr4, basescr128, total;
};

template <typename T>
__device__ __forceinline__ EntryLayout entry_layout(const AttnParams<T>& p, int b) {
  EntryLayout e;
  const int L = p.L[b];
  const bool c4 = p.comp_mask & TV_COMP_C4, c128 = p.comp_mask & TV_COMP_C128;
  const bool cap_ok = L >= 0 && L <= p.raw_cap && (!c4 || L / 4 <= p.c4_cap) &&
                      (!c128 || L / 128 <= p.c128_cap);
  if (!cap_ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(p.status, TV_ERR_CAPACITY);
    e.L = 0;
    e.n4 = e.n128 = e.t0 = e.nraw = e.nscr4 = e.nscr128 = 0;
    e.base128 = e.baseraw = e.basetree = e.basescr4 = e.basescr128 = e.total = 0;
    return e;
  }
  e.L = L;
  e.n4 = c4 ? (p.n_sel > 0 ? p.n_sel : L / 4) : 0;
  e.n128 = c128 ? L / 128 : 0;
  const int tail = p.tail_mode == TV_TAIL_WINDOW ? p.W : m_min_of(p.comp_mask) - 1;
  e.t0 = L - tail > 0 ? L - tail : 0;
  e.nraw = L - e.t0;
  e.nscr4 = c4 ? p.D : 0;
  e.nscr128 = c128 ? p.D : 0;
  e.base128 = e.n4;
  e.baseraw = e.base128 + e.n128;
  e.basetree = e.baseraw + e.nraw;
  e.basescr4 = e.basetree + p.D;
  e.basescr128 = e.basescr4 + e.nscr4;
  e.total = e.basescr128 + e.nscr128;
  return e;
}

struct EntryRef {
  const void* k;
  const void* v;
  int kind;
  int aux;   // raw position, or tree node id
};

template <typename T>
__device__ __forceinline__ EntryRef resolve_entry(const AttnParams<T>& p, const EntryLayout& lay,
                                                  int b, int e) {
  EntryRef r;
  r.kind = kEntryNone;
  r.aux = 0;
  r.k = r.v = nullptr;
  const int d = p.d;
  if (e < lay.base128) {
    int j = e;
    if (p.n_sel > 0) {
      j = p.sel[(int64_t)b * p.n_sel + e];
      if (j < 0 || j >= lay.L / 4) {
        record_error(p.status, TV_ERR_SELECTION);
        return r;
      }
    }
    const int64_t off = layer_row(p.pg, b, j, p.c4_cap, 4, p.status) * d;
    r.k = p.c4K + off;
    r.v = p.c4V + off;
    r.kind = kEntryShared;
  } else if (e < lay.baseraw) {
    const int64_t off = layer_row(p.pg, b, e - lay.base128, p.c128_cap, 128, p.status) * d;
    r.k = p.c128K + off;
    r.v = p.c128V + off;
    r.kind = kEntryShared;
  } else if (e < lay.basetree) {
    const int pos = lay.t0 + (e - lay.baseraw);
    const int64_t off = layer_row(p.pg, b, pos, p.raw_cap, 1, p.status) * d;
    r.k = p.rawK + off;
    r.v = p.rawV + off;
    r.kind = kEntryRaw;
    r.aux = pos;
  } else if (e < lay.basescr4) {
    const int u = e - lay.basetree;
    const int64_t off = ((int64_t)b * p.D + u) * d;
    r.k = p.treeK + off;
    r.v = p.treeV + off;
    r.kind = kEntryTree;
    r.aux = u;
  } else if (e < lay.basescr128) {
    const int u = e - lay.basescr4;
    const int64_t off = ((int64_t)b * p.D + u) * d;
    r.k = p.scrK4 + off;
    r.v = p.scrV4 + off;
    r.kind = kEntryScr4;
    r.aux = u;
  } else if (e < lay.total) {
    const int u = e - lay.basescr128;
    const int64_t off = ((int64_t)b * p.D + u) * d;
    r.k = p.scrK128 + off;
    r.v = p.scrV128 + off;
    r.kind = kEntryScr128;
    r.aux = u;
  }
  return r;
}

// Per-node visibility data taken from the plan.
struct NodeVis {
  uint64_t anc, vis4, vis128;
  int raw_lo, L;
};

template <typename T>
__device__ __forceinline__ NodeVis node_vis(const AttnParams<T>& p, int b, int v) {
  NodeVis n;
  const int64_t i = (int64_t)b * p.D + v;
  n.anc = p.anc[i];
  n.vis4 = (p.comp_mask & TV_COMP_C4) ? p.scr_vis4[i] : 0;
  n.vis128 = (p.comp_mask & TV_COMP_C128) ? p.scr_vis128[i] : 0;
  n.raw_lo = p.raw_lo[i];
  n.L = p.L[b];
  return n;
}

// Ancestors of v are numbered in increasing order along the root path (parents[u] < u), so the
// depth of an ancestor u is the number of v's ancestors numbered below u.
__device__ __forceinline__ bool entry_visible_kind(int kind, int aux, const NodeVis& n) {
  switch (kind) {
    case kEntryShared:
      return true;
    case kEntryRaw:
      return aux >= n.raw_lo;
    case kEntryTree: {
      if (!((n.anc >> aux) & 1ull)) return false;
      const int dep = __popcll(n.anc & ((1ull << aux) - 1ull));
      return n.L + dep >= n.raw_lo;
    }
    case kEntryScr4:
      return (n.vis4 >> aux) & 1ull;
    case kEntryScr128:
      return (n.vis128 >> aux) & 1ull;
    default:
      return false;
  }
}

__device__ __forceinline__ bool entry_visible(const EntryRef& r, const NodeVis& n) {
  return entry_visible_kind(r.kind, r.aux, n);
}

// Split-KV merge: a warp per (request, node, head) row, 8 rows per block; lane l owns columns
// 4l .. 4l+3 of every 128-column group and writes them with one store.  Every lane derives the
// chunk weights itself (a few dozen broadcast loads), so the column loads of all chunks are
// independent and the row needs no synchronisation.
// Chunk rows are d + 4 floats (16-byte aligned for d a multiple of 8): O partial, m (log2
// units), l.
template <typename T>
__global__ void merge_kernel(int rows, int d, int n_chunks, const float* __restrict__ part,
                             T* __restrict__ O, float* __restrict__ lse) {
  // a warp per row: lane l combines columns 4l .. 4l+3 of every 128-column group
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t stride = d + 4;
  const float* pr = part + (int64_t)row * n_chunks * stride;
  float M = -INFINITY;
  for (int c = 0; c < n_chunks; ++c)
    if (pr[c * stride + d + 1] > 0.f) M = fmaxf(M, pr[c * stride + d]);
  float denom = 0.f;
  for (int c = 0; c < n_chunks; ++c)
    if (pr[c * stride + d + 1] > 0.f) denom += exp2f(pr[c * stride + d] - M) * pr[c * stride + d + 1];
  const float inv = denom > 0.f ? 1.f / denom : 0.f;
  for (int i = 4 * lane; i < d; i += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < n_chunks; ++c) {
      const float* pc = pr + c * stride;
      if (pc[d + 1] > 0.f) {
        const float w = exp2f(pc[d] - M);
        const float4 v = *reinterpret_cast<const float4*>(pc + i);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
    store_f4(O + (int64_t)row * d + i,
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
  if (lane == 0)
    lse[row] = denom > 0.f ? (M + log2f(denom)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace tv

template <typename T>
int tv_launch_merge(int B, int DH, int d, int n_chunks, const float* part, T* O, float* lse,
                    cudaStream_t stream) {
  const int rows = B * DH;
  const int rows_per_block = 8;   // 256 threads, a warp per row
  tv::merge_kernel<T><<<(rows + rows_per_block - 1) / rows_per_block, 32 * rows_per_block, 0,
                         stream>>>(rows, d, n_chunks, part, O, lse);
  return tv_check_launch("tv_tree_verify_attn (merge)");
}

int tv_launch_attn_simt_bf16(const tv::AttnParams<__nv_bfloat16>& p, cudaStream_t stream);
int tv_launch_attn_simt_f32(const tv::AttnParams<float>& p, cudaStream_t stream);
