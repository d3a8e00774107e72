// Online sequence compression (C4 / C128), the scratch pad and the accepted-path refresh.
//
// "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference":
//   §2.2  CSA/HCA compress blocks of positions online, at two granularities (here m = 4, 128);
//   §3.2  a branch that closes a block after the tree diverges must be compressed on its own;
//   §4.2  those branch states live in a scratch pad; after acceptance only the accepted path's
//         raw tokens and compressed entries are committed to the persistent cache.
//
// The report gives no compression formula; the library's fixed stand-in is the gated block sum
//   z_t = K_t . g_m,  w = softmax(z) over the block,  entry = (sum_t w_t K_t, sum_t w_t V_t),
// evaluated in fp32 and stored in the cache dtype.  A C4 entry is one CTA's work; a C128 entry is
// one cluster's: eight CTAs own 16 tokens each, share the block maximum and their partial sums
// through distributed shared memory, and every K/V row of the block is loaded in one round trip.
// Prefill and the scratch pad run the same routine per granularity with the same thread layout, so
// an entry computed in the scratch pad is bit-identical to the one prefill computes for the same
// committed block.
#include <cooperative_groups.h>
#include <math.h>

#include "tv_common.cuh"

namespace tv {

constexpr int kThreads = 256;                   // every compressor CTA: eight warps
constexpr int kWarps = kThreads / 32;
constexpr int kC128Ranks = 8;                   // CTAs per 128-token block (one cluster)
constexpr int kC128Tokens = 128 / kC128Ranks;   // tokens per CTA: two per warp
static_assert(kC128Tokens == 2 * kWarps, "two C128 tokens per warp");

// Raw 16-byte vector and its conversion to fp32 (loads are issued first, converted later, so
// many loads are in flight at once).
template <typename T>
__device__ __forceinline__ uint4 ld16(const T* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void cvt16(uint4 u, __nv_bfloat16*, float* out) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    out[2 * k] = f.x;
    out[2 * k + 1] = f.y;
  }
}
__device__ __forceinline__ void cvt16(uint4 u, float*, float* out) {
  out[0] = __uint_as_float(u.x);
  out[1] = __uint_as_float(u.y);
  out[2] = __uint_as_float(u.z);
  out[3] = __uint_as_float(u.w);
}

template <typename T>
struct VecWidth;
template <>
struct VecWidth<__nv_bfloat16> {
  static constexpr int n = 8;
};
template <>
struct VecWidth<float> {
  static constexpr int n = 4;
};

// 16-byte asynchronous copy global -> shared.  The copies a thread issued are committed as a group
// (cp_async_commit); cp_async_wait(n) waits until at most the n most recent groups are pending;
// a barrier then makes every thread's copies visible to the CTA.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait(int pending) {
  if (pending > 0)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

constexpr int kMaxPairs = kMaxHeadDim / 2 / kC128Ranks;   // dimension pairs a rank finishes

// Shared memory of a C4 CTA (prefill and scratch pad).
template <typename T>
struct C4Smem {
  T rows4[4][2][kMaxHeadDim];   // the block's rows: token t: [0] = K row, [1] = V row
  float gate4[kMaxHeadDim];
  float z4[4];                  // gate logits
};

// Shared memory of a C128 cluster CTA (prefill and scratch pad).
template <typename T>
struct C128Smem {
  T rows[kC128Tokens][2][kMaxHeadDim];     // this rank's 16 block rows: [0] = K row, [1] = V row
  float gate128[kMaxHeadDim];
  float4 recv[2][kC128Ranks][kMaxPairs];   // by entry parity: sums (K 2p, K 2p+1, V 2p, V 2p+1)
                                           // of the dimension pairs this rank finishes, per
                                           // sending rank
  float2 ms[2][kC128Ranks];                // by entry parity: every rank's (max logit, sum of
                                           // weights)
  float z[kC128Tokens];                    // gate logits
  float w[kC128Tokens];                    // weights exp(z_t - m) (m: this rank's maximum)
};

// Copies rows (K and V) of the tokens t < n_tok with take[t] (all if take is null) into the row
// slots dst[t]: each thread issues 16-byte copies, all in flight at once.
template <typename T>
__device__ __forceinline__ void fetch_rows(T (*dst)[2][kMaxHeadDim], const T* const* srcK,
                                           const T* const* srcV, int n_tok, const bool* take,
                                           int d) {
  constexpr int VW = VecWidth<T>::n;
  const int per_row = d / VW;
  for (int t = 0; t < n_tok; ++t) {
    if (take != nullptr && !take[t]) continue;
    for (int c = threadIdx.x; c < 2 * per_row; c += blockDim.x) {
      const int which = c >= per_row;
      const int q = c - which * per_row;
      cp_async16(&dst[t][which][q * VW], (which ? srcV[t] : srcK[t]) + q * VW);
    }
  }
}

// A warp's view of one row: lane l holds the 16-byte groups l, l + 32, ... (KV of them at the
// largest head dimension; groups past d are zero).
template <typename T>
struct Lane16 {
  static constexpr int VW = VecWidth<T>::n;
  static constexpr int KV = kMaxHeadDim / (32 * VW);
};

// Gate logit z = K . g of one row, by one warp, from the lane's groups x[0..KV) of the row and
// the gate in shared memory: per lane in group then element order, then a butterfly sum over the
// lanes (every lane returns the same value).  The same arithmetic whether the row sits in shared
// memory or in registers.
template <typename T>
__device__ __forceinline__ float lane_logit(const uint4 (&x)[Lane16<T>::KV], const float* gate,
                                            int d, int lane) {
  constexpr int VW = Lane16<T>::VW;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < Lane16<T>::KV; ++k) {
    const int i = lane * VW + 32 * VW * k;
    if (i >= d) break;
    float f[VW];
    cvt16(x[k], (T*)nullptr, f);
#pragma unroll
    for (int e = 0; e < VW; ++e) acc = fmaf(f[e], gate[i + e], acc);
  }
  return warp_sum(acc);
}

template <typename T>
__device__ __forceinline__ float row_logit(const T* row, const float* gate, int d, int lane) {
  constexpr int VW = Lane16<T>::VW;
  uint4 x[Lane16<T>::KV];
#pragma unroll
  for (int k = 0; k < Lane16<T>::KV; ++k) {
    const int i = lane * VW + 32 * VW * k;
    x[k] = i < d ? *reinterpret_cast<const uint4*>(row + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  return lane_logit<T>(x, gate, d, lane);
}

// Two consecutive elements as fp32.
__device__ __forceinline__ float2 ld_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Weighted sums over n_tok token rows in shared memory for the dimension pair (2p, 2p+1): tokens
// in order, one fused multiply-add each.  Returns (K 2p, K 2p+1, V 2p, V 2p+1).
template <typename T, int N>
__device__ __forceinline__ float4 pair_sums(const T (*rows)[2][kMaxHeadDim], const float* w,
                                            int p) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int t = 0; t < N; ++t) {
    const float2 k = ld_pair(&rows[t][0][2 * p]);
    const float2 v = ld_pair(&rows[t][1][2 * p]);
    a.x = fmaf(w[t], k.x, a.x);
    a.y = fmaf(w[t], k.y, a.y);
    a.z = fmaf(w[t], v.x, a.z);
    a.w = fmaf(w[t], v.y, a.w);
  }
  return a;
}

// ---- C4: one entry per CTA -------------------------------------------------------------------
// One entry from the 4 rows in sm.rows4 (position order; the caller has fetched them): warp t
// forms logit z_t; with M = max z_t and w_t = exp(z_t - M), dimension i of the entry is
// (sum_t w_t K_t[i], tokens in order) / (sum_t w_t).  Prefill and the scratch pad both run this
// routine, so equal rows give bit-identical entries.  out2K / out2V (nullable): a second place
// the entry is written to.  pending_after: 1 if the caller committed one more copy group after
// this entry's rows (the C128 rows), which need not have landed yet.
template <typename T>
__device__ void entry4(int d, const float* gate, T* outK, T* outV, T* out2K, T* out2V,
                       int pending_after, C4Smem<T>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  cp_async_wait(pending_after);   // groups committed after this entry's rows may stay pending
  __syncthreads();
  if (warp < 4) {
    const float z = row_logit<T>(sm.rows4[warp][0], gate, d, lane);
    if (lane == 0) sm.z4[warp] = z;
  }
  __syncthreads();
  const float M = fmaxf(fmaxf(sm.z4[0], sm.z4[1]), fmaxf(sm.z4[2], sm.z4[3]));
  float w[4], S = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    w[t] = expf(sm.z4[t] - M);
    S += w[t];
  }
  for (int p = threadIdx.x; 2 * p < d; p += blockDim.x) {
    float4 a = pair_sums<T, 4>(sm.rows4, w, p);
    a.x /= S;
    a.y /= S;
    a.z /= S;
    a.w /= S;
    store_f(outK + 2 * p, a.x);
    store_f(outK + 2 * p + 1, a.y);
    store_f(outV + 2 * p, a.z);
    store_f(outV + 2 * p + 1, a.w);
    if (out2K != nullptr) {
      store_f(out2K + 2 * p, a.x);
      store_f(out2K + 2 * p + 1, a.y);
      store_f(out2V + 2 * p, a.z);
      store_f(out2V + 2 * p + 1, a.w);
    }
  }
  __syncthreads();   // rows4 and z4 are free for the next entry
}

// ---- C128: one entry per cluster --------------------------------------------------------------
// One 128-token entry by a cluster of eight CTAs: rank r holds the block's tokens 16r .. 16r+15
// in sm.rows (the caller has fetched them); warp w forms the logits of tokens 2w and 2w+1.  Each
// rank takes its own maximum m_r, forms w_t = exp(z_t - m_r) and, per dimension pair, sums w_t K_t
// and w_t V_t over its tokens in order; it sends the pair sums to the rank that finishes the pair
// and (m_r, sum_t w_t) to every rank -- one cluster barrier.  The finishing rank rescales the
// eight ranks' sums to M = max m_r (factor exp(m_r - M)), adds them in rank order and divides by
// the rescaled sum of weights.  All orders are fixed: the entry depends only on the block's rows,
// so prefill and the scratch pad agree bit for bit.  parity: the entry's index & 1 among the
// cluster's consecutive entries (the receive buffers alternate, so a rank that runs ahead into
// the next entry never writes a buffer that a slower rank still reads).  after_rows() runs on
// every thread once the rank's sums are sent, before the cluster barrier: the caller may refetch
// rows there (after a barrier of its own, since other threads may still read them).
template <typename T, typename AfterRows>
__device__ void entry128(int d, const float* gate, T* outK, T* outV, int parity, C128Smem<T>& sm,
                         AfterRows&& after_rows) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rank = (int)cl.block_rank();
  const int t0 = 2 * warp;
  const int ppr = (d / 2 + kC128Ranks - 1) / kC128Ranks;   // dimension pairs per rank
  cp_async_wait(0);
  __syncthreads();
  const float z0 = row_logit<T>(sm.rows[t0][0], gate, d, lane);
  const float z1 = row_logit<T>(sm.rows[t0 + 1][0], gate, d, lane);
  if (lane == 0) {
    sm.z[t0] = z0;
    sm.z[t0 + 1] = z1;
  }
  __syncthreads();
  float m = sm.z[0];
  for (int t = 1; t < kC128Tokens; ++t) m = fmaxf(m, sm.z[t]);
  if (threadIdx.x < kC128Tokens) sm.w[threadIdx.x] = expf(sm.z[threadIdx.x] - m);
  __syncthreads();
  for (int p = threadIdx.x; 2 * p < d; p += blockDim.x) {
    const float4 a = pair_sums<T, kC128Tokens>(sm.rows, sm.w, p);
    const int owner = p / ppr;
    *cl.map_shared_rank(&sm.recv[parity][rank][p - owner * ppr], owner) = a;
  }
  if (threadIdx.x < kC128Ranks) {   // (m, sum of weights) to every rank
    float s = 0.f;
    for (int t = 0; t < kC128Tokens; ++t) s += sm.w[t];
    *cl.map_shared_rank(&sm.ms[parity][rank], (int)threadIdx.x) = make_float2(m, s);
  }
  after_rows();
  cl.sync();   // every rank's sums have arrived
  pdl_wait();   // (scratch pad) the kernel before this one has completed before any store
  const int p = rank * ppr + (int)threadIdx.x;
  if ((int)threadIdx.x < ppr && 2 * p < d) {
    float M = sm.ms[parity][0].x;
    for (int q = 1; q < kC128Ranks; ++q) M = fmaxf(M, sm.ms[parity][q].x);
    float S = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < kC128Ranks; ++q) {
      const float f = expf(sm.ms[parity][q].x - M);
      const float4 x = sm.recv[parity][q][threadIdx.x];
      S = fmaf(f, sm.ms[parity][q].y, S);
      a.x = fmaf(f, x.x, a.x);
      a.y = fmaf(f, x.y, a.y);
      a.z = fmaf(f, x.z, a.z);
      a.w = fmaf(f, x.w, a.w);
    }
    store_f(outK + 2 * p, a.x / S);
    store_f(outK + 2 * p + 1, a.y / S);
    store_f(outV + 2 * p, a.z / S);
    store_f(outV + 2 * p + 1, a.w / S);
  }
  __syncthreads();   // the rows may be refetched for the next entry
}

// ---- prefill: every complete block of the committed prefix ---------------------------------
// C4: grid.x entry index (strided), grid.y request.
template <typename T>
__global__ void __launch_bounds__(kThreads) prefill4_kernel(
    Paging pg, int d, int64_t raw_cap, int64_t cap4, const T* __restrict__ rawK,
    const T* __restrict__ rawV, const int32_t* __restrict__ L, const float* __restrict__ g,
    T* __restrict__ CK, T* __restrict__ CV, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  C4Smem<T>& sm = *reinterpret_cast<C4Smem<T>*>(smem_raw);
  __shared__ const T* rowK[4];
  __shared__ const T* rowV[4];
  const int b = blockIdx.y;
  const int Lb = L[b];
  if (Lb < 0 || Lb > raw_cap || (int64_t)(Lb / 4) > cap4) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, TV_ERR_CAPACITY);
    return;
  }
  for (int i = threadIdx.x; i < d; i += blockDim.x) sm.gate4[i] = g[i];
  const int n = Lb / 4;
  for (int j = blockIdx.x; j < n; j += gridDim.x) {
    if (threadIdx.x < 4) {
      const int64_t row = layer_row(pg, b, (int64_t)j * 4 + threadIdx.x, raw_cap, 1, status);
      rowK[threadIdx.x] = rawK + row * d;
      rowV[threadIdx.x] = rawV + row * d;
    }
    __syncthreads();
    fetch_rows<T>(sm.rows4, rowK, rowV, 4, nullptr, d);
    cp_async_commit();
    const int64_t out = layer_row(pg, b, j, cap4, 4, status) * d;
    entry4<T>(d, sm.gate4, CK + out, CV + out, nullptr, nullptr, 0, sm);
  }
}

// C128: a cluster (8 CTAs along x) per entry; grid.y entry index (strided), grid.z request.
template <typename T>
__global__ void __cluster_dims__(kC128Ranks, 1, 1) __launch_bounds__(kThreads)
    prefill128_kernel(Paging pg, int d, int64_t raw_cap, int64_t cap_m, const T* __restrict__ rawK,
                      const T* __restrict__ rawV, const int32_t* __restrict__ L,
                      const float* __restrict__ g, T* __restrict__ CK, T* __restrict__ CV,
                      int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  C128Smem<T>& sm = *reinterpret_cast<C128Smem<T>*>(smem_raw);
  __shared__ const T* rowK[kC128Tokens];
  __shared__ const T* rowV[kC128Tokens];
  const int b = blockIdx.z;
  const int rank = (int)cooperative_groups::this_cluster().block_rank();
  const int Lb = L[b];
  if (Lb < 0 || Lb > raw_cap || (int64_t)(Lb / 128) > cap_m) {   // uniform over the cluster
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) record_error(status, TV_ERR_CAPACITY);
    return;
  }
  for (int i = threadIdx.x; i < d; i += blockDim.x) sm.gate128[i] = g[i];
  const int n = Lb / 128;
  int parity = 0;
  for (int j = blockIdx.y; j < n; j += gridDim.y, parity ^= 1) {
    if (threadIdx.x < kC128Tokens) {
      const int64_t row =
          layer_row(pg, b, (int64_t)j * 128 + kC128Tokens * rank + threadIdx.x, raw_cap, 1, status);
      rowK[threadIdx.x] = rawK + row * d;
      rowV[threadIdx.x] = rawV + row * d;
    }
    __syncthreads();
    fetch_rows<T>(sm.rows, rowK, rowV, kC128Tokens, nullptr, d);
    cp_async_commit();
    const int64_t out = layer_row(pg, b, j, cap_m, 128, status) * d;
    entry128<T>(d, sm.gate128, CK + out, CV + out, parity, sm, [] {});
  }
}

// Row pointers of token t (0..3) of the C4 block that node v closes: committed rows before L,
// then the rows of v's path.
template <typename T>
__device__ __forceinline__ void c4_rows(const Paging& pg, int b, int D, int d, int64_t raw_cap,
                                        int Lb, int v, const int* dep, const int* par,
                                        const T* rawK, const T* rawV, const T* treeK,
                                        const T* treeV, int t, const T** rowK4, const T** rowV4,
                                        int32_t* status) {
  const int p = Lb + dep[v] - 3 + t;   // >= 0 because pos + 1 is a positive multiple of 4
  if (p < Lb) {
    const int64_t row = layer_row(pg, b, p, raw_cap, 1, status);
    rowK4[t] = rawK + row * d;
    rowV4[t] = rawV + row * d;
  } else {
    int u = v;   // the ancestor of v at depth p - L
    for (int k = dep[v]; k > p - Lb; --k) u = par[u];
    const int64_t row = (int64_t)b * D + u;
    rowK4[t] = treeK + row * d;
    rowV4[t] = treeV + row * d;
  }
}

// Row pointer of this CTA's token t (block token 16 * rank + t) of the C128 block that the node
// with the given path closes at position pos128: a committed row before L, else a path row.
// Returns whether the token is a tree row.
template <typename T>
__device__ __forceinline__ bool c128_row(const Paging& pg, int b, int D, int d, int64_t raw_cap,
                                         int Lb, int pos128, int rank, const int* path,
                                         const T* rawK, const T* rawV, const T* treeK,
                                         const T* treeV, int t, const T** rowK, const T** rowV,
                                         int32_t* status) {
  const int p = pos128 + 1 - 128 + kC128Tokens * rank + t;   // >= 0
  if (p < Lb) {
    const int64_t row = layer_row(pg, b, p, raw_cap, 1, status);
    rowK[t] = rawK + row * d;
    rowV[t] = rawV + row * d;
    return false;
  }
  const int64_t row = (int64_t)b * D + path[p - Lb];
  rowK[t] = treeK + row * d;
  rowV[t] = treeV + row * d;
  return true;
}

// ---- scratch pad: entries of blocks closed by tree nodes ------------------------------------
// Node v's token sits at position pos_v = L + depth(v); row v of the C4 (C128) scratch pad is the
// entry of the block that token closes -- positions pos_v - m + 1 .. pos_v of prefix + path(v) --
// or zeros.

// The tree of one request in shared memory: validity, depths, first children and the cached
// chain (the root, its lowest-numbered child, ...), all nodes at once.  par[v] must be loaded and
// first[v] = D for v < D.  Returns (in *ok, uniformly) whether every parent precedes its child.
__device__ __forceinline__ void tree_structure(int D, const int* par, int* first, int* dep,
                                               int* cached, int* ok) {
  const int tid = threadIdx.x;
  if (tid < D) {
    const int p = par[tid];
    const bool good = (tid == 0) ? (p == -1) : (p >= 0 && p < tid);
    if (!good) *ok = 0;
    else if (tid > 0) atomicMin(&first[p], tid);
  }
  __syncthreads();
  if (tid < D && *ok) {
    int depth = 0, chain = 1;
    for (int u = tid; u != 0 && depth < D; ++depth) {   // parents precede children: ends at root
      const int q = par[u];
      if (first[q] != u) chain = 0;
      u = q;
    }
    dep[tid] = depth;
    if (cached != nullptr) cached[tid] = chain;
  }
  __syncthreads();
}

// Warp 0: the nodes (in node order) whose position closes an m-block, into list; returns the count
// on every lane of warp 0.
__device__ __forceinline__ int closing_nodes(int D, int Lb, const int* dep, int m, int* list) {
  const int lane = threadIdx.x & 31;
  int n = 0;
  for (int v0 = 0; v0 < D; v0 += 32) {
    const int v = v0 + lane;
    const bool c = v < D && ((Lb + dep[v] + 1) % m) == 0;
    const unsigned mask = __ballot_sync(0xffffffffu, c);
    if (c) list[n + __popc(mask & ((1u << lane) - 1u))] = v;
    n += __popc(mask);
  }
  return n;
}

// Shared memory of a scratch-pad CTA: its C4 block and its share of a C128 block side by side,
// so both fetches can be in flight together.
template <typename T>
struct BranchSmem {
  C4Smem<T> c4;
  C128Smem<T> c128;
};

// One cluster of eight CTAs per request (grid (8, B)).  The C4 entries and the zero rows are
// spread over the CTAs (round robin); the C128 entries, all at the one depth whose position
// closes a 128-block (D <= 64 < 128), are computed by the whole cluster one after another
// (entry128), the committed rows of their block fetched once.  With staging, a node on the
// cached chain also writes its raw row and its C4 entry to their final places past L.  Round
// trips: the length, parents and gates; then the CTA's first C4 block and its share of the C128
// block, in flight together.
template <typename T>
__global__ void __cluster_dims__(kC128Ranks, 1, 1) __launch_bounds__(kThreads)
    branch_kernel(Paging pg, int D, int d, int comp_mask, int64_t raw_cap, T* rawK, T* rawV,
                  int stage, int64_t c4_cap, T* c4K, T* c4V, const int32_t* __restrict__ L,
                  const T* __restrict__ treeK, const T* __restrict__ treeV,
                  const int32_t* __restrict__ parents, const float* __restrict__ g4,
                  const float* __restrict__ g128, T* scrK4, T* scrV4, T* scrK128, T* scrV128,
                  int32_t* status) {
  pdl_launch_dependents();   // the next kernel may start its prologue now
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BranchSmem<T>& sm = *reinterpret_cast<BranchSmem<T>*>(smem_raw);
  __shared__ int s_par[kMaxD], s_dep[kMaxD], s_first[kMaxD], s_cached[kMaxD];
  __shared__ int s_list4[kMaxD], s_list128[kMaxD];
  __shared__ int s_n4, s_n128, s_ok, s_L;
  __shared__ const T* rowK4[4];
  __shared__ const T* rowV4[4];
  __shared__ const T* rowK[kC128Tokens];
  __shared__ const T* rowV[kC128Tokens];
  __shared__ bool tree_tok[kC128Tokens];   // this CTA's C128 token is a tree row
  __shared__ int s_any_tree;               // some token of this CTA is a tree row
  __shared__ int path[kMaxD];              // path of the C128 entry in progress
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int rank = (int)cooperative_groups::this_cluster().block_rank();
  const bool has4 = comp_mask & TV_COMP_C4, has128 = comp_mask & TV_COMP_C128;
  // 1. the request's length, parents and the gates (one round trip)
  if (tid < D) {
    s_par[tid] = parents[(int64_t)b * D + tid];
    s_first[tid] = D;
  }
  if (tid == kMaxD) s_L = L[b];
  if (tid == 0) s_ok = 1;
  for (int i = tid; i < d; i += blockDim.x) {
    if (has4) sm.c4.gate4[i] = g4[i];
    if (has128) sm.c128.gate128[i] = g128[i];
  }
  __syncthreads();
  const int Lb = s_L;
  // 2. the tree and the closers
  tree_structure(D, s_par, s_first, s_dep, s_cached, &s_ok);
  const bool ok = s_ok && Lb >= 0 && Lb <= raw_cap;
  if (tid < 32) {
    const int n4 = (ok && has4) ? closing_nodes(D, Lb, s_dep, 4, s_list4) : 0;
    const int n128 = (ok && has128) ? closing_nodes(D, Lb, s_dep, 128, s_list128) : 0;
    if (tid == 0) {
      s_n4 = n4;
      s_n128 = n128;
      if (!ok && rank == 0)
        record_error(status, (Lb < 0 || Lb > raw_cap) ? TV_ERR_CAPACITY : TV_ERR_BAD_TREE);
    }
  }
  __syncthreads();
  const int n4 = s_n4, n128 = s_n128;
  const int pos128 = n128 > 0 ? Lb + s_dep[s_list128[0]] : 0;   // one depth closes 128-blocks
  auto c128_path = [&](int v) {   // thread 0: the path of node v
    for (int k = s_dep[v], u = v; k >= 0; --k) {
      path[k] = u;
      u = s_par[u];
    }
  };
  // 3. row pointers of this CTA's first C4 block and of its share of the first C128 block; the C4
  //    group is committed first, so its entry need not wait for the C128 rows
  if (n128 > 0 && tid == 0) c128_path(s_list128[0]);
  if (rank < n4 && tid >= 32 && tid < 36)
    c4_rows(pg, b, D, d, raw_cap, Lb, s_list4[rank], s_dep, s_par, rawK, rawV, treeK, treeV,
            tid - 32, rowK4, rowV4, status);
  __syncthreads();
  if (tid == 0) s_any_tree = 0;
  __syncthreads();
  if (n128 > 0 && tid < kC128Tokens) {
    tree_tok[tid] = c128_row(pg, b, D, d, raw_cap, Lb, pos128, rank, path, rawK, rawV, treeK,
                             treeV, tid, rowK, rowV, status);
    if (tree_tok[tid]) s_any_tree = 1;
  }
  __syncthreads();
  if (rank < n4) {
    fetch_rows<T>(sm.c4.rows4, rowK4, rowV4, 4, nullptr, d);
    cp_async_commit();
  }
  if (n128 > 0) {
    fetch_rows<T>(sm.c128.rows, rowK, rowV, kC128Tokens, nullptr, d);
    cp_async_commit();
  }
  // launched as a programmatic dependent: everything so far only read inputs; the kernel before
  // this one in the stream must be complete before the first write
  pdl_wait();
  // 4. per node (round robin over the CTAs): staging of the raw row, zero rows
  for (int v = rank; v < D; v += kC128Ranks) {
    const int pos = Lb + s_dep[v];
    const int64_t out = ((int64_t)b * D + v) * d;
    if (ok && stage && s_cached[v] && pos < raw_cap) {
      const int64_t dst = layer_row(pg, b, pos, raw_cap, 1, status) * d;
      for (int i = tid; i < d; i += blockDim.x) {
        rawK[dst + i] = treeK[out + i];
        rawV[dst + i] = treeV[out + i];
      }
    }
    const bool closes4 = ok && ((pos + 1) & 3) == 0;
    const bool closes128 = ok && ((pos + 1) & 127) == 0;
    for (int i = tid; i < d; i += blockDim.x) {
      if (has4 && !closes4) {
        store_f(scrK4 + out + i, 0.f);
        store_f(scrV4 + out + i, 0.f);
      }
      if (has128 && !closes128) {
        store_f(scrK128 + out + i, 0.f);
        store_f(scrV128 + out + i, 0.f);
      }
    }
  }
  // 5. C4 entries (round robin over the CTAs; the first one's rows are already in flight)
  for (int j = rank; j < n4; j += kC128Ranks) {
    const int v = s_list4[j];
    const int pos = Lb + s_dep[v];
    if (j != rank) {
      if (tid < 4) c4_rows(pg, b, D, d, raw_cap, Lb, v, s_dep, s_par, rawK, rawV, treeK, treeV,
                           tid, rowK4, rowV4, status);
      __syncthreads();
      fetch_rows<T>(sm.c4.rows4, rowK4, rowV4, 4, nullptr, d);
      cp_async_commit();
    }
    const int64_t out = ((int64_t)b * D + v) * d;
    const int64_t entry = (pos + 1) / 4 - 1;
    T* sK = nullptr;
    T* sV = nullptr;
    if (stage && s_cached[v] && entry < c4_cap) {   // C4 refreshes promptly
      const int64_t dst = layer_row(pg, b, entry, c4_cap, 4, status) * d;
      sK = c4K + dst;
      sV = c4V + dst;
    }
    entry4<T>(d, sm.c4.gate4, scrK4 + out, scrV4 + out, sK, sV, j == rank && n128 > 0 ? 1 : 0,
              sm.c4);
  }
  // 6. C128 entries, one after another by the whole cluster (uniform over the cluster); the
  //    block's committed rows stay in place, only the tree rows change between entries: a CTA
  //    holding tree rows fetches the next entry's as soon as its sums for this one are sent
  const bool any_tree = s_any_tree != 0;   // uniform over the CTA
  for (int j = 0; j < n128; ++j) {
    const int v = s_list128[j];
    const int64_t out = ((int64_t)b * D + v) * d;
    entry128<T>(d, sm.c128.gate128, scrK128 + out, scrV128 + out, j & 1, sm.c128, [&] {
      if (j + 1 < n128 && any_tree) {
        __syncthreads();   // every thread is done with this entry's rows
        if (tid == 0) c128_path(s_list128[j + 1]);
        __syncthreads();
        if (tid < kC128Tokens && tree_tok[tid])
          c128_row(pg, b, D, d, raw_cap, Lb, pos128, rank, path, rawK, rawV, treeK, treeV, tid,
                   rowK, rowV, status);
        __syncthreads();
        fetch_rows<T>(sm.c128.rows, rowK, rowV, kC128Tokens, tree_tok, d);
        cp_async_commit();
      }
    });
  }
}

// ---- refresh: commit the accepted path --------------------------------------------------------
// One CTA per request.  Copies the accepted tokens' K/V into the raw rows L .. L+n-1 and the
// scratch rows of accepted nodes that close a block into the persistent entries (all rows in
// parallel: each 16-byte chunk of each row is one thread's job), then advances L.  The inputs
// arrive in one round trip; accepted node i owns the job slots 3i (raw row), 3i+1 (C4 entry) and
// 3i+2 (C128 entry), so the job list is built in parallel with no scan.
__global__ void refresh_kernel(Paging pg, int D, int d, int es, int comp_mask, int64_t raw_cap,
                               int64_t c4_cap, int64_t c128_cap, int stage,
                               const int32_t* __restrict__ parents,
                               const int32_t* __restrict__ accept_len,
                               const int32_t* __restrict__ path_all, const char* treeK,
                               const char* treeV, const char* scrK4, const char* scrV4,
                               const char* scrK128, const char* scrV128, char* rawK, char* rawV,
                               char* c4K, char* c4V, char* c128K, char* c128V, int32_t* L,
                               int32_t* committed, int32_t* status) {
  // launched as a programmatic dependent of the acceptance walk, whose results it reads
  pdl_wait();
  constexpr int kSlots = 3 * kMaxD;
  __shared__ const char* s_srcK[kSlots];
  __shared__ const char* s_srcV[kSlots];
  __shared__ char* s_dstK[kSlots];
  __shared__ char* s_dstV[kSlots];
  __shared__ int s_path[kMaxD];
  __shared__ int s_par[kMaxD];
  __shared__ int s_L, s_n, s_ok, s_staged;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t row_bytes = (int64_t)d * es;
  if (tid < D) {
    s_path[tid] = path_all[(int64_t)b * D + tid];
    if (stage) s_par[tid] = parents[(int64_t)b * D + tid];
  }
  if (tid == 32) s_L = L[b];
  if (tid == 64) s_n = accept_len[b];
  __syncthreads();
  if (tid == 0) {
    const int Lb = s_L, n = s_n;
    int ok = 1, code = 0;
    if (n < 1 || n > D || Lb < 0) { ok = 0; code = TV_ERR_ARG; }
    for (int i = 0; ok && i < n; ++i)
      if (s_path[i] < 0 || s_path[i] >= D) { ok = 0; code = TV_ERR_ARG; }
    if (ok) {
      const int64_t Lnew = (int64_t)Lb + n;
      if (Lnew > raw_cap) { ok = 0; code = TV_ERR_CAPACITY; }
      if ((comp_mask & TV_COMP_C4) && Lnew / 4 > c4_cap) { ok = 0; code = TV_ERR_CAPACITY; }
      if ((comp_mask & TV_COMP_C128) && Lnew / 128 > c128_cap) { ok = 0; code = TV_ERR_CAPACITY; }
    }
    if (!ok) record_error(status, code);
    // with staging, the accepted nodes on the cached chain (the root, its lowest-numbered child,
    // ...) already sit in their final raw rows and C4 entries: the accepted path follows that
    // chain up to the first node where it leaves it
    int staged = 0;
    if (ok && stage) {
      int c = 0;
      while (staged < n && s_path[staged] == c) {
        ++staged;
        int next = -1;
        for (int u = c + 1; u < D; ++u)
          if (s_par[u] == c) {
            next = u;
            break;
          }
        if (next < 0) break;
        c = next;
      }
    }
    s_ok = ok;
    s_staged = staged;
  }
  __syncthreads();
  int32_t* cpos = committed + (int64_t)b * D;
  if (!s_ok) {
    for (int i = tid; i < D; i += blockDim.x) cpos[i] = -1;
    return;
  }
  const int Lb = s_L, n = s_n;
  if (tid < n) {
    const int i = tid;
    const int64_t src = ((int64_t)b * D + s_path[i]) * row_bytes;
    const bool on_chain = i < s_staged;
    const int e = Lb + i;
    const bool raw = !on_chain;
    const bool e4 = (comp_mask & TV_COMP_C4) && ((e + 1) & 3) == 0 && !on_chain;
    const bool e128 = (comp_mask & TV_COMP_C128) && ((e + 1) & 127) == 0;
    if (raw) {
      const int64_t dst = layer_row(pg, b, e, raw_cap, 1, status) * row_bytes;
      s_srcK[3 * i] = treeK + src;
      s_srcV[3 * i] = treeV + src;
      s_dstK[3 * i] = rawK + dst;
      s_dstV[3 * i] = rawV + dst;
    } else {
      s_srcK[3 * i] = nullptr;
    }
    if (e4) {
      const int64_t cd = layer_row(pg, b, (e + 1) / 4 - 1, c4_cap, 4, status) * row_bytes;
      s_srcK[3 * i + 1] = scrK4 + src;
      s_srcV[3 * i + 1] = scrV4 + src;
      s_dstK[3 * i + 1] = c4K + cd;
      s_dstV[3 * i + 1] = c4V + cd;
    } else {
      s_srcK[3 * i + 1] = nullptr;
    }
    if (e128) {
      const int64_t cd = layer_row(pg, b, (e + 1) / 128 - 1, c128_cap, 128, status) * row_bytes;
      s_srcK[3 * i + 2] = scrK128 + src;
      s_srcV[3 * i + 2] = scrV128 + src;
      s_dstK[3 * i + 2] = c128K + cd;
      s_dstV[3 * i + 2] = c128V + cd;
    } else {
      s_srcK[3 * i + 2] = nullptr;
    }
  }
  __syncthreads();
  // the copies, kCopyUnroll chunks per thread with all their loads in flight before the stores
  constexpr int kCopyUnroll = 4;
  const int chunks = (int)(row_bytes / 16);
  const int total = 3 * n * chunks;
  for (int k0 = tid; k0 < total; k0 += kCopyUnroll * blockDim.x) {
    uint4 vk[kCopyUnroll], vv[kCopyUnroll];
    int jc[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int k = k0 + u * blockDim.x;
      const int j = k / chunks, c = k - j * chunks;
      jc[u] = -1;
      if (k < total && s_srcK[j] != nullptr) {
        vk[u] = reinterpret_cast<const uint4*>(s_srcK[j])[c];
        vv[u] = reinterpret_cast<const uint4*>(s_srcV[j])[c];
        jc[u] = k;
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      if (jc[u] < 0) continue;
      const int j = jc[u] / chunks, c = jc[u] - j * chunks;
      reinterpret_cast<uint4*>(s_dstK[j])[c] = vk[u];
      reinterpret_cast<uint4*>(s_dstV[j])[c] = vv[u];
    }
  }
  for (int i = tid; i < D; i += blockDim.x) cpos[i] = i < n ? Lb + i : -1;
  __syncthreads();
  if (tid == 0) L[b] = Lb + n;
}

}  // namespace tv

// ---- launchers --------------------------------------------------------------------------------
template <typename K>
static int smem_ready(K kernel, size_t bytes, const char* what) {
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return tv_set_error(TV_ERR_CUDA, "%s: cudaFuncSetAttribute failed: %s", what,
                        cudaGetErrorString(e));
  }
  return TV_OK;
}

template <typename T>
static int launch_prefill_t(const tv_shape* s, const void* rawK, const void* rawV,
                            const int32_t* L, const float* g4, const float* g128, void* c4K,
                            void* c4V, void* c128K, void* c128V, int32_t* status,
                            cudaStream_t stream) {
  const int d = s->d;
  if (s->comp_mask & TV_COMP_C4) {
    const size_t smem = sizeof(tv::C4Smem<T>);
    static const int ready = smem_ready(tv::prefill4_kernel<T>, smem, "tv_prefill_compress (C4)");
    if (ready != TV_OK) return ready;
    const int64_t cap = s->c4_cap;
    const unsigned gx = (unsigned)(cap < 1 ? 1 : (cap > (1 << 20) ? (1 << 20) : cap));
    tv::prefill4_kernel<T><<<dim3(gx, s->B), tv::kThreads, smem, stream>>>(
        tv::paging_of(s), d, s->raw_cap, cap, (const T*)rawK, (const T*)rawV, L, g4, (T*)c4K,
        (T*)c4V, status);
    if (int rc = tv_check_launch("tv_prefill_compress (C4)")) return rc;
  }
  if (s->comp_mask & TV_COMP_C128) {
    const size_t smem = sizeof(tv::C128Smem<T>);
    static const int ready =
        smem_ready(tv::prefill128_kernel<T>, smem, "tv_prefill_compress (C128)");
    if (ready != TV_OK) return ready;
    const int64_t cap = s->c128_cap;
    const unsigned gy = (unsigned)(cap < 1 ? 1 : (cap > 65535 ? 65535 : cap));
    tv::prefill128_kernel<T><<<dim3(tv::kC128Ranks, gy, s->B), tv::kThreads, smem, stream>>>(
        tv::paging_of(s), d, s->raw_cap, cap, (const T*)rawK, (const T*)rawV, L, g128,
        (T*)c128K, (T*)c128V, status);
    if (int rc = tv_check_launch("tv_prefill_compress (C128)")) return rc;
  }
  return TV_OK;
}

int tv_launch_prefill(const tv_shape* s, const void* rawK, const void* rawV, const int32_t* L,
                      const float* g4, const float* g128, void* c4K, void* c4V, void* c128K,
                      void* c128V, int32_t* status, cudaStream_t stream) {
  if (s->dtype == TV_BF16)
    return launch_prefill_t<__nv_bfloat16>(s, rawK, rawV, L, g4, g128, c4K, c4V, c128K, c128V,
                                           status, stream);
  return launch_prefill_t<float>(s, rawK, rawV, L, g4, g128, c4K, c4V, c128K, c128V, status,
                                 stream);
}

template <typename T>
static int launch_branch_t(const tv_shape* s, void* rawK, void* rawV, void* c4K, void* c4V,
                           const int32_t* L, const void* treeK, const void* treeV,
                           const int32_t* parents, const float* g4, const float* g128,
                           void* scrK4, void* scrV4, void* scrK128, void* scrV128,
                           int32_t* status, cudaStream_t stream) {
  const size_t smem = sizeof(tv::BranchSmem<T>);
  static const int ready = smem_ready(tv::branch_kernel<T>, smem, "tv_branch_compress");
  if (ready != TV_OK) return ready;
  // a programmatic dependent of the kernel before it (normally the plan): it reads the tree and
  // the prefix while that kernel finishes, and writes only after it has completed
  const cudaError_t e = tv::launch_pdl(
      tv::branch_kernel<T>, dim3(tv::kC128Ranks, s->B), dim3(tv::kThreads), smem, stream,
      tv::paging_of(s), s->D, s->d, s->comp_mask, s->raw_cap, (T*)rawK, (T*)rawV,
      (int)s->stage_chain, s->c4_cap, (T*)c4K, (T*)c4V, L, (const T*)treeK, (const T*)treeV,
      parents, g4, g128, (T*)scrK4, (T*)scrV4, (T*)scrK128, (T*)scrV128, status);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return tv_set_error(TV_ERR_CUDA, "tv_branch_compress: launch failed: %s",
                        cudaGetErrorString(e));
  }
  return tv_check_launch("tv_branch_compress");
}

int tv_launch_branch(const tv_shape* s, void* rawK, void* rawV, void* c4K, void* c4V,
                     const int32_t* L, const void* treeK, const void* treeV,
                     const int32_t* parents, const float* g4, const float* g128, void* scrK4,
                     void* scrV4, void* scrK128, void* scrV128, int32_t* status,
                     cudaStream_t stream) {
  if (s->dtype == TV_BF16)
    return launch_branch_t<__nv_bfloat16>(s, rawK, rawV, c4K, c4V, L, treeK, treeV, parents, g4,
                                          g128, scrK4, scrV4, scrK128, scrV128, status, stream);
  return launch_branch_t<float>(s, rawK, rawV, c4K, c4V, L, treeK, treeV, parents, g4, g128,
                                scrK4, scrV4, scrK128, scrV128, status, stream);
}

int tv_launch_refresh(const tv_shape* s, const int32_t* parents, const int32_t* accept_len,
                      const int32_t* path,
                      const void* treeK, const void* treeV, const void* scrK4, const void* scrV4,
                      const void* scrK128, const void* scrV128, void* rawK, void* rawV,
                      void* c4K, void* c4V, void* c128K, void* c128V, int32_t* L,
                      int32_t* committed, int32_t* status, cudaStream_t stream) {
  const int es = s->dtype == TV_BF16 ? 2 : 4;
  const cudaError_t e = tv::launch_pdl(
      tv::refresh_kernel, dim3(s->B), dim3(256), 0, stream, tv::paging_of(s), s->D, s->d, es,
      s->comp_mask, s->raw_cap, s->c4_cap, s->c128_cap, (int)s->stage_chain, parents,
      accept_len, path, (const char*)treeK, (const char*)treeV, (const char*)scrK4,
      (const char*)scrV4, (const char*)scrK128, (const char*)scrV128, (char*)rawK, (char*)rawV,
      (char*)c4K, (char*)c4V, (char*)c128K, (char*)c128V, L, committed, status);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return tv_set_error(TV_ERR_CUDA, "tv_refresh_commit: launch failed: %s",
                        cudaGetErrorString(e));
  }
  return tv_check_launch("tv_refresh_commit");
}
