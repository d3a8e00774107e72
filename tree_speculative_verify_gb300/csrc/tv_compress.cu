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
// evaluated in fp32 and stored in the cache dtype.  All three kernels call the same device
// routine with the same thread layout, so an entry computed in the scratch pad is bit-identical
// to the one prefill would compute for the same committed block.
#include <math.h>

#include "tv_common.cuh"

namespace tv {

constexpr int kCompressThreads = 512;
constexpr int kRedFloats = kCompressThreads * 8;   // group partials: blockDim * (16 B / 2 B)
static_assert(2 * kRedFloats * 4 <= 40 * 1024, "group partials must fit static shared memory");

// Vector load of N consecutive elements as fp32.
template <typename T, int N>
struct Vec;
template <>
struct Vec<__nv_bfloat16, 8> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      out[2 * k] = f.x;
      out[2 * k + 1] = f.y;
    }
  }
};
template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float* out) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    out[0] = f.x;
    out[1] = f.y;
    out[2] = f.z;
    out[3] = f.w;
  }
};
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

// One compressed entry from the m token rows rowK[t] / rowV[t] (t in position order).
// Whole-CTA routine (kCompressThreads threads); w_smem holds m floats, red 2*kRedFloats.
// Reduction orders depend only on the thread layout, which all callers share, so every caller
// computes bit-identical entries for the same block.  Loads are 16-byte vectors and the token loops are unrolled so that
// many loads are in flight: a 128-token block is 256 KB of K and V.
template <typename T>
__device__ void gated_block_sum(const T* const* rowK, const T* const* rowV, int m, int d,
                                const float* __restrict__ g, T* outK, T* outV, float* w_smem,
                                float* red) {
  constexpr int VW = VecWidth<T>::n;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  // 1. gate logits z_t = K_t . g: warp per token (token t on warp t % nwarps), lanes over 16-byte
  //    vectors of the row (lane l: dims l*VW + 32*VW*k); each warp loads a batch of its tokens
  //    before using any, and keeps its slice of g in registers
  constexpr int KVMAX = 512 / (32 * VW);   // vectors per lane at the largest head dim
  constexpr int U1 = 8 / KVMAX;            // tokens per batch
  float gr[KVMAX][VW];
#pragma unroll
  for (int k = 0; k < KVMAX; ++k) {
    const int i = lane * VW + 32 * VW * k;
#pragma unroll
    for (int e = 0; e < VW; ++e) gr[k][e] = i < d ? g[i + e] : 0.f;
  }
  for (int t0 = warp; t0 < m; t0 += nwarps * U1) {
    uint4 raw[U1][KVMAX];
#pragma unroll
    for (int u = 0; u < U1; ++u) {
      const int t = t0 + u * nwarps;
#pragma unroll
      for (int k = 0; k < KVMAX; ++k) {
        const int i = lane * VW + 32 * VW * k;
        raw[u][k] = (t < m && i < d) ? ld16(rowK[t] + i) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U1; ++u) {
      const int t = t0 + u * nwarps;
      if (t >= m) break;   // warp-uniform
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < KVMAX; ++k) {
        if (lane * VW + 32 * VW * k >= d) break;
        float kv[VW];
        cvt16(raw[u][k], (T*)nullptr, kv);
#pragma unroll
        for (int e = 0; e < VW; ++e) acc = fmaf(kv[e], gr[k][e], acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) w_smem[t] = acc;
    }
  }
  __syncthreads();
  // 2. softmax over the m logits
  if (warp == 0) {
    float mx = -INFINITY;
    for (int t = lane; t < m; t += 32) mx = fmaxf(mx, w_smem[t]);
    mx = warp_max(mx);
    float s = 0.f;
    for (int t = lane; t < m; t += 32) {
      const float e = expf(w_smem[t] - mx);
      w_smem[t] = e;
      s += e;
    }
    s = warp_sum(s);
    const float inv = 1.f / s;
    __syncwarp();
    for (int t = lane; t < m; t += 32) w_smem[t] *= inv;
  }
  __syncthreads();
  // 3. weighted sums: the threads form G groups of d/VW; thread (group gi, slot li) owns dims
  //    li*VW .. li*VW+VW-1 and the tokens gi, gi+G, ...; the group partials are then added in
  //    group order (a fixed order, so the result does not depend on timing)
  const int per_group = d / VW;
  int G = blockDim.x / per_group;
  if (G > m) G = m;
  const int gi = tid / per_group, li = tid % per_group;
  if (gi < G) {
    const int i = li * VW;
    float ak[VW], av[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) ak[e] = av[e] = 0.f;
    constexpr int U3 = 4;   // tokens whose K and V vectors are loaded before use
    for (int t0 = gi; t0 < m; t0 += G * U3) {
      uint4 rk[U3], rv[U3];
#pragma unroll
      for (int u = 0; u < U3; ++u) {
        const int t = t0 + u * G;
        rk[u] = t < m ? ld16(rowK[t] + i) : make_uint4(0u, 0u, 0u, 0u);
        rv[u] = t < m ? ld16(rowV[t] + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U3; ++u) {
        const int t = t0 + u * G;
        if (t >= m) break;
        const float w = w_smem[t];
        float kv[VW], vv[VW];
        cvt16(rk[u], (T*)nullptr, kv);
        cvt16(rv[u], (T*)nullptr, vv);
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          ak[e] = fmaf(w, kv[e], ak[e]);
          av[e] = fmaf(w, vv[e], av[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      red[(gi * d + i + e) * 2] = ak[e];
      red[(gi * d + i + e) * 2 + 1] = av[e];
    }
  }
  __syncthreads();
  for (int i = tid; i < d; i += blockDim.x) {
    float ak = 0.f, av = 0.f;
    for (int k = 0; k < G; ++k) {
      ak += red[(k * d + i) * 2];
      av += red[(k * d + i) * 2 + 1];
    }
    store_f(outK + i, ak);
    store_f(outV + i, av);
  }
}

// ---- prefill: every complete block of the committed prefix ---------------------------------
// grid.x: entry index (strided), grid.y: request.
template <typename T>
__global__ void __launch_bounds__(kCompressThreads, 2) prefill_kernel(Paging pg, int m, int d, int64_t raw_cap, int64_t cap_m,
                               const T* __restrict__ rawK, const T* __restrict__ rawV,
                               const int32_t* __restrict__ L, const float* __restrict__ g,
                               T* __restrict__ CK, T* __restrict__ CV, int32_t* status) {
  __shared__ const T* rowK[128];
  __shared__ const T* rowV[128];
  __shared__ float w[128];
  __shared__ float red[2 * kRedFloats];
  const int b = blockIdx.y;
  const int Lb = L[b];
  if (Lb < 0 || Lb > raw_cap || (int64_t)(Lb / m) > cap_m) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, TV_ERR_CAPACITY);
    return;
  }
  const int n = Lb / m;
  for (int j = blockIdx.x; j < n; j += gridDim.x) {
    for (int t = threadIdx.x; t < m; t += blockDim.x) {
      const int64_t row = layer_row(pg, b, (int64_t)j * m + t, raw_cap, 1, status);
      rowK[t] = rawK + row * d;
      rowV[t] = rawV + row * d;
    }
    __syncthreads();
    const int64_t out = layer_row(pg, b, j, cap_m, m, status) * d;
    gated_block_sum<T>(rowK, rowV, m, d, g, CK + out, CV + out, w, red);
    __syncthreads();
  }
}

// ---- scratch pad: entries of blocks closed by tree nodes ------------------------------------
// grid: (D, B, active compressors).  Row v of the scratch pad of compressor m is written either
// with the block that v's token closes (positions pos_v - m + 1 .. pos_v of prefix + path(v)) or
// with zeros.
template <typename T>
__global__ void __launch_bounds__(kCompressThreads, 2) branch_kernel(Paging pg, int D, int d, int comp_mask, int64_t raw_cap,
                              T* rawK, T* rawV, int stage, int64_t c4_cap, T* c4K, T* c4V,
                              const int32_t* __restrict__ L, const T* __restrict__ treeK,
                              const T* __restrict__ treeV, const int32_t* __restrict__ parents,
                              const float* __restrict__ g4, const float* __restrict__ g128,
                              T* scrK4, T* scrV4, T* scrK128, T* scrV128, int32_t* status) {
  __shared__ const T* rowK[128];
  __shared__ const T* rowV[128];
  __shared__ float w[128];
  __shared__ float red[2 * kRedFloats];
  __shared__ int path[kMaxD];   // path[k] = ancestor of v at depth k
  __shared__ int s_par[kMaxD];
  __shared__ int s_depth;
  __shared__ int s_ok;
  __shared__ int s_cached;   // v lies on the round's cached chain
  const int v = blockIdx.x;
  const int b = blockIdx.y;
  int which = blockIdx.z;  // index among active compressors
  int m;
  if ((comp_mask & TV_COMP_C4) && which == 0) {
    m = 4;
  } else {
    m = 128;
  }
  const float* g = (m == 4) ? g4 : g128;
  T* outK = (m == 4) ? scrK4 : scrK128;
  T* outV = (m == 4) ? scrV4 : scrV128;
  const int64_t out = ((int64_t)b * D + v) * d;
  const int Lb = L[b];
  const int32_t* par = parents + (int64_t)b * D;

  // the request's parent array in one round trip; the chain walk then runs in shared memory
  for (int u = threadIdx.x; u < D; u += blockDim.x) s_par[u] = par[u];
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = (Lb >= 0 && Lb <= raw_cap) ? 1 : 0;
    int dep = 0;
    int u = v;
    int chain[kMaxD];
    for (int step = 0; step < D && ok; ++step) {
      chain[dep] = u;
      if (u == 0) break;
      const int p = s_par[u];
      if (p < 0 || p >= u) { ok = 0; break; }
      u = p;
      ++dep;
    }
    if (ok && s_par[0] != -1) ok = 0;
    int cached = 0;
    if (ok) {
      for (int k = 0; k <= dep; ++k) path[k] = chain[dep - k];
      // cached chain: every step goes to the lowest-numbered child of the previous node
      cached = 1;
      for (int k = 0; k < dep && cached; ++k)
        for (int u = 1; u < path[k + 1]; ++u)
          if (s_par[u] == path[k]) {
            cached = 0;
            break;
          }
    } else {
      record_error(status, (Lb < 0 || Lb > raw_cap) ? TV_ERR_CAPACITY : TV_ERR_BAD_TREE);
    }
    s_depth = dep;
    s_ok = ok;
    s_cached = cached;
  }
  __syncthreads();
  const int pos = Lb + s_depth;
  const bool closes = s_ok && ((pos + 1) % m == 0);
  // staging (refresh skip): the cached chain's raw row goes to its final place past L now, once
  // per node (by the CTA of the first active compressor)
  const bool stage_here = stage && s_ok && s_cached;
  if (stage_here && which == 0 && pos < raw_cap) {
    const int64_t dst = layer_row(pg, b, pos, raw_cap, 1, status) * d;
    const int64_t src = ((int64_t)b * D + v) * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
      rawK[dst + i] = treeK[src + i];
      rawV[dst + i] = treeV[src + i];
    }
  }
  if (!closes) {
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
      store_f(outK + out + i, 0.f);
      store_f(outV + out + i, 0.f);
    }
    return;
  }
  for (int t = threadIdx.x; t < m; t += blockDim.x) {
    const int p = pos + 1 - m + t;   // >= 0 because pos + 1 is a positive multiple of m
    if (p < Lb) {
      const int64_t row = layer_row(pg, b, p, raw_cap, 1, status);
      rowK[t] = rawK + row * d;
      rowV[t] = rawV + row * d;
    } else {
      const int64_t row = (int64_t)b * D + path[p - Lb];
      rowK[t] = treeK + row * d;
      rowV[t] = treeV + row * d;
    }
  }
  __syncthreads();
  gated_block_sum<T>(rowK, rowV, m, d, g, outK + out, outV + out, w, red);
  // C4 refreshes promptly: a cached-chain node's C4 entry is also staged in its final place
  // (C128 entries wait for the accepted path)
  const int64_t entry = (pos + 1) / 4 - 1;
  if (stage_here && m == 4 && entry < c4_cap) {
    __syncthreads();   // the entry this CTA just wrote is visible to all its threads
    const int64_t dst = layer_row(pg, b, entry, c4_cap, 4, status) * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
      c4K[dst + i] = outK[out + i];
      c4V[dst + i] = outV[out + i];
    }
  }
}

// ---- refresh: commit the accepted path --------------------------------------------------------
// One CTA per request.  Copies the accepted tokens' K/V into the raw rows L .. L+n-1 and the
// scratch rows of accepted nodes that close a block into the persistent entries (all rows in
// parallel: each 16-byte chunk of each row is one thread's job), then advances L.
__global__ void refresh_kernel(Paging pg, int D, int d, int es, int comp_mask, int64_t raw_cap,
                               int64_t c4_cap, int64_t c128_cap, int stage,
                               const int32_t* __restrict__ parents,
                               const int32_t* __restrict__ accept_len,
                               const int32_t* __restrict__ path_all, const char* treeK,
                               const char* treeV, const char* scrK4, const char* scrV4,
                               const char* scrK128, const char* scrV128, char* rawK, char* rawV,
                               char* c4K, char* c4V, char* c128K, char* c128V, int32_t* L,
                               int32_t* committed, int32_t* status) {
  constexpr int kMaxJobs = 3 * kMaxD;   // raw rows + C4 entries + C128 entries
  __shared__ int s_ok;
  __shared__ int s_L;
  __shared__ int s_n;
  __shared__ int s_jobs;
  __shared__ const char* s_srcK[kMaxJobs];
  __shared__ const char* s_srcV[kMaxJobs];
  __shared__ char* s_dstK[kMaxJobs];
  __shared__ char* s_dstV[kMaxJobs];
  const int b = blockIdx.x;
  const int64_t row_bytes = (int64_t)d * es;
  const int32_t* path = path_all + (int64_t)b * D;
  if (threadIdx.x == 0) {
    const int Lb = L[b];
    const int n = accept_len[b];
    int ok = 1, code = 0;
    if (n < 1 || n > D || Lb < 0) { ok = 0; code = TV_ERR_ARG; }
    for (int i = 0; ok && i < n; ++i)
      if (path[i] < 0 || path[i] >= D) { ok = 0; code = TV_ERR_ARG; }
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
      const int32_t* par = parents + (int64_t)b * D;
      int c = 0;
      while (staged < n && path[staged] == c) {
        ++staged;
        int next = -1;
        for (int u = c + 1; u < D; ++u)
          if (par[u] == c) {
            next = u;
            break;
          }
        if (next < 0) break;
        c = next;
      }
    }
    int jobs = 0;
    if (ok) {
      for (int i = 0; i < n; ++i) {
        const int64_t src = ((int64_t)b * D + path[i]) * row_bytes;
        const bool on_chain = i < staged;
        if (!on_chain) {
          const int64_t dst = layer_row(pg, b, Lb + i, raw_cap, 1, status) * row_bytes;
          s_srcK[jobs] = treeK + src;
          s_srcV[jobs] = treeV + src;
          s_dstK[jobs] = rawK + dst;
          s_dstV[jobs] = rawV + dst;
          ++jobs;
        }
        const int e = Lb + i;
        if ((comp_mask & TV_COMP_C4) && ((e + 1) & 3) == 0 && !on_chain) {
          const int64_t cd = layer_row(pg, b, (e + 1) / 4 - 1, c4_cap, 4, status) * row_bytes;
          s_srcK[jobs] = scrK4 + src;
          s_srcV[jobs] = scrV4 + src;
          s_dstK[jobs] = c4K + cd;
          s_dstV[jobs] = c4V + cd;
          ++jobs;
        }
        if ((comp_mask & TV_COMP_C128) && ((e + 1) & 127) == 0) {
          const int64_t cd = layer_row(pg, b, (e + 1) / 128 - 1, c128_cap, 128, status) * row_bytes;
          s_srcK[jobs] = scrK128 + src;
          s_srcV[jobs] = scrV128 + src;
          s_dstK[jobs] = c128K + cd;
          s_dstV[jobs] = c128V + cd;
          ++jobs;
        }
      }
    }
    s_ok = ok;
    s_L = Lb;
    s_n = n;
    s_jobs = jobs;
  }
  __syncthreads();
  int32_t* cpos = committed + (int64_t)b * D;
  if (!s_ok) {
    for (int i = threadIdx.x; i < D; i += blockDim.x) cpos[i] = -1;
    return;
  }
  const int chunks = (int)(row_bytes / 16);
  const int total = s_jobs * chunks;
  for (int k = threadIdx.x; k < total; k += blockDim.x) {
    const int j = k / chunks, c = k - j * chunks;
    reinterpret_cast<uint4*>(s_dstK[j])[c] = reinterpret_cast<const uint4*>(s_srcK[j])[c];
    reinterpret_cast<uint4*>(s_dstV[j])[c] = reinterpret_cast<const uint4*>(s_srcV[j])[c];
  }
  for (int i = threadIdx.x; i < D; i += blockDim.x) cpos[i] = i < s_n ? s_L + i : -1;
  __syncthreads();
  if (threadIdx.x == 0) L[b] = s_L + s_n;
}

}  // namespace tv

// ---- launchers --------------------------------------------------------------------------------
template <typename T>
static int launch_prefill_t(const tv_shape* s, const void* rawK, const void* rawV,
                            const int32_t* L, const float* g4, const float* g128, void* c4K,
                            void* c4V, void* c128K, void* c128V, int32_t* status,
                            cudaStream_t stream) {
  const int d = s->d;
  if (s->comp_mask & TV_COMP_C4) {
    const int64_t cap = s->c4_cap;
    const unsigned gx = (unsigned)(cap < 1 ? 1 : (cap > (1 << 20) ? (1 << 20) : cap));
    tv::prefill_kernel<T><<<dim3(gx, s->B), tv::kCompressThreads, 0, stream>>>(
        tv::paging_of(s), 4, d, s->raw_cap, cap, (const T*)rawK, (const T*)rawV, L, g4, (T*)c4K, (T*)c4V, status);
    if (int rc = tv_check_launch("tv_prefill_compress (C4)")) return rc;
  }
  if (s->comp_mask & TV_COMP_C128) {
    const int64_t cap = s->c128_cap;
    const unsigned gx = (unsigned)(cap < 1 ? 1 : (cap > (1 << 20) ? (1 << 20) : cap));
    tv::prefill_kernel<T><<<dim3(gx, s->B), tv::kCompressThreads, 0, stream>>>(
        tv::paging_of(s), 128, d, s->raw_cap, cap, (const T*)rawK, (const T*)rawV, L, g128, (T*)c128K,
        (T*)c128V, status);
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

int tv_launch_branch(const tv_shape* s, void* rawK, void* rawV, void* c4K, void* c4V, const int32_t* L,
                     const void* treeK, const void* treeV, const int32_t* parents,
                     const float* g4, const float* g128, void* scrK4, void* scrV4,
                     void* scrK128, void* scrV128, int32_t* status, cudaStream_t stream) {
  const int n_comp = ((s->comp_mask & TV_COMP_C4) ? 1 : 0) + ((s->comp_mask & TV_COMP_C128) ? 1 : 0);
  const dim3 grid(s->D, s->B, n_comp);
  if (s->dtype == TV_BF16) {
    using T = __nv_bfloat16;
    tv::branch_kernel<T><<<grid, tv::kCompressThreads, 0, stream>>>(
        tv::paging_of(s), s->D, s->d, s->comp_mask, s->raw_cap, (T*)rawK, (T*)rawV,
        s->stage_chain, s->c4_cap, (T*)c4K, (T*)c4V, L,
        (const T*)treeK, (const T*)treeV, parents, g4, g128, (T*)scrK4, (T*)scrV4,
        (T*)scrK128, (T*)scrV128, status);
  } else {
    using T = float;
    tv::branch_kernel<T><<<grid, tv::kCompressThreads, 0, stream>>>(
        tv::paging_of(s), s->D, s->d, s->comp_mask, s->raw_cap, (T*)rawK, (T*)rawV,
        s->stage_chain, s->c4_cap, (T*)c4K, (T*)c4V, L,
        (const T*)treeK, (const T*)treeV, parents, g4, g128, (T*)scrK4, (T*)scrV4,
        (T*)scrK128, (T*)scrV128, status);
  }
  return tv_check_launch("tv_branch_compress");
}

int tv_launch_refresh(const tv_shape* s, const int32_t* parents, const int32_t* accept_len,
                      const int32_t* path,
                      const void* treeK, const void* treeV, const void* scrK4, const void* scrV4,
                      const void* scrK128, const void* scrV128, void* rawK, void* rawV,
                      void* c4K, void* c4V, void* c128K, void* c128V, int32_t* L,
                      int32_t* committed, int32_t* status, cudaStream_t stream) {
  const int es = s->dtype == TV_BF16 ? 2 : 4;
  tv::refresh_kernel<<<s->B, 256, 0, stream>>>(
      tv::paging_of(s), s->D, s->d, es, s->comp_mask, s->raw_cap, s->c4_cap, s->c128_cap,
      s->stage_chain, parents, accept_len, path,
      (const char*)treeK, (const char*)treeV, (const char*)scrK4, (const char*)scrV4,
      (const char*)scrK128, (const char*)scrV128, (char*)rawK, (char*)rawV, (char*)c4K,
      (char*)c4V, (char*)c128K, (char*)c128V, L, committed, status);
  return tv_check_launch("tv_refresh_commit");
}
