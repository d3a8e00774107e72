// Indexer top-k: the selected C4 entries of the sparse prefix attention, chosen on the device.
//
// "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference" §2.2:
// CSA is compressed *sparse* attention -- a query reads a selected subset of the compressed C4
// entries.  The report gives no selection rule; the long-context workload's stand-in scores entry
// j of request b as q_idx[b] . k_idx[b][j] (dimension d_idx) and keeps the n_sel best, equal
// scores going to the lower index, listed in ascending order.
//
// Precision: the scores decide an integer selection, so the kernel fixes them exactly: bf16
// inputs; each product rounded to fp32 (exact for bf16 operands) and added to the running fp32
// sum in index order i = 0 .. d_idx-1 with one round-to-nearest-even per addition and no fused
// multiply-add (products by round-to-nearest packed fp32 multiplies, sums by __fadd_rn).
//
// Two kernels:
//   1. score_kernel, over every SM: CTA (t, b) forms the scores of one tile of request b's C4
//      entries from a coalesced copy of their indexer keys in shared memory (one thread per
//      entry) and writes them to the workspace;
//   select_kernel, a cluster of eight CTAs per request, CTA r owning the request's r-th contiguous
//   eighth of the entries (their order-preserving keys staged in shared memory):
//   2. an 8-bit-digit radix select of the n_sel-th largest key over the whole request: per pass
//      every CTA counts its keys into a shared-memory histogram and stores it into every rank's
//      shared memory (distributed shared memory), and after one cluster barrier each CTA adds the
//      eight histograms up locally and picks the same digit;
//   3. the kept entries in ascending order: every warp counts the entries above the threshold and
//      the ties in its contiguous index range, CTAs in rank order (each pushes its counts to the
//      higher ranks before one last cluster barrier) and warps in index order place them (ties:
//      the lowest indices), and each warp writes its own.
//   The select kernel is a programmatic dependent of the score kernel: its launch overlaps the
//   scoring, and it waits for the scores before it reads them.
#include <cooperative_groups.h>

#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kTopkRanks = 8;        // CTAs per request (one cluster)
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
// Keys a select CTA stages in shared memory (24 KB): its share of a request of up to 8 x 6144 C4
// entries.  A larger share reads its scores from the workspace in each pass.
constexpr int kStageKeys = 6144;
constexpr int kMaxIdxVec = 32;       // 16-byte vectors of the indexer query (d_idx <= 256)
constexpr int kScoreThreads = 256;
constexpr int kScoreTileBytes = 32768;   // indexer keys of one score CTA

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Order-preserving map of an fp32 score to an unsigned key (larger score -> larger key); -0 and
// +0 map to the same key.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The products a0 b0 and a1 b1 by one packed fp32 multiply, each rounded to nearest (as __fmul_rn).
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float& p0,
                                        float& p1) {
  uint64_t a, b, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(d));
}

// Rows per score CTA: kScoreTileBytes of indexer keys of dimension d_idx = 8 nvec.
__host__ __device__ __forceinline__ int score_rows(int nvec) { return kScoreTileBytes / (16 * nvec); }

// grid (ceil(c4_cap / score_rows), B).  CTA (t, b) scores entries t RT .. t RT + RT - 1 of request
// b (those below L[b] / 4) into score_ws[b][j].  A request whose L is negative or past the
// capacity is skipped (the select kernel reports it).
__global__ void __launch_bounds__(kScoreThreads, 4)
    score_kernel(int64_t c4_cap, int d_idx, const uint16_t* __restrict__ q_idx,
                 const uint16_t* __restrict__ k_idx, const int32_t* __restrict__ L,
                 float* __restrict__ score_ws) {
  pdl_launch_dependents();   // the select kernel may be placed; it waits for these scores
  __shared__ uint4 ktile[kScoreTileBytes / 16];
  __shared__ float4 qf[2 * kMaxIdxVec];   // the query in fp32 (exact)
  const int b = blockIdx.y, tid = threadIdx.x;
  const int nvec = d_idx / 8, RT = score_rows(nvec);
  const int64_t n4 = L[b] >= 0 ? L[b] / 4 : -1;
  const int64_t j0 = (int64_t)blockIdx.x * RT;
  if (n4 < 0 || n4 > c4_cap || j0 >= n4) return;
  const int rows = (int)(n4 - j0 < RT ? n4 - j0 : RT);
  // the tile's rows as contiguous 16-byte chunks; chunk c of row r sits at r * nvec + (c ^ (r & 7))
  // when nvec is a multiple of 8, so the threads' row-wise reads do not collide on banks
  const int swz = (nvec & 7) == 0 ? 7 : 0;
  const uint4* src = reinterpret_cast<const uint4*>(k_idx + ((int64_t)b * c4_cap + j0) * d_idx);
  for (int i = tid; i < rows * nvec; i += blockDim.x) {
    const int r = i / nvec, c = i - r * nvec;
    cp_async16(ktile + r * nvec + (c ^ (r & swz)), src + i);
  }
  if (tid < nvec) {
    const uint4 qa = reinterpret_cast<const uint4*>(q_idx + (int64_t)b * d_idx)[tid];
    qf[2 * tid] = make_float4(bf16_lo(qa.x), bf16_hi(qa.x), bf16_lo(qa.y), bf16_hi(qa.y));
    qf[2 * tid + 1] = make_float4(bf16_lo(qa.z), bf16_hi(qa.z), bf16_lo(qa.w), bf16_hi(qa.w));
  }
  cp_async_wait_all();
  __syncthreads();
  float* sc = score_ws + (int64_t)b * c4_cap + j0;
  for (int r = tid; r < rows; r += blockDim.x) {
    float sacc = 0.f;
    for (int c = 0; c < nvec; ++c) {
      const uint4 ka = ktile[r * nvec + (c ^ (r & swz))];
      const float4 qa = qf[2 * c], qb = qf[2 * c + 1];
      const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
      const uint32_t kw[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {   // element 2h (low half) before 2h+1 (high half)
        float p0, p1;
        mul2_rn(qv[2 * h], qv[2 * h + 1], bf16_lo(kw[h]), bf16_hi(kw[h]), p0, p1);
        sacc = __fadd_rn(sacc, p0);
        sacc = __fadd_rn(sacc, p1);
      }
    }
    sc[r] = sacc;
  }
}

// grid (8, B), clusters of 8 along x; launched as a programmatic dependent of score_kernel.
// score_ws: [B][c4_cap] fp32 scores.
__global__ void __cluster_dims__(kTopkRanks, 1, 1) __launch_bounds__(kTopkThreads)
    select_kernel(int64_t c4_cap, int n_sel, const int32_t* __restrict__ L,
                  const float* __restrict__ score_ws, int32_t* __restrict__ sel,
                  int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) uint32_t keys[];   // this CTA's keys (when staged)
  __shared__ unsigned hist[256];      // this CTA's histogram of the pass
  // every rank's histogram of the pass, pushed here by that rank; by pass parity, so that a rank
  // that runs ahead never overwrites a histogram this CTA still adds up
  __shared__ unsigned hall[2][kTopkRanks][256];
  __shared__ unsigned ghist[256];     // the pass's histogram of the whole request
  __shared__ int warp_gt[kTopkWarps], warp_eq[kTopkWarps];
  __shared__ int2 before[kTopkRanks];  // (above, equal) counts of the lower ranks, pushed by them
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem;
  pdl_wait();   // the scores are complete and visible
  const int b = blockIdx.y;
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int Lb = L[b];
  const int64_t n4l = Lb >= 0 ? Lb / 4 : -1;
  int32_t* out = sel + (int64_t)b * n_sel;
  if (n4l < n_sel || n4l > c4_cap) {   // uniform over the cluster
    if (rank == 0) {
      if (tid == 0) record_error(status, n4l > c4_cap ? TV_ERR_CAPACITY : TV_ERR_SELECTION);
      for (int i = tid; i < n_sel; i += blockDim.x) out[i] = -1;
    }
    return;
  }
  const int n4 = (int)n4l;   // < 2^31: the shape check bounds B * c4_cap
  const int per = (n4 + kTopkRanks - 1) / kTopkRanks;
  const int lo = min(n4, rank * per), hi = min(n4, lo + per), n = hi - lo;
  const bool staged = per <= kStageKeys;   // uniform over the cluster
  const float* sc = score_ws + (int64_t)b * c4_cap;
  if (tid == 0) {
    s_prefix = 0u;
    s_mask = 0u;
    s_krem = n_sel;
  }
  if (tid < 256) hist[tid] = 0u;
  // 1. this CTA's keys (the padding up to whole 16-byte vectors: key 0, never counted)
  if (staged) {   // all of a thread's loads in flight at once
    constexpr int kPerThread = (kStageKeys + kTopkThreads - 1) / kTopkThreads;
    float v[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int j = lo + tid + k * kTopkThreads;
      v[k] = j < hi ? sc[j] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int j = lo + tid + k * kTopkThreads;
      if (j < hi) keys[j - lo] = score_key(v[k]);
    }
    if (tid < ((-n) & 3)) keys[n + tid] = 0u;
  }
  __syncthreads();
  auto key_at = [&](int j) -> uint32_t { return staged ? keys[j - lo] : score_key(sc[j]); };
  // 2. radix select of the n_sel-th largest key of the request, most significant digit first
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, par = pass & 1;
    const uint32_t prefix = s_prefix, mask = s_mask;
    auto count = [&](uint32_t key) {
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    };
    if (staged) {
      const uint4* k4 = reinterpret_cast<const uint4*>(keys);
      for (int v = tid; v < (n + 3) >> 2; v += blockDim.x) {
        const uint4 x = k4[v];
        const int j = 4 * v;
        count(x.x);
        if (j + 1 < n) count(x.y);
        if (j + 2 < n) count(x.z);
        if (j + 3 < n) count(x.w);
      }
    } else {
      for (int j = lo + tid; j < hi; j += blockDim.x) count(score_key(sc[j]));
    }
    __syncthreads();
    if (tid < 256) {   // bin tid to every rank (stores, none awaited), then cleared for the next pass
      const unsigned h = hist[tid];
#pragma unroll
      for (int r = 0; r < kTopkRanks; ++r) *cl.map_shared_rank(&hall[par][rank][tid], r) = h;
      hist[tid] = 0u;
    }
    cl.sync();   // every rank's histogram of this pass has arrived
    if (tid < 256) {   // bin tid summed over the ranks, in rank order
      unsigned t = 0u;
#pragma unroll
      for (int r = 0; r < kTopkRanks; ++r) t += hall[par][r][tid];
      ghist[tid] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (descending); an inclusive scan over lanes gives the
      // count of keys in the digits above each lane's group
      const int krem = s_krem;
      int c[8], sum = 0;
#pragma unroll
      for (int qd = 0; qd < 8; ++qd) {
        c[qd] = (int)ghist[255 - 8 * lane - qd];
        sum += c[qd];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < krem && incl >= krem);
      if (lane == __ffs(hit) - 1) {
        int above = excl, digit = 0;
        for (int qd = 0; qd < 8; ++qd) {
          if (above + c[qd] >= krem) {
            digit = 255 - 8 * lane - qd;
            break;
          }
          above += c[qd];
        }
        s_krem = krem - above;
        s_prefix = prefix | ((uint32_t)digit << shift);
        s_mask = mask | (255u << shift);
      }
    }
    __syncthreads();
  }
  const uint32_t T = s_prefix;   // key of the n_sel-th best entry
  const int need_eq = s_krem;    // entries with key == T to keep: the lowest-indexed ones
  // 3. warp w owns the contiguous range [lo + w R, lo + (w + 1) R) of this CTA's entries, read 32
  //    consecutive keys at a time: counts, placed over the CTAs (rank order) and the warps
  const int R = (n + kTopkWarps - 1) / kTopkWarps;
  const int wlo = lo + min(n, warp * R), whi = lo + min(n, warp * R + R);
  int gt = 0, eq = 0;
  for (int j0 = wlo; j0 < whi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < whi ? key_at(j) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, j < whi && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, j < whi && key == T));
  }
  if (lane == 0) {
    warp_gt[warp] = gt;
    warp_eq[warp] = eq;
  }
  __syncthreads();
  if (tid == 0) {   // this CTA's counts to every higher rank
    int a = 0, e = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      a += warp_gt[w];
      e += warp_eq[w];
    }
    for (int r = rank + 1; r < kTopkRanks; ++r)
      *cl.map_shared_rank(&before[rank], r) = make_int2(a, e);
  }
  cl.sync();   // every lower rank's counts have arrived (the last access to a peer's memory)
  int gt_before = 0, eq_before = 0;
  for (int r = 0; r < rank; ++r) {
    gt_before += before[r].x;
    eq_before += before[r].y;
  }
  for (int w = 0; w < warp; ++w) {
    gt_before += warp_gt[w];
    eq_before += warp_eq[w];
  }
  int pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
  int eq_seen = eq_before;
  for (int j0 = wlo; j0 < whi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < whi ? key_at(j) : 0u;
    const bool is_gt = j < whi && key > T, is_eq = j < whi && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
    const bool take = is_gt || (is_eq && eq_seen + __popc(eqm & lt_mask) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(tm & lt_mask)] = j;
    pos += __popc(tm);
    eq_seen += __popc(eqm);
  }
}

}  // namespace
}  // namespace tv

int tv_launch_indexer(const tv_shape* s, int d_idx, const void* q_idx, const void* k_idx,
                      const int32_t* L, int32_t* sel, void* workspace, int32_t* status,
                      cudaStream_t stream) {
  float* score_ws = reinterpret_cast<float*>(workspace);
  const int RT = tv::score_rows(d_idx / 8);
  const int64_t tiles = (s->c4_cap + RT - 1) / RT;
  if (tiles > 0) {
    tv::score_kernel<<<dim3((unsigned)tiles, s->B), tv::kScoreThreads, 0, stream>>>(
        s->c4_cap, d_idx, reinterpret_cast<const uint16_t*>(q_idx),
        reinterpret_cast<const uint16_t*>(k_idx), L, score_ws);
    if (int rc = tv_check_launch("tv_indexer_topk (scores)")) return rc;
  }
  // shared memory for the staged keys, sized by the capacity (rounded up to whole 16-byte vectors)
  const int64_t per = (s->c4_cap + tv::kTopkRanks - 1) / tv::kTopkRanks;
  const int64_t staged = per <= tv::kStageKeys ? per : 0;
  const size_t smem = (size_t)((staged + 3) / 4 * 4) * sizeof(uint32_t);
  tv::launch_pdl(tv::select_kernel, dim3(tv::kTopkRanks, s->B), dim3(tv::kTopkThreads), smem,
                 stream, (int64_t)s->c4_cap, (int)s->n_sel, L, (const float*)score_ws, sel,
                 status);
  return tv_check_launch("tv_indexer_topk");
}
