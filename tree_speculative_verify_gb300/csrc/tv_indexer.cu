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
// multiply-add (__fmul_rn / __fadd_rn).
//
// Two kernels:
//   score_kernel   one thread per (request, entry): the fp32 score into the workspace.
//   select_kernel  one 1024-thread CTA per request: an 8-bit-digit radix select (four passes over
//                  the request's scores, shared-memory histograms) finds the n_sel-th largest key;
//                  then every warp counts the entries above it and the ties in its contiguous
//                  index range (32 consecutive keys per step), the warps' counts place its kept
//                  entries, and it writes them in ascending order (ties: the lowest indices).
#include <mutex>

#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kSelThreads = 1024;
// Keys staged in shared memory when a request has at most this many C4 entries (160 KB): the four
// radix passes and the final pass then read shared memory instead of re-reading the scores.
constexpr int kSmemKeys = 40960;

// Order-preserving map of an fp32 score to an unsigned key (larger score -> larger key); -0 and
// +0 map to the same key.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void score_kernel(int B, int64_t c4_cap, int d_idx, const uint16_t* __restrict__ q_idx,
                             const uint16_t* __restrict__ k_idx, const int32_t* __restrict__ L,
                             float* __restrict__ score) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * c4_cap) return;
  const int b = (int)(t / c4_cap);
  const int64_t j = t - (int64_t)b * c4_cap;
  const int Lb = L[b];
  if (Lb < 0 || j >= Lb / 4) return;
  const uint4* q = reinterpret_cast<const uint4*>(q_idx + (int64_t)b * d_idx);
  const uint4* k = reinterpret_cast<const uint4*>(k_idx + t * d_idx);
  float s = 0.f;
  for (int c = 0; c < d_idx / 8; ++c) {
    const uint4 qa = q[c], ka = k[c];
    const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w}, kw[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {   // element 2h (low half) before 2h+1 (high half)
      s = __fadd_rn(s, __fmul_rn(bf16_lo(qw[h]), bf16_lo(kw[h])));
      s = __fadd_rn(s, __fmul_rn(bf16_hi(qw[h]), bf16_hi(kw[h])));
    }
  }
  score[t] = s;
}

// The radix select and the ordered write for one request of n4 keys.  kStaged: the keys are in
// shared memory (read four at a time in the histogram passes); otherwise each pass re-reads the
// scores.  The shared-memory arrays come from the kernel.
template <bool kStaged>
__device__ __forceinline__ void select_request(int n4, int n_sel, const uint32_t* keys_smem,
                                               const float* __restrict__ sc,
                                               int32_t* __restrict__ out, unsigned* hist,
                                               int* warp_gt, int* warp_eq, uint32_t* s_prefix,
                                               uint32_t* s_mask, int* s_krem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  auto key_at = [&](int j) -> uint32_t { return kStaged ? keys_smem[j] : score_key(sc[j]); };
  if (threadIdx.x == 0) {
    *s_prefix = 0u;
    *s_mask = 0u;
    *s_krem = n_sel;
  }
  __syncthreads();
  // radix select of the n_sel-th largest key, most significant digit first (shared-memory atomics
  // measured faster here than merging equal bins within a warp first)
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    const uint32_t prefix = *s_prefix, mask = *s_mask;
    auto count = [&](uint32_t key) {
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    };
    if (kStaged) {
      // four keys per 16-byte load; keys past n4 in the last vector are not counted
      const uint4* k4 = reinterpret_cast<const uint4*>(keys_smem);
      const int n16 = (n4 + 3) >> 2;
      for (int q = threadIdx.x; q < n16; q += blockDim.x) {
        const uint4 v = k4[q];
        const int j = 4 * q;
        count(v.x);
        if (j + 1 < n4) count(v.y);
        if (j + 2 < n4) count(v.z);
        if (j + 3 < n4) count(v.w);
      }
    } else {
      for (int j = threadIdx.x; j < n4; j += blockDim.x) count(score_key(sc[j]));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (descending); an inclusive scan over lanes gives the
      // count of keys in the digits above each lane's group
      const int krem = *s_krem;
      int c[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = (int)hist[255 - 8 * lane - q];
        sum += c[q];
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
        for (int q = 0; q < 8; ++q) {
          if (above + c[q] >= krem) {
            digit = 255 - 8 * lane - q;
            break;
          }
          above += c[q];
        }
        *s_krem = krem - above;
        *s_prefix = prefix | ((uint32_t)digit << shift);
        *s_mask = mask | (255u << shift);
      }
    }
    __syncthreads();
  }
  const uint32_t T = *s_prefix;   // key of the n_sel-th best entry
  const int need_eq = *s_krem;    // entries with key == T to keep: the lowest-indexed ones
  // warp w owns the contiguous index range [w * R, (w + 1) * R), read 32 consecutive keys at a
  // time: count, one scan over the warps, then write the kept entries in ascending order
  const int n_warps = blockDim.x >> 5;
  const int R = (n4 + n_warps - 1) / n_warps;
  const int lo = warp * R, hi = lo + R < n4 ? lo + R : n4;
  int gt = 0, eq = 0;
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < hi ? key_at(j) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, j < hi && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, j < hi && key == T));
  }
  if (lane == 0) {
    warp_gt[warp] = gt;
    warp_eq[warp] = eq;
  }
  __syncthreads();
  int gt_before = 0, eq_before = 0;
  for (int w = 0; w < warp; ++w) {
    gt_before += warp_gt[w];
    eq_before += warp_eq[w];
  }
  int pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
  int eq_seen = eq_before;
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < hi ? key_at(j) : 0u;
    const bool is_gt = j < hi && key > T, is_eq = j < hi && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, is_eq);
    const bool take = is_gt || (is_eq && eq_seen + __popc(eqm & lt_mask) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(tm & lt_mask)] = j;
    pos += __popc(tm);
    eq_seen += __popc(eqm);
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(int64_t c4_cap, int n_sel,
                                                             const int32_t* __restrict__ L,
                                                             const float* __restrict__ score,
                                                             int32_t* __restrict__ sel,
                                                             int32_t* status) {
  extern __shared__ __align__(16) uint32_t keys_smem[];
  __shared__ unsigned hist[256];
  __shared__ int warp_gt[32], warp_eq[32];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem;
  const int b = blockIdx.x;
  const int Lb = L[b];
  const int64_t n4 = Lb >= 0 ? Lb / 4 : -1;
  int32_t* out = sel + (int64_t)b * n_sel;
  if (n4 < n_sel || n4 > c4_cap) {
    if (threadIdx.x == 0) record_error(status, n4 > c4_cap ? TV_ERR_CAPACITY : TV_ERR_SELECTION);
    for (int i = threadIdx.x; i < n_sel; i += blockDim.x) out[i] = -1;
    return;
  }
  // n4 < 2^31: the shape check bounds B * c4_cap
  const float* sc = score + (int64_t)b * c4_cap;
  if (n4 <= kSmemKeys) {
#pragma unroll 8
    for (int j = threadIdx.x; j < (int)n4; j += blockDim.x) keys_smem[j] = score_key(sc[j]);
    if (threadIdx.x < (unsigned)((-n4) & 3)) keys_smem[n4 + threadIdx.x] = 0u;   // whole vectors
    select_request<true>((int)n4, n_sel, keys_smem, sc, out, hist, warp_gt, warp_eq, &s_prefix,
                         &s_mask, &s_krem);
  } else {
    select_request<false>((int)n4, n_sel, keys_smem, sc, out, hist, warp_gt, warp_eq, &s_prefix,
                          &s_mask, &s_krem);
  }
}

}  // namespace
}  // namespace tv

int tv_launch_indexer(const tv_shape* s, int d_idx, const void* q_idx, const void* k_idx,
                      const int32_t* L, int32_t* sel, void* workspace, int32_t* status,
                      cudaStream_t stream) {
  float* score = reinterpret_cast<float*>(workspace);
  const int64_t n = (int64_t)s->B * s->c4_cap;
  if (n > 0) {
    tv::score_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        s->B, s->c4_cap, d_idx, reinterpret_cast<const uint16_t*>(q_idx),
        reinterpret_cast<const uint16_t*>(k_idx), L, score);
    if (int rc = tv_check_launch("tv_indexer_topk (scores)")) return rc;
  }
  // shared memory for the staged keys, sized by the capacity (requests with more entries than
  // kSmemKeys read the scores from global memory instead)
  // (rounded up to whole 16-byte vectors: the histogram passes read four keys at a time)
  const int64_t staged = s->c4_cap < tv::kSmemKeys ? s->c4_cap : tv::kSmemKeys;
  const size_t smem = (size_t)((staged + 3) / 4 * 4) * sizeof(uint32_t);
  // once per device (a plain host call that also stays out of any stream being captured)
  static std::mutex attr_mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return tv_check_launch("tv_indexer_topk (device query)");
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(tv::select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(tv::kSmemKeys * sizeof(uint32_t))) != cudaSuccess)
        return tv_check_launch("tv_indexer_topk (shared-memory attribute)");
      attr_set[dev] = true;
    }
  }
  tv::select_kernel<<<s->B, tv::kSelThreads, smem, stream>>>(s->c4_cap, s->n_sel, L, score, sel,
                                                             status);
  return tv_check_launch("tv_indexer_topk (select)");
}
