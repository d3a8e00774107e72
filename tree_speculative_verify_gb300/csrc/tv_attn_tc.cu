// Branch-aware causal tree-verify attention on the 5th-generation tensor cores (tcgen05), bf16,
// head dim 512, for sm_103a.
//
// "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference":
// §3.1 every candidate attends to the accepted context plus its own ancestors; §3.2 / §4.2 blocks
// closed inside the tree are seen only through the branch's scratch-pad entries.  With H query
// heads sharing one K/V head, all D*H query rows of a request read the same compressed prefix, so
// the prefix part is a dense (D*H) x entries x 512 contraction -- tensor-core work.
//
// Work item: a CTA pair (a cluster of 2) for request b, two consecutive 128-row tiles of the
// request's D*H query rows (node-major), one half of the value dimension (256 of 512 columns of
// O) and one chunk of the request's KV tiles.  The pair runs cta_group::2 MMAs (M = 256): the
// leader issues them, each CTA's tensor core works on its own 128 rows, and every K / V tile is
// split between the two CTAs' shared memory, so each SM ingests half of it.  (The rate at which
// TMA fills one SM's shared memory, not the tensor cores, bounds a one-CTA design here.)  The two
// value halves of a row tile compute the same S = Q K^T: a 128-row, 512-column fp32 O would fill
// all 512 TMEM columns and leave none for S.
//
// KV tiles (<= 128 entries each), in order: persistent C4 entries, persistent C128 entries, the raw
// tail (positions t0 .. L-1), and one "extra" tile of 32 entries: the tree tokens (0..7), the C4
// scratch rows (8..15), the C128 scratch rows (16..23) and 8 zero rows.  Shared tiles are visible
// to every row; raw and extra tiles are filtered per tree node with the plan (raw_lo, ancestor
// mask, scratch visibility) inside the softmax warps.
//
// Warp roles (352 threads per CTA):
//   warp 0      TMA producer: Q once (8 boxes of 128 x 64, completing on the leader's barrier like
//               every other copy of the pair); then, through a 3-slot ring of 32 KB,
//               this CTA's share of every tile: for S, two slots of four 64-dim slices of N/2
//               entries; for PV, one slot of the tile's entries x 128 value columns
//   warp 1      both CTAs: allocate / free 512 TMEM columns (cta_group::2).  Leader lane 0 issues
//               S_t = Q K_t^T  (M=256, N=entries rounded to 16, K=512; A and B K-major)
//               O  += P_t V_t   (M=256, N=256, K=entries; A = P in TMEM, B = V MN-major)
//               and releases ring slots, S buffers and O in both CTAs with multicast commits.
//               Both CTAs' TMA loads complete on the leader's ring barriers (cta_group::2 TMA).
//   warps 2..9  softmax, two threads per query row (one per half of a tile's columns): read S_t
//               from TMEM, mask, online softmax with a lazily updated row maximum, write P_t back
//               into the S columns as packed bf16, rescale O in TMEM when the maximum grows by
//               more than 2^8, and finally write O.
//   warp 10     lane 0: once every softmax warp of the CTA has stored P_t, signals the leader's
//               p_full (leader: local arrive with expect_tx; follower: a 4-byte st.async).
// TMEM columns: S/P double buffer at [0,128) and [128,256), O at [256,512).
// Every mbarrier wait is bounded; on timeout the CTA records TV_ERR_TIMEOUT, stops issuing work,
// drains its own copies and MMAs (bounded) and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "tv_attn_tc.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace tc {

using namespace sm100;

constexpr int kSmxWarps = 8;           // softmax warps: 4 (a thread per row) or 8 (two per row)
constexpr int kSigWarp = 2 + kSmxWarps;          // forwards "P ready" to the leader
constexpr int kThreads = 64 + 32 * kSmxWarps + 32;   // producer, MMA issuer, softmax, signal
// Ring of 32 KB slots: the rate at which one SM's TMA copies complete is set mostly by the
// number of mbarrier transactions (about 0.3 us each, nearly independent of their size up to
// 64 KB), so a tile's K share (64 KB) takes two slots and its V share (32 KB) one.
constexpr int kSlots = 3;
constexpr int kSlotBytes = 32768;
constexpr int kKSlices = 4;        // 64-dim K slices (64 entries x 128 B, 8 KB) per slot
constexpr int kVBlock = 16384;     // V slot: two 64-column blocks of 128 entries
constexpr int kQBytes = 8 * 16384;
constexpr int kDp = 8;                 // rows per section of the extra tile (D <= 8)
constexpr int kExtraEntries = 32;      // tree | C4 scratch | C128 scratch | zeros
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.f;   // log2 units: P values stay below 2^8

enum TileKind { kC4 = 0, kC128 = 1, kRaw = 2, kExtra = 3 };

struct Params {
  CUtensorMap mQ;
  CUtensorMap mC4K, mC4V, mC128K, mC128V, mRawK, mRawV;
  CUtensorMap mTreeK, mTreeV, mS4K, mS4V, mS128K, mS128V;
  int B, D, H, DH, W, tail_mode, comp_mask, n_pairs, n_chunks;
  int n_sel;       // > 0: the C4 maps point at the gathered selected entries, n_sel per request
  int tree_rows;   // B * D: the first row index past the tree / scratch tensors (zero fill)
  int64_t raw_cap, c4_cap, c128_cap;
  const int32_t* L;
  const int32_t* raw_lo;
  const uint64_t* anc;
  const uint64_t* vis4;
  const uint64_t* vis128;
  float scale_log2;
  __nv_bfloat16* O;
  float* lse;
  float* part;          // split-KV partials (n_chunks > 1)
  const int32_t* order; // requests by decreasing tile count (longest first)
  int32_t* status;
  Paging pg;       // paged pools: C4 tiles are read through the page table; the C128 entries and
                   // the raw tail are first gathered into the workspace (contiguous per request)
  int tail_rows;   // rows per request of the gathered raw tail (paged pools only)
};

struct Layout {
  int L, n4, n128, t0, nraw, T4, T128, Traw, T;
};

struct Tile {
  int kind, row0, valid, nqk;
};

__device__ __forceinline__ Layout layout_of(const Params& p, int b) {
  Layout y;
  const int L = p.L[b];
  const bool c4 = p.comp_mask & TV_COMP_C4, c128 = p.comp_mask & TV_COMP_C128;
  const int n4 = c4 ? (p.n_sel > 0 ? p.n_sel : L / 4) : 0;
  const bool ok = L >= 0 && L <= p.raw_cap && n4 <= p.c4_cap && (!c128 || L / 128 <= p.c128_cap);
  if (!ok) {
    y.L = y.n4 = y.n128 = y.t0 = y.nraw = y.T4 = y.T128 = y.Traw = y.T = 0;
    return y;
  }
  y.L = L;
  y.n4 = n4;
  y.n128 = c128 ? L / 128 : 0;
  const int tail = p.tail_mode == TV_TAIL_WINDOW ? p.W : m_min_of(p.comp_mask) - 1;
  y.t0 = L - tail > 0 ? L - tail : 0;
  y.nraw = L - y.t0;
  y.T4 = (y.n4 + 127) / 128;
  y.T128 = (y.n128 + 127) / 128;
  y.Traw = (y.nraw + 127) / 128;
  y.T = y.T4 + y.T128 + y.Traw + 1;
  return y;
}

__device__ __forceinline__ Tile tile_of(const Layout& y, int t) {
  Tile x;
  if (t < y.T4) {
    x.kind = kC4;
    x.row0 = 128 * t;
    x.valid = min(128, y.n4 - x.row0);
  } else if (t < y.T4 + y.T128) {
    x.kind = kC128;
    x.row0 = 128 * (t - y.T4);
    x.valid = min(128, y.n128 - x.row0);
  } else if (t < y.T4 + y.T128 + y.Traw) {
    x.kind = kRaw;
    x.row0 = y.t0 + 128 * (t - y.T4 - y.T128);
    x.valid = min(128, y.L - x.row0);
  } else {
    x.kind = kExtra;
    x.row0 = 0;
    x.valid = kExtraEntries;
  }
  x.nqk = (x.valid + 15) & ~15;
  return x;
}

// Longest-processing-time-first order of the requests: the pair scheduler starts the longest
// requests first, so the last wave holds the shortest work items.  rank(b) = number of requests
// with more tiles, ties broken by index; order[rank(b)] = b.
__global__ void order_kernel(Params p, int32_t* order) {
  extern __shared__ int tiles[];   // B tile counts
  for (int j = threadIdx.x; j < p.B; j += blockDim.x) tiles[j] = layout_of(p, j).T;
  __syncthreads();
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
    const int tb = tiles[b];
    int rank = 0;
    for (int j = 0; j < p.B; ++j) rank += (tiles[j] > tb || (tiles[j] == tb && j < b)) ? 1 : 0;
    order[rank] = b;
  }
}

// Selected C4 entries ("sparse" prefix attention): copies entry sel[b][i] of request b's K and V
// into row i of a dense per-request buffer, so the attention kernel reads the selection as
// contiguous tiles.  One warp per selected entry; an index outside 0 .. L/4 - 1 (or past the C4
// capacity) records TV_ERR_SELECTION and leaves a zero row.
__global__ void gather_sel_kernel(Paging pg, int B, int n_sel, int64_t c4_cap,
                                  const int32_t* __restrict__ L,
                                  const int32_t* __restrict__ sel, const uint4* __restrict__ c4K,
                                  const uint4* __restrict__ c4V, uint4* __restrict__ gK,
                                  uint4* __restrict__ gV, int32_t* status) {
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)B * n_sel) return;
  const int b = (int)(w / n_sel);
  const int j = sel[w];
  const int Lb = L[b];
  const bool ok = Lb >= 0 && j >= 0 && j < Lb / 4 && j < c4_cap;
  if (!ok && lane == 0) record_error(status, TV_ERR_SELECTION);
  constexpr int kRowU4 = 512 * 2 / 16;   // 64 x 16 B per bf16 row of 512
  const int64_t src = ok ? layer_row(pg, b, j, c4_cap, 4, status) * kRowU4 : 0;
  const int64_t dst = w * kRowU4;
  for (int i = lane; i < kRowU4; i += 32) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    gK[dst + i] = ok ? c4K[src + i] : z;
    gV[dst + i] = ok ? c4V[src + i] : z;
  }
}

// Paged pools: copies each request's C128 entries 0 .. c128_cap-1 and its raw tail (positions
// t0 .. t0 + tail_rows - 1) from the pools into contiguous workspace rows; rows past L/128 or past
// L are zero (the attention loads whole 64-row boxes and masks the extra entries, so they must be
// finite).  One warp per row; grid.y = request.
__global__ void gather_paged_kernel(Paging pg, int comp_mask, int W, int tail_mode,
                                    int64_t raw_cap, int64_t c128_cap, int tail_rows,
                                    const int32_t* __restrict__ L, const uint4* __restrict__ c128K,
                                    const uint4* __restrict__ c128V, const uint4* __restrict__ rawK,
                                    const uint4* __restrict__ rawV, uint4* gK128, uint4* gV128,
                                    uint4* gKraw, uint4* gVraw, int32_t* status) {
  constexpr int kRowU4 = 512 * 2 / 16;
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int Lb = L[b];
  const bool c128 = comp_mask & TV_COMP_C128;
  const int64_t n128 = c128 ? c128_cap : 0;
  const int tail = tail_mode == TV_TAIL_WINDOW ? W : m_min_of(comp_mask) - 1;
  const int t0 = Lb - tail > 0 ? Lb - tail : 0;
  const bool ok = Lb >= 0 && Lb <= raw_cap;
  const int64_t rows = n128 + tail_rows;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w < rows;
       w += (int64_t)gridDim.x * (blockDim.x / 32)) {
    const uint4* sK = nullptr;
    const uint4* sV = nullptr;
    uint4 *dK, *dV;
    if (w < n128) {
      if (ok && w < Lb / 128) {
        const int64_t r = layer_row(pg, b, w, c128_cap, 128, status);
        sK = c128K + r * kRowU4;
        sV = c128V + r * kRowU4;
      }
      dK = gK128 + ((int64_t)b * c128_cap + w) * kRowU4;
      dV = gV128 + ((int64_t)b * c128_cap + w) * kRowU4;
    } else {
      const int64_t pos = t0 + (w - n128);
      if (ok && pos < Lb) {
        const int64_t r = layer_row(pg, b, pos, raw_cap, 1, status);
        sK = rawK + r * kRowU4;
        sV = rawV + r * kRowU4;
      }
      dK = gKraw + ((int64_t)b * tail_rows + (w - n128)) * kRowU4;
      dV = gVraw + ((int64_t)b * tail_rows + (w - n128)) * kRowU4;
    }
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int i = lane; i < kRowU4; i += 32) {
      dK[i] = sK ? sK[i] : z;
      dV[i] = sV ? sV[i] : z;
    }
  }
}

struct __align__(1024) Smem {
  uint8_t q[kQBytes];
  uint8_t ring[kSlots][kSlotBytes];
  uint64_t full[kSlots];       // (leader) both CTAs' shares of a fill have landed
  uint64_t empty[kSlots];      // the pair's MMAs are done with the slot
  uint64_t q_full;             // (leader) both CTAs' Q rows have landed
  uint64_t s_full[2];
  uint64_t p_full[2];          // (leader) P written by both CTAs' softmax warps: the leader's
                               // arrive with expect_tx(4) + the follower's 4-byte st.async
  uint32_t p_flag[2];          // (leader) landing word of the follower's st.async
  uint64_t p_local[2];         // this CTA's softmax warps have written P (one arrive per warp)
  uint64_t pv_done;
  uint64_t o_full;
  uint64_t drain;
  float xmax[2][2][128];       // [tile parity][column half][row] partial row maxima
  int xok[2][2][4];            // [tile parity][column half][lane quadrant] the warp carries on
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ void fail(Smem& sm, int32_t* status) {
  if (atomicExch(&sm.abort, 1) == 0) record_error(status, TV_ERR_TIMEOUT);
}

// Row (in its tensor map) of entry `idx` of a C4 / C128 / raw tile of request b.  Contiguous
// caches: b * cap + idx.  Paged pools: C4 rows through the page table (a 64-row box never crosses
// a C4 page: a page holds a multiple of 128 entries and tiles start at multiples of 128); C128
// entries and raw positions from the gathered copies in the workspace.
template <bool kPaged>
__device__ __forceinline__ int64_t tile_row(const Params& p, int kind, int b, int64_t idx,
                                            int t0) {
  if (kind == kC4) {
    if (kPaged && p.n_sel == 0) return layer_row(p.pg, b, idx, p.c4_cap, 4, p.status);
    return (int64_t)b * p.c4_cap + idx;
  }
  if (kind == kC128) return (int64_t)b * p.c128_cap + idx;
  if (kPaged) return (int64_t)b * p.tail_rows + (idx - t0);
  return (int64_t)b * p.raw_cap + idx;
}

// ---- producer (warp 0 of both CTAs) --------------------------------------------------------
template <bool kPaged>
__device__ void producer(const Params& p, Smem& sm, int b, int rt, int half, uint32_t rank,
                         const Layout& y, int tb, int te) {
  const int lane = threadIdx.x & 31;
  int slot = 0;
  uint32_t phase = 0;
  bool issued[kSlots];
  uint32_t issued_phase[kSlots];
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    issued[i] = false;
    issued_phase[i] = 0;
  }
  if (lane == 0) {
    // both CTAs' Q rows complete on the leader's q_full: the pair's MMAs read both
    const uint32_t q_bar = mapa_cluster(smem_u32(&sm.q_full), 0);
    if (rank == 0) mbar_arrive_expect_tx(&sm.q_full, 2 * kQBytes);
    for (int s = 0; s < 8; ++s)
      tma_load_3d_pair(sm.q + s * 16384, &p.mQ, 64 * s, 128 * rt, b, q_bar);
  }
  auto acquire = [&]() -> bool {
    if (!mbar_wait(&sm.empty[slot], phase ^ 1, &sm.abort, kTimeoutNs)) {
      if (lane == 0) fail(sm, p.status);
      return false;
    }
    return true;
  };
  auto advance = [&]() {
    issued[slot] = true;
    issued_phase[slot] = phase;
    if (++slot == kSlots) {
      slot = 0;
      phase ^= 1;
    }
  };
  const int tree_row = b * p.D;
  // both CTAs' shares of a fill complete on the leader's full[slot]; the leader expects both
  auto leader_full = [&](int sl) { return mapa_cluster(smem_u32(&sm.full[sl]), 0); };
  auto expect = [&](uint32_t bytes) {
    if (rank == 0) mbar_arrive_expect_tx(&sm.full[slot], 2 * bytes);
  };
  // S operand: this CTA holds entries [rank * nqk/2, (rank+1) * nqk/2) of the tile; one slot
  // holds four 64-dim slices of those (up to 64) entries, 8 KB each.
  // rows of a tile's boxes (this CTA's K half, the two V halves), computed one tile ahead so that
  // with paged pools the page-table reads are in flight while the producer waits for slots
  struct Rows {
    int k, v0, v1;
  };
  auto rows_of = [&](int t) -> Rows {
    Rows r{0, 0, 0};
    if (t < tb || t >= te) return r;
    const Tile x = tile_of(y, t);
    if (x.kind == kExtra) return r;
    r.k = (int)tile_row<kPaged>(p, x.kind, b, x.row0 + (int)rank * (x.nqk / 2), y.t0);
    r.v0 = (int)tile_row<kPaged>(p, x.kind, b, x.row0, y.t0);
    r.v1 = kPaged ? (int)tile_row<kPaged>(p, x.kind, b, x.row0 + 64, y.t0) : r.v0 + 64;
    return r;
  };
  auto load_k = [&](const Tile& x, const Rows& rw) -> bool {
    const int nh = x.nqk / 2;
    for (int j = 0; j < 512 / (64 * kKSlices); ++j) {
      if (!acquire()) return false;
      if (lane == 0) {
        uint8_t* dst = sm.ring[slot];
        const uint32_t bar = leader_full(slot);
        if (x.kind == kExtra) {
          // leader: tree rows | C4 scratch rows; follower: C128 scratch rows | zero rows
          expect(kKSlices * 2 * kDp * 128);
          for (int ks = 0; ks < kKSlices; ++ks) {
            const int xcol = 64 * (kKSlices * j + ks);
            uint8_t* d = dst + ks * 8192;
            if (rank == 0) {
              tma_load_2d_pair(d, &p.mTreeK, xcol, tree_row, bar);
              tma_load_2d_pair(d + kDp * 128, &p.mS4K, xcol, tree_row, bar);
            } else {
              tma_load_2d_pair(d, &p.mS128K, xcol, tree_row, bar);
              tma_load_2d_pair(d + kDp * 128, &p.mTreeK, xcol, p.tree_rows, bar);
            }
          }
        } else {
          const CUtensorMap* m = x.kind == kC4 ? &p.mC4K : x.kind == kC128 ? &p.mC128K : &p.mRawK;
          const int r = rw.k;
          expect(kSlotBytes);
          for (int ks = 0; ks < kKSlices; ++ks)
            tma_load_2d_pair(dst + ks * 8192, m, 64 * (kKSlices * j + ks), r, bar);
        }
      }
      advance();
    }
    return true;
  };
  // PV operand: every entry of the tile, this CTA's 128 of the pair's 256 value columns; one slot
  // holds the tile's entries as two 64-column blocks of 128 rows (rows past the tile's entry
  // count rounded up to 64 are not loaded).
  auto load_v = [&](const Tile& x, const Rows& rw) -> bool {
    const int nvh = (x.nqk + 63) / 64;   // 64-row halves to load
    const int col0 = 256 * half + 128 * (int)rank;
    {
      if (!acquire()) return false;
      if (lane == 0) {
        uint8_t* dst = sm.ring[slot];
        const uint32_t bar = leader_full(slot);
        if (x.kind == kExtra) {
          expect(2 * 4 * kDp * 128);
          for (int cb = 0; cb < 2; ++cb) {
            uint8_t* d = dst + cb * kVBlock;
            const int xc = col0 + 64 * cb;
            tma_load_2d_pair(d, &p.mTreeV, xc, tree_row, bar);
            tma_load_2d_pair(d + kDp * 128, &p.mS4V, xc, tree_row, bar);
            tma_load_2d_pair(d + 2 * kDp * 128, &p.mS128V, xc, tree_row, bar);
            tma_load_2d_pair(d + 3 * kDp * 128, &p.mTreeV, xc, p.tree_rows, bar);   // zeros
          }
        } else {
          const CUtensorMap* m = x.kind == kC4 ? &p.mC4V : x.kind == kC128 ? &p.mC128V : &p.mRawV;
          expect(nvh * 2 * 8192);
          for (int h = 0; h < nvh; ++h) {
            const int r = h == 0 ? rw.v0 : rw.v1;
            for (int cb = 0; cb < 2; ++cb)
              tma_load_2d_pair(dst + cb * kVBlock + h * 8192, m, col0 + 64 * cb, r, bar);
          }
        }
      }
      advance();
    }
    return true;
  };
  bool ok = true;
  Rows prev = rows_of(tb - 1), cur = rows_of(tb);
  for (int t = tb; t < te && ok; ++t) {
    const Rows next = rows_of(t + 1);
    ok = load_k(tile_of(y, t), cur);
    if (ok && t > tb) ok = load_v(tile_of(y, t - 1), prev);
    prev = cur;
    cur = next;
  }
  if (ok && te > tb) load_v(tile_of(y, te - 1), prev);
  // drain: no copy issued by the pair may still be in flight when the CTA exits (the leader's
  // full and q_full barriers count both CTAs' shares; the closing cluster barrier covers the
  // follower)
  if (rank == 0) {
    volatile int never = 0;
    for (int i = 0; i < kSlots; ++i)
      if (issued[i]) mbar_wait(&sm.full[i], issued_phase[i], &never, kTimeoutNs / 4);
    mbar_wait(&sm.q_full, 0, &never, kTimeoutNs / 4);
  }
}

// ---- leader lane 0 of warp 1: the pair's MMAs ---------------------------------------------------
__device__ void mma_issuer(const Params& p, Smem& sm, const Layout& y, int tb, int te) {
  const uint32_t tmem = sm.tmem;
  const uint16_t pair = 0x3;
  int slot = 0;
  uint32_t phase = 0;
  auto wait_slot = [&]() -> bool {
    if (!mbar_wait(&sm.full[slot], phase, &sm.abort, kTimeoutNs)) {
      fail(sm, p.status);
      return false;
    }
    tc_fence_after();
    return true;
  };
  auto release = [&]() {
    mma2_commit_mc(&sm.empty[slot], pair);
    if (++slot == kSlots) {
      slot = 0;
      phase ^= 1;
    }
  };
  bool ok = mbar_wait(&sm.q_full, 0, &sm.abort, kTimeoutNs);
  if (!ok) fail(sm, p.status);
  tc_fence_after();
  const uint32_t q_base = smem_u32(sm.q);
  const uint32_t idO = idesc_bf16_f32(256, 256, 0, 1);
  auto pv = [&](int j) -> bool {
    const Tile x = tile_of(y, tb + j);
    if (!mbar_wait(&sm.p_full[j & 1], (j >> 1) & 1, &sm.abort, kTimeoutNs)) {
      fail(sm, p.status);
      return false;
    }
    tc_fence_after();
    const int nks = x.nqk / 16;
    {
      if (!wait_slot()) return false;
      const uint32_t vbase = smem_u32(sm.ring[slot]);
      for (int ks = 0; ks < nks; ++ks) {
        const uint64_t bdesc = smem_desc_sw128(vbase + 2048 * ks, kVBlock, 1024);
        mma2_ts(tmem + 256, tmem + 128 * (j & 1) + 8 * ks, bdesc, idO, (j > 0 || ks > 0) ? 1u : 0u);
      }
      release();
    }
    mma2_commit_mc(&sm.pv_done, pair);
    return true;
  };
  const int n = te - tb;
  for (int i = 0; i < n && ok; ++i) {
    const Tile x = tile_of(y, tb + i);
    const uint32_t idS = idesc_bf16_f32(256, x.nqk, 0, 0);
    const uint32_t d_s = tmem + 128 * (i & 1);
    for (int j = 0; j < 512 / (64 * kKSlices) && ok; ++j) {
      if (!wait_slot()) {
        ok = false;
        break;
      }
      const uint32_t kbase = smem_u32(sm.ring[slot]);
      for (int ks = 0; ks < kKSlices; ++ks)
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = smem_desc_sw128(q_base + (kKSlices * j + ks) * 16384 + 32 * kk, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kbase + ks * 8192 + 32 * kk, 16, 1024);
          mma2_ss(d_s, a, bd, idS, (j | ks | kk) ? 1u : 0u);
        }
      release();
    }
    if (!ok) break;
    mma2_commit_mc(&sm.s_full[i & 1], pair);
    if (i >= 1) ok = pv(i - 1);
  }
  if (ok && n > 0) ok = pv(n - 1);
  if (ok) mma2_commit_mc(&sm.o_full, pair);
  // drain every MMA this thread issued before TMEM is released
  mma2_commit_mc(&sm.drain, 0x1);
  volatile int never = 0;
  mbar_wait(&sm.drain, 0, &never, kTimeoutNs / 4);
}

// ---- softmax / epilogue (softmax warps of both CTAs) ----------------------------------------
// kSmxWarps warps; warp w (>= 2) serves TMEM lane quadrant w % 4 (rows 32*(w%4) .. +31).  With 8
// warps, two threads share a row (column half ch = (w-2)/4 each) and exchange their partial row
// maxima through shared memory once per tile; with 4 warps one thread owns the whole row.  Both
// threads of a row apply the same running maximum; partial row sums are combined at the end.
constexpr int kCh = kSmxWarps / 4;          // threads per row
constexpr int kColsPerThread = 128 / kCh;   // S columns per thread and tile
constexpr int kOColsPerThread = 256 / kCh;  // O columns per thread

__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
}

// ---- signal warp: P of tile i is in both CTAs' TMEM -> the leader's MMA issuer ----------------
// Lane 0 waits until all softmax warps of this CTA have stored P_i (local barrier).  The leader
// then arrives on its own p_full with expect_tx(4); the follower completes those 4 bytes with an
// asynchronous 4-byte store into the leader's shared memory (st.async with complete_tx), which
// lands much sooner than a cluster-scope release-arrive.  The follower cannot signal tile i + 2
// before p_full(i) completed: its S(i+2) needs the leader's PV(i), issued after p_full(i).
__device__ void p_signal(const Params& p, Smem& sm, int n, uint32_t rank) {
  const uint32_t flag_leader[2] = {mapa_cluster(smem_u32(&sm.p_flag[0]), 0),
                                   mapa_cluster(smem_u32(&sm.p_flag[1]), 0)};
  const uint32_t bar_leader[2] = {mapa_cluster(smem_u32(&sm.p_full[0]), 0),
                                  mapa_cluster(smem_u32(&sm.p_full[1]), 0)};
  for (int i = 0; i < n; ++i) {
    const int sb = i & 1;
    if (!mbar_wait(&sm.p_local[sb], (i >> 1) & 1, &sm.abort, kTimeoutNs)) {
      fail(sm, p.status);
      return;
    }
    if (rank == 0)
      mbar_arrive_expect_tx(&sm.p_full[sb], 4);
    else
      st_async_signal(flag_leader[sb], (uint32_t)i, bar_leader[sb]);
  }
}

__device__ void softmax_epilogue(const Params& p, Smem& sm, int b, int rt, int half, int chunk,
                                 const Layout& y, int tb, int te) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int ch = (warp - 2) >> 2;           // always 0 with 4 softmax warps
  const int row = 32 * quad + lane;
  const int grow = 128 * rt + row;
  const bool row_ok = grow < p.DH;
  const uint32_t tmem = sm.tmem;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const float sl2 = p.scale_log2;

  // per-row visibility of the raw tail and of the extra tile
  int raw_lo = 0;
  uint32_t extra_mask = 0;   // bit j: entry j of the extra tile is visible
  if (row_ok) {
    const int v = grow / p.H;
    const int64_t i = (int64_t)b * p.D + v;
    const uint64_t an = p.anc[i];
    raw_lo = p.raw_lo[i];
    const uint64_t v4 = (p.comp_mask & TV_COMP_C4) ? p.vis4[i] : 0;
    const uint64_t v128 = (p.comp_mask & TV_COMP_C128) ? p.vis128[i] : 0;
    for (int u = 0; u < p.D; ++u) {
      if ((an >> u) & 1ull) {
        const int dep = __popcll(an & ((1ull << u) - 1ull));
        if (y.L + dep >= raw_lo) extra_mask |= 1u << u;
      }
      if ((v4 >> u) & 1ull) extra_mask |= 1u << (kDp + u);
      if ((v128 >> u) & 1ull) extra_mask |= 1u << (2 * kDp + u);
    }
  }

  float m_ref = -INFINITY, l_run = 0.f;
  const int n = te - tb;
  // The two warps of a row (column halves) meet at one named barrier per tile and one after the
  // tiles.  A warp whose bounded wait ran out still takes each barrier until both warps leave the
  // tile loop together (each tile's exchange carries both warps' flags), so neither waits on the
  // other forever.
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    const Tile x = tile_of(y, tb + i);
    const int sb = i & 1;
    const int c0 = kColsPerThread * ch;     // first S column of this thread
    // the wait result is made warp-uniform: tcgen05.ld below is warp-collective
    if (ok && !__all_sync(0xffffffffu,
                          mbar_wait(&sm.s_full[sb], (i >> 1) & 1, &sm.abort, kTimeoutNs))) {
      fail(sm, p.status);
      ok = false;
    }
    float s[kColsPerThread];
    float raw_max = -INFINITY;
    if (ok) {
      tc_fence_after();
      {
        uint32_t* sr = reinterpret_cast<uint32_t*>(s);
#pragma unroll
        for (int c = 0; c < kColsPerThread / 32; ++c)
          if (c0 + 32 * c < x.nqk)
            tmem_ld32(tmem + lane_base + 128 * sb + c0 + 32 * c,
                      *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
        tmem_wait_ld();
      }
      // row maximum of the visible raw logits (scale > 0, so the scaled maximum follows)
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
      const bool full_tile = (x.kind == kC4 || x.kind == kC128) && x.valid >= 128;
      if (full_tile) {
#pragma unroll
        for (int j = 0; j < kColsPerThread; ++j) mx[j & 7] = fmaxf(mx[j & 7], s[j]);
      } else {
#pragma unroll
        for (int j = 0; j < kColsPerThread; ++j) {
          const int col = c0 + j;
          bool vis = col < x.valid;
          if (x.kind == kRaw) vis = vis && (x.row0 + col >= raw_lo);
          if (x.kind == kExtra) vis = col < 32 && ((extra_mask >> (col & 31)) & 1u);
          s[j] = vis ? s[j] : -INFINITY;
          mx[j & 7] = fmaxf(mx[j & 7], s[j]);
        }
      }
      raw_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                      fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
    }
    if (kCh == 2) {
      sm.xmax[sb][ch][row] = raw_max;
      if (lane == 0) sm.xok[sb][ch][quad] = ok ? 1 : 0;
      pair_sync(quad);
      raw_max = fmaxf(raw_max, sm.xmax[sb][ch ^ 1][row]);
      if (ok && !sm.xok[sb][ch ^ 1][quad]) {   // the row's other warp gave up
        fail(sm, p.status);
        ok = false;
      }
    }
    if (!ok) break;
    const float mt = raw_max * sl2;
    const bool grow_max = mt > m_ref + kRescaleThreshold;
    const float m_new = grow_max ? mt : m_ref;
    const float alpha = (grow_max && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
    // rescale this thread's O columns in TMEM before P_i is accumulated onto them (rare)
    const bool need_rescale = grow_max && m_ref != -INFINITY && i > 0;
    if (__any_sync(0xffffffffu, need_rescale)) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.pv_done, (i - 1) & 1, &sm.abort, kTimeoutNs))) {
        fail(sm, p.status);
        ok = false;   // the tile loop ends at the next exchange, together with the other warp
        continue;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kOColsPerThread / 8; ++c) {
        uint32_t r[8];
        const uint32_t col = tmem + lane_base + 256 + kOColsPerThread * ch + 8 * c;
        tmem_ld8(col, r);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
        tmem_st8(col, r);
      }
      tmem_wait_st();
    }
    const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
    float sum[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sum[k] = 0.f;
#pragma unroll
    for (int c = 0; c < kColsPerThread / 64; ++c) {
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = ex2_approx(fmaf(s[64 * c + 2 * j], sl2, neg_m));
        const float p1 = ex2_approx(fmaf(s[64 * c + 2 * j + 1], sl2, neg_m));
        sum[j & 3] += p0 + p1;
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        pk[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      // P column k holds entries 2k and 2k+1
      if (c0 + 64 * c < x.nqk) tmem_st32(tmem + lane_base + 128 * sb + (c0 >> 1) + 32 * c, pk);
    }
    const float tsum = (sum[0] + sum[1]) + (sum[2] + sum[3]);
    l_run = l_run * alpha + tsum;
    m_ref = m_new;
    tmem_wait_st();
    tc_fence_before();
    // each warp's rows of P are in TMEM; the signal warp forwards the CTA's readiness to the
    // leader, so no softmax warp waits for the cross-CTA arrive
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.p_local[sb]);
  }
  if (ok && n > 0) {
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full, 0, &sm.abort, kTimeoutNs))) {
      fail(sm, p.status);
      ok = false;
    }
  }
  float l_tot = l_run;
  if (kCh == 2) {
    // combine the two partial row sums (both threads of a row share m_ref); once o_full has been
    // observed every copy and MMA of this CTA's ring is done, so its first slot holds the exchange
    float* xsum = reinterpret_cast<float*>(sm.ring[0]);
    xsum[128 * ch + row] = l_run;
    pair_sync(quad);
    l_tot = l_run + xsum[128 * (ch ^ 1) + row];
  }
  if (!ok) return;
  tc_fence_after();
  const int d = 512;
  const int ocol = 256 * half + kOColsPerThread * ch;   // first O column of this thread
  if (p.n_chunks == 1) {
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    __nv_bfloat16* orow = p.O + ((int64_t)b * p.DH + grow) * d + ocol;
    for (int c = 0; c < kOColsPerThread / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + 256 + kOColsPerThread * ch + 32 * c, r);
      tmem_wait_ld();
      if (row_ok) {
        uint4 w[4];
        uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * k]) * inv,
                                                         __uint_as_float(r[2 * k + 1]) * inv);
          wp[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = w[k];
      }
    }
    if (row_ok && half == 0 && ch == 0)
      p.lse[(int64_t)b * p.DH + grow] =
          l_tot > 0.f ? (m_ref + log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
  } else {
    float* prow = p.part + (((int64_t)b * p.DH + grow) * p.n_chunks + chunk) * (d + 4);
    for (int c = 0; c < kOColsPerThread / 32; ++c) {
      uint32_t r[32];
      if (n > 0) {
        tmem_ld32(tmem + lane_base + 256 + kOColsPerThread * ch + 32 * c, r);
        tmem_wait_ld();
      }
      if (row_ok) {
        float4* dst = reinterpret_cast<float4*>(prow + ocol + 32 * c);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k] = n > 0 ? make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                       __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (row_ok && half == 0 && ch == 0) {
      prow[d] = m_ref;
      prow[d + 1] = l_tot;
    }
  }
}

// kPaged: the persistent cache is in page pools (C4 tiles through the page table, C128 entries
// and the raw tail from gathered copies); a separate instantiation keeps the contiguous path's
// producer free of the page-table work.
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // the swizzled operand tiles need 1 KB alignment; the dynamic window starts 1 KB aligned
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.status, TV_ERR_CUDA);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid: clusters of 2 consecutive CTAs = the row tiles 2*pair and 2*pair+1
  const uint32_t rank = blockIdx.x & 1;
  int x = blockIdx.x >> 1;
  const int half = x & 1;
  x >>= 1;
  const int pair_idx = x % p.n_pairs;
  x /= p.n_pairs;
  const int chunk = x % p.n_chunks;
  const int b = p.order[x / p.n_chunks];
  const int rt = 2 * pair_idx + (int)rank;

  const Layout y = layout_of(p, b);   // identical in both CTAs of the pair
  if (y.T == 0) {
    if (threadIdx.x == 0) record_error(p.status, TV_ERR_CAPACITY);
    return;
  }
  const int tb = (int)((int64_t)y.T * chunk / p.n_chunks);
  const int te = (int)((int64_t)y.T * (chunk + 1) / p.n_chunks);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.p_full[0], 1);
    mbar_init(&sm.p_full[1], 1);
    mbar_init(&sm.p_local[0], kSmxWarps);
    mbar_init(&sm.p_local[1], kSmxWarps);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.mQ);
    prefetch_tmap(&p.mC4K);
    prefetch_tmap(&p.mC4V);
  }
  if (warp == 1) {
    tmem_alloc2(&sm.tmem, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers exist before any remote arrive or pair MMA
  tc_fence_after();

  if (tb < te) {
    if (warp == 0) {
      producer<kPaged>(p, sm, b, rt, half, rank, y, tb, te);
    } else if (warp == 1) {
      if (lane == 0) {
        if (rank == 0) mma_issuer(p, sm, y, tb, te);
      }
      __syncwarp();
    } else if (warp == kSigWarp) {
      if (lane == 0) p_signal(p, sm, te - tb, rank);
      __syncwarp();
    } else {
      softmax_epilogue(p, sm, b, rt, half, chunk, y, tb, te);
    }
  } else if (warp >= 2 && warp < kSigWarp) {
    softmax_epilogue(p, sm, b, rt, half, chunk, y, tb, te);   // empty chunk: l = 0
  }

  tc_fence_before();
  cluster_sync();   // the leader's MMAs are drained and no remote arrive is still in flight
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(sm.tmem, 512);
}

}  // namespace tc
}  // namespace tv

// ---- host side ----------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D (rows x 512) or 3-D (B x rows x 512) bf16 map with the 128-byte swizzle, box 64 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int rank, uint64_t rows, uint64_t batch,
              uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr) return false;
  cuuint64_t dims[3] = {512, rows, batch};
  cuuint64_t strides[2] = {512 * 2, rows * 512 * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int n_pairs_of(const tv_shape* s) { return ((s->D * s->H + 127) / 128 + 1) / 2; }

// Number of KV chunks per request.  Clusters of 2 CTAs run one per SM pair; a cluster costs about
// (its tiles + 2) tile-times (the Q load and the epilogue).  With T the largest tile count the
// capacities allow, pick the chunk count that minimises waves x (ceil(T / n) + 2); a larger count
// must win by more than 10 % (splitting adds fp32 partials and a merge pass).
int tc_chunks(const tv_shape* s) {
  static int pair_slots = 0;
  if (pair_slots == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2)
      sms = 152;
    cudaGetLastError();
    pair_slots = sms / 2;
  }
  int64_t max_tiles = 1 + (s->tail_mode == TV_TAIL_WINDOW ? (s->W + 127) / 128 : 1);
  if (s->comp_mask & TV_COMP_C4) max_tiles += ((s->n_sel > 0 ? s->n_sel : s->c4_cap) + 127) / 128;
  if (s->comp_mask & TV_COMP_C128) max_tiles += (s->c128_cap + 127) / 128;
  const int64_t clusters1 = (int64_t)s->B * n_pairs_of(s) * 2;   // two value halves
  int best = 1;
  int64_t best_cost = -1;
  for (int n = 1; n <= 64 && n <= max_tiles; ++n) {
    const int64_t waves = (clusters1 * n + pair_slots - 1) / pair_slots;
    const int64_t cost = waves * ((max_tiles + n - 1) / n + 2);
    if (best_cost < 0 || 10 * cost < 9 * best_cost) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

}  // namespace

bool tv_tc_shape_ok(const tv_shape* s) {
  return s->dtype == TV_BF16 && s->d == 512 && s->D <= tv::tc::kDp &&
         s->B <= 12288 &&   // the ranking kernel keeps one int per request in shared memory
         (int64_t)s->B * s->raw_cap < ((int64_t)1 << 31) &&
         (int64_t)s->B * s->c4_cap < ((int64_t)1 << 31) &&
         (int64_t)s->B * s->n_sel < ((int64_t)1 << 31) &&
         (int64_t)s->B * s->c128_cap < ((int64_t)1 << 31);
}

bool tv_tc_available() {
  static int cached = -1;
  if (cached < 0) {
    int dev = 0, major = 0, minor = 0;
    cached = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess)
      cached = (major == 10 && minor == 3 && encode_fn() != nullptr) ? 1 : 0;
    cudaGetLastError();
  }
  return cached == 1;
}

// Workspace: the request order (B int32, padded to 256 B), the gathered selected C4 entries (K
// then V, B x n_sel x 512 bf16 each, when n_sel > 0), then the split-KV partials.
static size_t order_bytes(const tv_shape* s) { return ((size_t)s->B * 4 + 255) / 256 * 256; }
static size_t gather_bytes(const tv_shape* s) {
  return s->n_sel > 0 ? (size_t)s->B * s->n_sel * 512 * 2 : 0;   // one of K / V (multiple of 1 KB)
}
// Paged pools: rows per request of the gathered raw tail (a whole number of 128-row tiles).
static int tail_rows_of(const tv_shape* s) {
  const int tail = s->tail_mode == TV_TAIL_WINDOW ? s->W : tv::m_min_of(s->comp_mask) - 1;
  return 128 * (((tail > 0 ? tail : 1) + 127) / 128);
}
static size_t paged_c128_bytes(const tv_shape* s) {   // one of K / V
  return s->page_tokens > 0 && (s->comp_mask & TV_COMP_C128) ? (size_t)s->B * s->c128_cap * 1024
                                                               : 0;
}
static size_t paged_raw_bytes(const tv_shape* s) {    // one of K / V
  return s->page_tokens > 0 ? (size_t)s->B * tail_rows_of(s) * 1024 : 0;
}
static size_t pre_partial_bytes(const tv_shape* s) {
  return order_bytes(s) + 2 * gather_bytes(s) + 2 * paged_c128_bytes(s) + 2 * paged_raw_bytes(s);
}

size_t tv_tc_workspace_size(const tv_shape* s) {
  const int n = tc_chunks(s);
  size_t bytes = pre_partial_bytes(s);
  if (n > 1) bytes += (size_t)s->B * s->D * s->H * n * (s->d + 4) * sizeof(float);
  return bytes;
}

int tv_launch_attn_tc(const tv_shape* s, const tv::AttnParams<__nv_bfloat16>& a, void* workspace,
                      cudaStream_t stream) {
  using namespace tv::tc;
  Params p;   // copied into the launch's parameter buffer
  const int DH = s->D * s->H;
  const uint64_t B = (uint64_t)s->B;
  // an inactive compressor's maps are pointed at the raw buffer (never read: its tiles are empty)
  const bool c4 = s->comp_mask & TV_COMP_C4, c128 = s->comp_mask & TV_COMP_C128;
  char* ws = reinterpret_cast<char*>(workspace);
  const void* c4K = c4 ? a.c4K : a.rawK;
  const void* c4V = c4 ? a.c4V : a.rawV;
  const bool gathered = c4 && s->n_sel > 0;
  if (gathered) {
    c4K = ws + order_bytes(s);
    c4V = ws + order_bytes(s) + gather_bytes(s);
  }
  const bool paged = s->page_tokens > 0;
  const void* c128K = c128 ? a.c128K : a.rawK;
  const void* c128V = c128 ? a.c128V : a.rawV;
  const void* rawK = a.rawK;
  const void* rawV = a.rawV;
  char* g128 = ws + order_bytes(s) + 2 * gather_bytes(s);
  char* graw = g128 + 2 * paged_c128_bytes(s);
  if (paged) {
    if (c128) {
      c128K = g128;
      c128V = g128 + paged_c128_bytes(s);
    }
    rawK = graw;
    rawV = graw + paged_raw_bytes(s);
  }
  const void* s4K = c4 ? a.scrK4 : a.treeK;
  const void* s4V = c4 ? a.scrV4 : a.treeV;
  const void* s128K = c128 ? a.scrK128 : a.treeK;
  const void* s128V = c128 ? a.scrV128 : a.treeV;
  auto rows_or_one = [](uint64_t r) { return r > 0 ? r : (uint64_t)1; };
  // rows of each map: contiguous caches B x cap; paged C4 pool pages x P/4; gathered copies B x n
  const uint64_t rawrows = rows_or_one(paged ? B * (uint64_t)tail_rows_of(s)
                                             : B * (uint64_t)s->raw_cap);
  const uint64_t c4rows = rows_or_one(
      gathered ? B * (uint64_t)s->n_sel
               : !c4 ? rawrows
                     : paged ? (uint64_t)s->n_pool_pages * (s->page_tokens / 4)
                             : B * (uint64_t)s->c4_cap);
  const uint64_t c128rows = rows_or_one(c128 ? B * (uint64_t)s->c128_cap : rawrows);
  if (!c4) {
    c4K = rawK;
    c4V = rawV;
  }
  if (!c128) {
    c128K = rawK;
    c128V = rawV;
  }
  const uint64_t trows = B * (uint64_t)s->D;
  bool ok = make_map(&p.mQ, a.Q, 3, DH, B, 128);
  ok = ok && make_map(&p.mC4K, c4K, 2, c4rows, 1, 64) && make_map(&p.mC4V, c4V, 2, c4rows, 1, 64);
  ok = ok && make_map(&p.mC128K, c128K, 2, c128rows, 1, 64) &&
       make_map(&p.mC128V, c128V, 2, c128rows, 1, 64);
  ok = ok && make_map(&p.mRawK, rawK, 2, rawrows, 1, 64) &&
       make_map(&p.mRawV, rawV, 2, rawrows, 1, 64);
  ok = ok && make_map(&p.mTreeK, a.treeK, 2, trows, 1, kDp) &&
       make_map(&p.mTreeV, a.treeV, 2, trows, 1, kDp);
  ok = ok && make_map(&p.mS4K, s4K, 2, trows, 1, kDp) && make_map(&p.mS4V, s4V, 2, trows, 1, kDp);
  ok = ok && make_map(&p.mS128K, s128K, 2, trows, 1, kDp) &&
       make_map(&p.mS128V, s128V, 2, trows, 1, kDp);
  if (!ok) return tv_set_error(TV_ERR_CUDA, "tv_tree_verify_attn: tensor-map encoding failed");
  p.B = s->B;
  p.D = s->D;
  p.H = s->H;
  p.DH = DH;
  p.W = s->W;
  p.tail_mode = s->tail_mode;
  p.comp_mask = s->comp_mask;
  p.n_pairs = n_pairs_of(s);
  p.n_chunks = tc_chunks(s);
  p.tree_rows = (int)trows;
  p.raw_cap = s->raw_cap;
  p.c4_cap = gathered ? s->n_sel : s->c4_cap;
  p.n_sel = gathered ? s->n_sel : 0;
  p.c128_cap = s->c128_cap;
  p.pg = tv::paging_of(s);
  p.tail_rows = tail_rows_of(s);
  p.L = a.L;
  p.raw_lo = a.raw_lo;
  p.anc = a.anc;
  p.vis4 = a.scr_vis4;
  p.vis128 = a.scr_vis128;
  p.scale_log2 = a.scale_log2;
  p.O = a.O;
  p.lse = a.lse;
  int32_t* order = reinterpret_cast<int32_t*>(workspace);
  p.order = order;
  p.part = reinterpret_cast<float*>(ws + pre_partial_bytes(s));
  p.status = a.status;
  if (gathered && s->B > 0) {
    const int64_t rows = (int64_t)s->B * s->n_sel;
    gather_sel_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        tv::paging_of(s), s->B, s->n_sel, s->c4_cap, a.L, a.sel, reinterpret_cast<const uint4*>(a.c4K),
        reinterpret_cast<const uint4*>(a.c4V), reinterpret_cast<uint4*>(ws + order_bytes(s)),
        reinterpret_cast<uint4*>(ws + order_bytes(s) + gather_bytes(s)), a.status);
    if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05 selection gather)")) return rc;
  }
  if (paged && s->B > 0) {
    const int64_t rows = (c128 ? s->c128_cap : 0) + tail_rows_of(s);
    const unsigned gx = (unsigned)((rows + 7) / 8 < 4096 ? (rows + 7) / 8 : 4096);
    gather_paged_kernel<<<dim3(gx, s->B), 256, 0, stream>>>(
        tv::paging_of(s), s->comp_mask, s->W, s->tail_mode, s->raw_cap, s->c128_cap,
        tail_rows_of(s), a.L, reinterpret_cast<const uint4*>(a.c128K),
        reinterpret_cast<const uint4*>(a.c128V), reinterpret_cast<const uint4*>(a.rawK),
        reinterpret_cast<const uint4*>(a.rawV), reinterpret_cast<uint4*>(g128),
        reinterpret_cast<uint4*>(g128 + paged_c128_bytes(s)), reinterpret_cast<uint4*>(graw),
        reinterpret_cast<uint4*>(graw + paged_raw_bytes(s)), a.status);
    if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05 paged gather)")) return rc;
  }
  // one CTA ranks all requests (B <= 12288 fits its default shared memory)
  order_kernel<<<1, 1024, (size_t)s->B * sizeof(int), stream>>>(p, order);
  if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05 schedule)")) return rc;
  const size_t smem = sizeof(Smem);
  // once per device (a plain host call that also stays out of any stream being captured)
  static std::mutex attr_mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return tv_check_launch("tv_tree_verify_attn (tcgen05 device query)");
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess ||
          cudaFuncSetAttribute(attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return tv_check_launch("tv_tree_verify_attn (tcgen05 shared-memory attribute)");
      attr_set[dev] = true;
    }
  }
  const unsigned grid = (unsigned)(s->B * p.n_chunks * p.n_pairs * 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = paged ? cudaLaunchKernelEx(&cfg, attn_kernel<true>, p)
                               : cudaLaunchKernelEx(&cfg, attn_kernel<false>, p);
  if (le != cudaSuccess)
    return tv_check_launch("tv_tree_verify_attn (tcgen05 pair launch)");
  if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05)")) return rc;
  if (p.n_chunks > 1)
    return tv_launch_merge<__nv_bfloat16>(s->B, DH, 512, p.n_chunks, p.part, a.O, a.lse, stream);
  return TV_OK;
}
