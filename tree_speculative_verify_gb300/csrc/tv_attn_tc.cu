// Branch-aware causal tree-verify attention on the 5th-generation tensor cores (tcgen05), bf16,
// head dim 512, for sm_103a.
//
// "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference":
// §3.1 every candidate attends to the accepted context plus its own ancestors; §3.2 / §4.2 blocks
// closed inside the tree are seen only through the branch's scratch-pad entries.  With H query
// heads sharing one K/V head, all D*H query rows of a request read the same compressed prefix, so
// the prefix part is a dense (D*H) x entries x 512 contraction -- tensor-core work.
//
// Work item: request b, two consecutive 128-row tiles of the request's D*H query rows
// (node-major) and one chunk of the request's KV tiles.  A persistent grid holds one cluster of
// four CTAs per resident cluster slot; cluster c walks the longest-first item list in a snake
// order (item c, then 2G-1-c, 2G+c, ...), and tile counters run across its items, so barriers,
// TMEM and the rings are set up once.  The cluster is two CTA pairs that split the work of every
// KV tile by stage rather than by data:
//   pair S (ranks 0-1)   S_t = Q K_t^T with cta_group::2 MMAs (M = 256: each CTA's tensor core on
//                        its own 128 rows; N = tile entries; K = 512, A = Q from TMEM, B = K from
//                        shared memory, split between the two CTAs), then the online softmax; each
//                        CTA stages its rows' bf16 P_t (with the rows' rescale factors) and one bulk
//                        shared-memory copy takes it to the CTA of the other pair that holds the
//                        same rows
//   pair O (ranks 2-3)   O += P_t V_t with cta_group::2 MMAs (A = P from shared memory, B = V,
//                        N = 2 x 256 value columns), O for all 512 columns in TMEM
// A 128-row fp32 O of all 512 columns fills the 512 TMEM columns of a CTA, so S and O cannot share
// one; Q (512 dims as packed bf16 = 256 columns) and two S buffers fill pair S's TMEM instead.
// Every S element is computed once, both pairs issue the same number of equally sized MMAs per
// tile, and pair S keeps no Q in shared memory, which leaves it a deep ring of K slots.  The
// running row maximum lives in pair S; when it grows (lazily, by more than 2^8) pair S sends the
// rescale factor with P and pair O rescales its O rows before accumulating P_t.
//
// KV tiles (<= 128 entries each), in order: persistent C4 entries, persistent C128 entries, the raw
// tail (positions t0 .. L-1), and one "extra" tile of 32 entries: the tree tokens (0..7), the C4
// scratch rows (8..15), the C128 scratch rows (16..23) and 8 zero rows.  Shared tiles are visible
// to every row; raw and extra tiles are filtered per tree node inside the softmax warps with a
// 64-bit column mask per row built from the plan (raw_lo, ancestor mask, scratch visibility).
//
// Warp roles (352 threads per CTA):
//   warp 0      TMA producer: pair S, the item's Q rows (through four ring slots, then copied into
//               TMEM) and this CTA's half of every tile's K entries x 512 dims (two 32 KB slots of
//               a 5-slot ring); pair O, the tile's entries x this CTA's 256 value columns (two
//               32 KB slots of a 4-slot ring).  All copies of a pair complete on its leader's
//               barriers (cta_group::2 TMA).
//   warp 1      both CTAs: allocate / free 512 TMEM columns (cta_group::2); the leader's lane 0
//               issues the pair's MMAs and releases ring slots and buffers with multicast commits
//   warps 2..9  pair S: Q rows into TMEM, then per tile the softmax, two threads per query row
//               (one per half of the tile's columns) sharing one running maximum; pair O: per
//               tile the (rare) O rescale, and at the end of an item O / l out through TMA stores
//               from a staging copy in the idle V ring
//   warp 10     lane 0: forwards this CTA's per-tile readiness to its pair leader (leader: local
//               arrive with expect_tx; follower: a 4-byte st.async), and moves P to pair O
// TMEM columns: pair S: S buffers at [0,128) and [128,256), Q at [256,512); pair O: O at [0,512).
// Every wait is bounded; on timeout the CTA records TV_ERR_TIMEOUT, sets the abort flag of all
// four CTAs, stops issuing work, drains its own copies and MMAs (bounded) and frees its TMEM.
// Launch chain.  On the contiguous dense path with up to kRankMax requests the kernel is a
// programmatic dependent of the kernel before it in the stream (in a round: the scratch pad) and
// ranks the requests itself in its prologue (from the lengths L, which that kernel does not
// write): it streams the prefix tiles while the scratch pad still runs, and waits for that
// kernel only where it reads what the round's earlier kernels wrote -- the softmax warps before
// the plan's masks (at the first item's first raw or extra tile; later items read them at their
// start), the producer before the scratch rows (the extra tile, each item's last), every thread
// before a global write -- and before it exits, so that its completion still implies theirs.  The lengths are read once, in
// the prologue, through L2.  Otherwise (larger batches, selection lists, page pools) the
// requests are ranked by order_kernel, which this kernel waits for before it starts.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "tv_attn_tc.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace tc {

using namespace sm100;

constexpr int kClusterCtas = 4;
constexpr int kSmxWarps = 8;                     // softmax / rescale warps, two threads per row
constexpr int kSigWarp = 2 + kSmxWarps;          // forwards per-tile readiness to the pair leader
constexpr int kThreads = 64 + 32 * kSmxWarps + 32;   // producer, MMA issuer, role warps, signal
constexpr int kSlotBytes = 32768;
constexpr int kSSlots = 5;      // pair S: K ring (a tile's K share is two slots of 4 x 64 dims)
constexpr int kQSlots = 4;      // pair S: an item's Q rows arrive through four ring slots
constexpr int kOSlots = 4;      // pair O: V ring (a tile's V share is two slots of 128 columns)
constexpr int kKSlices = 4;     // 64-dim K slices (64 entries x 128 B, 8 KB) per slot
constexpr int kVBlock = 16384;  // V slot: two 64-column blocks of 128 entries
constexpr int kPBytes = 32768;  // P of one tile for one CTA's rows: 128 rows x 128 entries bf16
constexpr int kPMsg = kPBytes + 128 * 4;   // P and the rows' rescale factors, sent as one copy
constexpr int kPBuf = 33 * 1024;           // a P buffer (1 KB aligned)
constexpr int kDp = 8;          // rows per section of the extra tile (D <= 8)
constexpr int kExtraEntries = 32;   // tree | C4 scratch | C128 scratch | zeros
constexpr int kRankMax = 2048;      // batches up to this size are ranked in the kernel's prologue

// The wait for the kernel this one depends on, at most once per thread (waited: this thread has
// waited, or the whole CTA did in the prologue); a repeated griddepcontrol.wait is not free.
__device__ __forceinline__ void pdl_wait_once(bool& waited) {
  if (!waited) {
    pdl_wait();
    waited = true;
  }
}
constexpr uint32_t kTmemQ = 256;     // pair S: Q columns
constexpr uint64_t kTimeoutNs = 2000000000ull;   // default bound of every wait
constexpr float kRescaleThreshold = 8.f;   // log2 units: P values stay below 2^8

enum TileKind { kC4 = 0, kC128 = 1, kRaw = 2, kExtra = 3 };

struct Params {
  CUtensorMap mQ, mO;   // [B][DH][512], box 64 x 128 x 1: Q rows in, O rows out
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
  int64_t rows_c4, rows_c128, rows_raw;   // row extents of the C4, C128 and raw maps
  uint64_t timeout_ns;   // bound of every wait (kTimeoutNs unless a test shortens it)
  int withhold_tile;     // test aid: the producers never issue this tile's K copies (-1: none)
};

struct Layout {
  int L, n4, n128, t0, nraw, T4, T128, Traw, T;
};

struct Tile {
  int kind, row0, valid, nqk;
};

__device__ __forceinline__ Layout layout_for(const Params& p, int L) {
  Layout y;
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
__device__ __forceinline__ Layout layout_of(const Params& p, int b) { return layout_for(p, p.L[b]); }

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
  // a programmatic dependent of the scratch-pad kernel: waits for it, then lets the attention
  // kernel start its prologue
  pdl_wait();
  pdl_launch_dependents();
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

// Shared memory.  The operand buffers differ between the two pairs; the barriers and small arrays
// sit at the same offsets in every CTA, so a commit or an asynchronous store of one pair can
// target the other pair's barriers by offset.
struct Header {
  uint64_t full[kSSlots];      // (pair leader) both CTAs' shares of a fill have landed
  uint64_t empty[kSSlots];     // the pair's MMAs are done with the slot
  uint64_t q_full;             // pair S (leader): both CTAs' Q rows are in TMEM (one per item)
  uint64_t q_local;            // pair S: this CTA's role warps have written their Q rows
  uint64_t q_tma;              // pair S: this CTA's Q rows have landed in the ring (TMA)
  uint64_t s_full[2];          // pair S: S_t is in TMEM
  uint64_t s_read[2];          // pair S: this CTA's softmax warps have read S_t (one per warp)
  uint64_t s_free[2];          // pair S (leader): both CTAs' softmax warps have read S_t
  uint64_t p_staged[2];        // pair S: this CTA's softmax warps have staged P_t (one per warp)
  uint64_t stage_free;         // pair S: the copy of the staged P_{t-1} has read the buffer
  uint64_t p_free[2];          // pair S: pair O's MMAs are done with the P buffer of parity t
  uint64_t p_in[2];            // pair O: the row partner's P_t and rescale factors have landed
  uint64_t p_local[2];         // pair O: this CTA's role warps have applied tile t's rescale
  uint64_t p_full[2];          // pair O (leader): both CTAs are ready for PV_t
  uint64_t pv_done;            // pair O: PV_t complete
  uint64_t o_full;             // pair O: every PV of the item complete (one per item)
  uint64_t o_free;             // pair O: the role warps have read the item's O out of TMEM
  uint64_t stage_full;         // pair O: the role warps have staged the item's O rows
  uint64_t v_free;             // pair O: the epilogue is done with the V ring
  uint64_t ml_full[2];         // pair O: [item parity] the row partner's final (m, l) landed
  uint64_t drain;
  uint32_t flag[4];            // (leader) landing words of the follower's 4-byte signals
  float xmax[2][2][128];       // pair S: [tile parity][column half][row] partial row maxima
  float xsum[2][128];          // pair S: [column half][row] partial row sums
  float ml[2][128][2];         // pair O: [item parity][row] final (m, l) sent by pair S
  int xok[2][2][4];            // pair S: [tile parity][column half][lane quadrant] carries on
  int xok_end[2][4];           // pair S: [column half][lane quadrant] carries on after an item
  uint32_t tmem;
  int abort;
  int32_t len[kRankMax];       // the requests' lengths L (read once, in the prologue)
  uint16_t order[kRankMax];    // requests by decreasing tile count (ranked in the prologue)
  uint16_t tiles[kRankMax];    // tile counts of the requests (clamped to 65535; ranking only)
};
// A P buffer holds 128 rows x 128 entries of bf16 P as two 64-entry panels (K-major, 128-byte
// swizzle), followed by the 128 rows' fp32 rescale factors.
constexpr int kBufBytes = (kSSlots * kSlotBytes + kPBuf) > (2 * kPBuf + kOSlots * kSlotBytes)
                              ? (kSSlots * kSlotBytes + kPBuf)
                              : (2 * kPBuf + kOSlots * kSlotBytes);
struct __align__(1024) Smem {
  // pair S: the K ring (kSSlots x 32 KB, which also carries each item's Q), then one P staging
  // buffer; pair O: two P buffers, then the V ring (kOSlots x 32 KB)
  uint8_t buf[kBufBytes];
  Header h;
};
static_assert(kQSlots * kSlotBytes == 8 * 16384 && kQSlots <= kSSlots, "Q takes four K slots");
static_assert(sizeof(Smem) <= 232448, "shared memory of one CTA exceeds the 227 KB limit");

// 3-D tile load into this CTA's shared memory, completing this CTA's own mbarrier.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t cluster_addr, uint32_t v,
                                             uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
          cluster_addr),
      "r"(v), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t cluster_addr, uint32_t a, uint32_t b,
                                            uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
          cluster_addr),
      "r"(a), "r"(b), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void fail(Smem& sm, int32_t* status) {
  if (atomicExch(&sm.h.abort, 1) == 0) {
    record_error(status, TV_ERR_TIMEOUT);
    // the other three CTAs stop waiting on this one
    const uint32_t me = cluster_rank();
    for (uint32_t r = 0; r < kClusterCtas; ++r)
      if (r != me) st_cluster_u32(mapa_cluster(smem_u32(&sm.h.abort), r), 1u);
  }
}

// A per-tile signal from a CTA to its pair leader: the leader arrives on its own barrier with
// expect_tx(4); the follower completes those 4 bytes with an asynchronous store into the leader's
// shared memory, which lands much sooner than a cluster-scope release-arrive.
__device__ __forceinline__ void signal_leader(Smem& sm, uint64_t* bar, uint32_t* flag, bool leader,
                                              uint32_t leader_rank, uint32_t value) {
  if (leader)
    mbar_arrive_expect_tx(bar, 4);
  else
    st_async_b32(mapa_cluster(smem_u32(flag), leader_rank), value,
                 mapa_cluster(smem_u32(bar), leader_rank));
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

// Split-KV partial row of (request, row, chunk); the bounds-checked build confines it to the
// workspace (row 0 on a violation).
// (rows past D*H -- the last row tile's padding -- are never stored and are not checked)
__device__ __forceinline__ int64_t part_row(const Params& p, int b, int grow, int chunk) {
  const int64_t i = ((int64_t)b * p.DH + grow) * p.n_chunks + chunk;
  if (grow >= p.DH) return i;
  return tv_in_range(i, 0, (int64_t)p.B * p.DH * p.n_chunks, p.status, 4) ? i : 0;
}

// Bounds-checked build: a prefix tile's first row lies inside its map (rows past it, in the
// padding of a ragged tile, are filled with zeros by the copy and masked).
__device__ __forceinline__ bool tile_rows_ok(const Params& p, int kind, int64_t row) {
  const int64_t n = kind == kC4 ? p.rows_c4 : kind == kC128 ? p.rows_c128 : p.rows_raw;
  return tv_in_range(row, 0, n, p.status, 1);
}

// A descriptor's start-address field is (address >> 4) in its low 14 bits; every operand here
// lies below 256 KB of shared memory, so adding (offset >> 4) never carries out of the field.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t byte_offset) {
  return desc + (uint64_t)(byte_offset >> 4);
}

// ---- work items ----------------------------------------------------------------------------------
// The grid holds one cluster per resident cluster slot; cluster c walks the longest-first list of
// work items (request, pair of row tiles, KV chunk) in a snake order: item c in round 0,
// G + (G-1-c) in round 1, 2G + c in round 2, ... for G clusters, so that every cluster gets a mix
// of long and short items.  Every role of every CTA of the cluster walks the same list.
struct Item {
  int b, rt, chunk, tb, te;
  Layout y;
};

__device__ __forceinline__ bool item_at(const Params& p, const Smem& sm, int k, uint32_t sub,
                                        Item& it) {
  const int G = (int)(gridDim.x / kClusterCtas), c = (int)(blockIdx.x / kClusterCtas);
  const int pos = (k & 1) ? k * G + (G - 1 - c) : k * G + c;
  if (pos >= p.B * p.n_chunks * p.n_pairs) return false;
  int x = pos;
  const int pair_idx = x % p.n_pairs;
  x /= p.n_pairs;
  it.chunk = x % p.n_chunks;
  if (p.order != nullptr) {
    it.b = p.order[x / p.n_chunks];
    it.y = layout_of(p, it.b);
  } else {
    it.b = sm.h.order[x / p.n_chunks];
    it.y = layout_for(p, sm.h.len[it.b]);
  }
  it.rt = 2 * pair_idx + (int)sub;
  if (it.y.T == 0) {   // capacity exceeded: nothing is computed for this request
    it.tb = it.te = 0;
    if (threadIdx.x == 0) record_error(p.status, TV_ERR_CAPACITY);
    return true;
  }
  it.tb = (int)((int64_t)it.y.T * it.chunk / p.n_chunks);
  it.te = (int)((int64_t)it.y.T * (it.chunk + 1) / p.n_chunks);
  return true;
}

// ---- ring of slots shared by a pair (the leader's full barriers count both CTAs' shares) ------
struct Ring {
  uint8_t* base;
  int n;         // slots
  int slot;
  uint32_t phase;
  __device__ void advance() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// ---- producer (warp 0, lane 0 does the copies) -------------------------------------------------
// Pair S: per item, its Q rows (eight 64-dim slices, two per slot) through the four ring slots on
// this CTA's own q_tma barrier (these fills complete the slots' full barriers without bytes), then
// this CTA's half of every tile's K entries (N/2 rows), all 512 dims, in two slots of four 64-dim
// slices.  Pair O: every entry of each tile for this CTA's 256 value columns, in two slots (one
// per 256-column group of O) of two 64-column blocks; rows past the tile's entry count rounded up
// to 64 are not loaded.
template <bool kPaged, bool kOverlap>
__device__ void producer(const Params& p, Smem& sm, bool role_s, uint32_t sub) {
  const int lane = threadIdx.x & 31;
  const uint32_t leader = cluster_rank() & ~1u;
  bool waited = !kOverlap;   // (without the overlap the prologue waited)
  Ring r{role_s ? sm.buf : sm.buf + 2 * kPBuf, role_s ? kSSlots : kOSlots, 0, 0};
  bool issued[kSSlots];
  uint32_t issued_phase[kSSlots];
#pragma unroll
  for (int i = 0; i < kSSlots; ++i) {
    issued[i] = false;
    issued_phase[i] = 0;
  }
  auto acquire = [&]() -> bool {
    if (!mbar_wait(&sm.h.empty[r.slot], r.phase ^ 1, &sm.h.abort, p.timeout_ns)) {
      if (lane == 0) fail(sm, p.status);
      return false;
    }
    return true;
  };
  auto leader_full = [&]() { return mapa_cluster(smem_u32(&sm.h.full[r.slot]), leader); };
  auto expect = [&](uint32_t bytes) {
    if (sub == 0) mbar_arrive_expect_tx(&sm.h.full[r.slot], 2 * bytes);
  };
  auto finish = [&](bool loads) {
    issued[r.slot] = loads;
    issued_phase[r.slot] = r.phase;
    r.advance();
  };
  bool ok = true;
  int q = 0;   // non-empty items so far
  Item it;
  for (int k = 0; ok && item_at(p, sm, k, sub, it); ++k) {
    if (it.tb >= it.te) continue;
    const int b = it.b;
    const Layout& y = it.y;
    const int tree_row = tv_in_range(b * p.D, 0, p.tree_rows, p.status, 2) ? b * p.D : 0;
    // pair O: the previous item's epilogue stages O in the V ring; its slots are free again
    // once the role warps report v_free
    if (!role_s && q > 0 && !mbar_wait(&sm.h.v_free, (q - 1) & 1, &sm.h.abort, p.timeout_ns)) {
      if (lane == 0) fail(sm, p.status);
      break;
    }
    ++q;
    if (role_s) {
      for (int j = 0; j < kQSlots && ok; ++j) {
        if (!acquire()) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (j == 0) mbar_arrive_expect_tx(&sm.h.q_tma, 8 * 16384);
          for (int s = 2 * j; s < 2 * j + 2; ++s)
            tma_load_3d(r.base + r.slot * kSlotBytes + (s & 1) * 16384, &p.mQ, 64 * s,
                        128 * it.rt, b, &sm.h.q_tma);
          if (sub == 0) mbar_arrive(&sm.h.full[r.slot]);
        }
        finish(false);
      }
    }
    // tile rows are computed one tile ahead, so that with paged pools the page-table reads are
    // in flight while the producer waits for slots
    auto row_of = [&](int t) -> int2 {
      int2 rw = make_int2(0, 0);
      if (t < it.tb || t >= it.te) return rw;
      const Tile x = tile_of(y, t);
      if (x.kind == kExtra) return rw;
      if (role_s) {
        rw.x = (int)tile_row<kPaged>(p, x.kind, b, x.row0 + (int)sub * (x.nqk / 2), y.t0);
      } else {
        rw.x = (int)tile_row<kPaged>(p, x.kind, b, x.row0, y.t0);
        rw.y = kPaged ? (int)tile_row<kPaged>(p, x.kind, b, x.row0 + 64, y.t0) : rw.x + 64;
      }
      return rw;
    };
    int2 cur = row_of(it.tb);
    for (int t = it.tb; t < it.te && ok; ++t) {
      const int2 next = row_of(t + 1);
      const Tile x = tile_of(y, t);
      if (kOverlap && x.kind == kExtra) pdl_wait_once(waited);   // the scratch rows
      for (int g = 0; g < 2 && ok; ++g) {
        if (!acquire()) {
          ok = false;
          break;
        }
        uint8_t* dst = r.base + r.slot * kSlotBytes;
        const uint32_t bar = leader_full();
        bool loads = true;
        if (role_s) {
          loads = t != p.withhold_tile;   // test aid: the MMA issuer's wait for it runs out
          if (lane == 0 && loads) {
            if (x.kind == kExtra) {
              // leader: tree rows | C4 scratch rows; follower: C128 scratch rows | zero rows
              expect(kKSlices * 2 * kDp * 128);
              for (int ks = 0; ks < kKSlices; ++ks) {
                const int xcol = 64 * (kKSlices * g + ks);
                uint8_t* d = dst + ks * 8192;
                if (sub == 0) {
                  tma_load_2d_pair(d, &p.mTreeK, xcol, tree_row, bar);
                  tma_load_2d_pair(d + kDp * 128, &p.mS4K, xcol, tree_row, bar);
                } else {
                  tma_load_2d_pair(d, &p.mS128K, xcol, tree_row, bar);
                  tma_load_2d_pair(d + kDp * 128, &p.mTreeK, xcol, p.tree_rows, bar);
                }
              }
            } else {
              const CUtensorMap* m =
                  x.kind == kC4 ? &p.mC4K : x.kind == kC128 ? &p.mC128K : &p.mRawK;
              expect(kSlotBytes);
              // (the follower loads the tile's second half, which may lie wholly in the padding
              // past the map: checked is the leader's first row; a failed check still issues the
              // copies, from row 0, so the barrier completes)
              const int row = (sub == 1 || tile_rows_ok(p, x.kind, cur.x)) ? cur.x : 0;
              for (int ks = 0; ks < kKSlices; ++ks)
                tma_load_2d_pair(dst + ks * 8192, m, 64 * (kKSlices * g + ks), row, bar);
            }
          }
        } else if (lane == 0) {
          const int col0 = 256 * g + 128 * (int)sub;
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
            const CUtensorMap* m =
                x.kind == kC4 ? &p.mC4V : x.kind == kC128 ? &p.mC128V : &p.mRawV;
            const int nvh = (x.nqk + 63) / 64;   // 64-row halves to load
            expect(nvh * 2 * 8192);
            for (int h = 0; h < nvh; ++h) {
              const int hr = h == 0 ? cur.x : cur.y;
              const int row = tile_rows_ok(p, x.kind, hr) ? hr : 0;
              for (int cb = 0; cb < 2; ++cb)
                tma_load_2d_pair(dst + cb * kVBlock + h * 8192, m, col0 + 64 * cb, row, bar);
            }
          }
        }
        finish(loads);
      }
      cur = next;
    }
  }
  // drain: no copy issued by the pair may still be in flight when the CTA exits (the leader's
  // full barriers count both CTAs' shares; the closing cluster barrier covers the follower)
  if (sub == 0 && lane == 0) {
    volatile int never = 0;
    for (int i = 0; i < r.n; ++i)
      if (issued[i]) mbar_wait(&sm.h.full[i], issued_phase[i], &never, p.timeout_ns / 4);
  }
}

// ---- pair leaders, lane 0 of warp 1: the MMAs ------------------------------------------------
// One thread issues every MMA of a pair, and a tcgen05.mma is accepted only about as fast as the
// issuing thread reaches it: the instructions between two MMAs are not hidden behind the tensor
// pipe.  So descriptors are built once, each MMA adds a compile-time offset, and the K-step loops
// are unrolled without run-time branches.  Tile counters run across items, so the parities of the
// per-tile barriers and buffers continue from one item to the next.
__device__ __forceinline__ bool wait_ring(const Params& p, Smem& sm, const Ring& r) {
  if (!mbar_wait(&sm.h.full[r.slot], r.phase, &sm.h.abort, p.timeout_ns)) {
    fail(sm, p.status);
    return false;
  }
  tc_fence_after();
  return true;
}

// Pair S: S_t = Q K_t^T into S buffer t & 1 (M = 256, N = the tile's entries, K = 512: A = Q from
// TMEM columns [256, 512), B = K from the ring).
__device__ void mma_s(const Params& p, Smem& sm) {
  const uint32_t tmem = sm.h.tmem;
  const uint16_t pair = 0x3;
  Ring r{sm.buf, kSSlots, 0, 0};
  const uint64_t ring_desc = smem_desc_sw128(smem_u32(sm.buf), 16, 1024);
  int g = 0, q = 0;   // tiles and non-empty items so far
  bool ok = true;
  Item it;
  for (int k = 0; ok && item_at(p, sm, k, 0, it); ++k) {
    const int n = it.te - it.tb;
    if (n <= 0) continue;
    if (!mbar_wait(&sm.h.q_full, q & 1, &sm.h.abort, p.timeout_ns)) {
      fail(sm, p.status);
      break;
    }
    tc_fence_after();
    ++q;
    // Q is in both CTAs' TMEM: the ring slots that carried it go back to the producers
    for (int i = 0; i < kQSlots; ++i) {
      mma2_commit_mc(&sm.h.empty[r.slot], pair);
      r.advance();
    }
    for (int i = 0; i < n && ok; ++i, ++g) {
      const Tile x = tile_of(it.y, it.tb + i);
      const uint32_t idS = idesc_bf16_f32(256, x.nqk, 0, 0);
      const uint32_t d_s = tmem + 128 * (g & 1);
      // both CTAs' softmax warps have read S_{g-2} out of this buffer
      if (g >= 2 &&
          !mbar_wait(&sm.h.s_free[g & 1], ((g - 2) >> 1) & 1, &sm.h.abort, p.timeout_ns)) {
        fail(sm, p.status);
        ok = false;
        break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!wait_ring(p, sm, r)) {
          ok = false;
          break;
        }
        const uint64_t kd = desc_add(ring_desc, (uint32_t)r.slot * kSlotBytes);
#pragma unroll
        for (int m = 0; m < 4 * kKSlices; ++m)
          mma2_ts(d_s, tmem + kTmemQ + 8 * (4 * kKSlices * h + m),
                  desc_add(kd, (m >> 2) * 8192 + 32 * (m & 3)), idS, (h | m) ? 1u : 0u);
        mma2_commit_mc(&sm.h.empty[r.slot], pair);
        r.advance();
      }
      if (!ok) break;
      mma2_commit_mc(&sm.h.s_full[g & 1], pair);
    }
  }
  // drain every MMA this thread issued before TMEM is released
  mma2_commit_mc(&sm.h.drain, 0x1);
  volatile int never = 0;
  mbar_wait(&sm.h.drain, 0, &never, p.timeout_ns / 4);
}

// Pair O: O[:, 256j .. 256j+255] += P_t V_t[:, 256j .. 256j+255] for j = 0, 1 (M = 256, N = 256,
// K = the tile's entries: A = P from the P buffer of parity t, B = V from the ring).  An item's
// first PV waits until the previous item's O has left TMEM.
__device__ void mma_o(const Params& p, Smem& sm) {
  const uint32_t tmem = sm.h.tmem;
  const uint16_t pair = 0xC, pair_s = 0x3;
  Ring r{sm.buf + 2 * kPBuf, kOSlots, 0, 0};
  const uint64_t p_desc = smem_desc_sw128(smem_u32(sm.buf), 16, 1024);
  const uint64_t ring_desc = smem_desc_sw128(smem_u32(r.base), kVBlock, 1024);
  const uint32_t idO = idesc_bf16_f32(256, 256, 0, 1);
  int g = 0, q = 0;
  bool ok = true;
  Item it;
  for (int k = 0; ok && item_at(p, sm, k, 0, it); ++k) {
    const int n = it.te - it.tb;
    if (n <= 0) continue;
    if (q > 0 && !mbar_wait(&sm.h.o_free, (q - 1) & 1, &sm.h.abort, p.timeout_ns)) {
      fail(sm, p.status);
      break;
    }
    for (int i = 0; i < n && ok; ++i, ++g) {
      const Tile x = tile_of(it.y, it.tb + i);
      const int nks = x.nqk / 16;
      if (!mbar_wait(&sm.h.p_full[g & 1], (g >> 1) & 1, &sm.h.abort, p.timeout_ns)) {
        fail(sm, p.status);
        ok = false;
        break;
      }
      tc_fence_after();
      // P of this tile: two 64-entry panels of 128 rows x 128 B (K-major, 128-byte swizzle)
      const uint64_t pd = desc_add(p_desc, (uint32_t)(g & 1) * kPBuf);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (!wait_ring(p, sm, r)) {
          ok = false;
          break;
        }
        const uint64_t vd = desc_add(ring_desc, (uint32_t)r.slot * kSlotBytes);
        const uint32_t od = tmem + 256 * j;
        if (nks == 8) {
          mma2_ss(od, pd, vd, idO, i > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 1; ks < 8; ++ks)
            mma2_ss(od, desc_add(pd, (ks >> 2) * 16384 + 32 * (ks & 3)),
                    desc_add(vd, 2048 * ks), idO, 1u);
        } else {
          for (int ks = 0; ks < nks; ++ks)
            mma2_ss(od, desc_add(pd, (ks >> 2) * 16384 + 32 * (ks & 3)),
                    desc_add(vd, 2048 * ks), idO, (i > 0 || ks > 0) ? 1u : 0u);
        }
        mma2_commit_mc(&sm.h.empty[r.slot], pair);
        r.advance();
      }
      if (!ok) break;
      mma2_commit_mc(&sm.h.pv_done, pair);
      mma2_commit_mc(&sm.h.p_free[g & 1], pair_s);   // pair S may overwrite this P buffer
    }
    if (!ok) break;
    mma2_commit_mc(&sm.h.o_full, pair);
    ++q;
  }
  mma2_commit_mc(&sm.h.drain, (uint16_t)(1u << cluster_rank()));
  volatile int never = 0;
  mbar_wait(&sm.h.drain, 0, &never, p.timeout_ns / 4);
}

// ---- signal warps (lane 0) -----------------------------------------------------------------------
// Pair S: Q in this CTA's TMEM -> q_full; S_t read by this CTA's softmax warps -> s_free; and the
// P transfer: once this CTA's softmax warps have staged P_t (and pair O's MMAs are done with the
// destination buffer, the PV of tile t-2), one bulk copy takes the staging buffer to the row
// partner's P buffer of parity t and completes its p_in barrier; once the copy has read the
// staging buffer, P_{t+1} may be staged there.
// Pair O: tile t's rescale applied and P_t landed in this CTA -> p_full.
// A follower cannot signal tile t + 2 before the leader's barrier of tile t completed (the
// pipelines make the later signal depend on the earlier one), so two parities suffice.
__device__ void signal_s(const Params& p, Smem& sm, uint32_t rank) {
  const uint32_t leader = rank & ~1u;
  const bool is_leader = (rank & 1u) == 0;
  const uint32_t partner = rank + 2;
  const uint32_t dst0 = mapa_cluster(smem_u32(sm.buf), partner);
  const uint32_t bar0 = mapa_cluster(smem_u32(&sm.h.p_in[0]), partner);
  const uint32_t src0 = smem_u32(sm.buf + kSSlots * kSlotBytes);
  int g = 0, q = 0;
  Item it;
  for (int k = 0; item_at(p, sm, k, rank & 1u, it); ++k) {
    const int n = it.te - it.tb;
    if (n <= 0) continue;
    if (!mbar_wait(&sm.h.q_local, q & 1, &sm.h.abort, p.timeout_ns)) {
      fail(sm, p.status);
      break;
    }
    ++q;
    signal_leader(sm, &sm.h.q_full, &sm.h.flag[0], is_leader, leader, (uint32_t)q);
    bool ok = true;
    for (int i = 0; i < n; ++i, ++g) {
      const int sb = g & 1;
      const uint32_t ph = (g >> 1) & 1;
      if (!mbar_wait(&sm.h.s_read[sb], ph, &sm.h.abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      signal_leader(sm, &sm.h.s_free[sb], &sm.h.flag[1 + sb], is_leader, leader, (uint32_t)g);
      if (!mbar_wait(&sm.h.p_staged[sb], ph, &sm.h.abort, p.timeout_ns) ||
          (g >= 2 && !mbar_wait(&sm.h.p_free[sb], ((g - 2) >> 1) & 1, &sm.h.abort,
                                p.timeout_ns))) {
        ok = false;
        break;
      }
      asm volatile(
          "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
          "[%3];" ::"r"(dst0 + (uint32_t)sb * kPBuf),
          "r"(src0), "r"((uint32_t)kPMsg), "r"(bar0 + (uint32_t)sb * 8)
          : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // the copy has read the staging buffer: P_{g+1} may be staged there
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      mbar_arrive(&sm.h.stage_free);
    }
    if (!ok) {
      fail(sm, p.status);
      break;
    }
  }
  // every copy has read its source before the CTA moves on
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ void signal_o(const Params& p, Smem& sm, uint32_t rank) {
  const uint32_t leader = rank & ~1u;
  const bool is_leader = (rank & 1u) == 0;
  int g = 0;
  Item it;
  for (int k = 0; item_at(p, sm, k, rank & 1u, it); ++k) {
    const int n = it.te - it.tb;
    bool ok = true;
    for (int i = 0; i < n; ++i, ++g) {
      if (!mbar_wait(&sm.h.p_local[g & 1], (g >> 1) & 1, &sm.h.abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      signal_leader(sm, &sm.h.p_full[g & 1], &sm.h.flag[1 + (g & 1)], is_leader, leader,
                    (uint32_t)g);
    }
    if (!ok) {
      fail(sm, p.status);
      break;
    }
  }
}

// ---- pair S role warps: Q into TMEM, then the softmax ------------------------------------------
// Warp w (2..9) serves TMEM lane quadrant w % 4 (rows 32*(w%4) .. +31) and column half
// ch = (w-2)/4 of each tile.  The two threads of a row exchange their partial row maxima through
// shared memory once per tile and apply the same running maximum.
__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
}

// The plan's visibility of one query row: (raw_lo << 32) | extra-tile mask (bit j: entry j of
// the extra tile is visible); 0 for a row past D*H (grow < 0).  With wait, first the wait for the
// kernel this one depends on (the plan's results come from an earlier kernel).  Not inlined: it
// stays out of the softmax's tile loop.
__device__ __noinline__ uint64_t row_masks(const Params& p, int b, int grow, int L, bool wait) {
  if (wait) pdl_wait();
  if (grow < 0) return 0;
  const int v = grow / p.H;
  const int64_t i = (int64_t)b * p.D + v;
  const uint64_t an = p.anc[i];
  const int raw_lo = p.raw_lo[i];
  const uint64_t v4 = (p.comp_mask & TV_COMP_C4) ? p.vis4[i] : 0;
  const uint64_t v128 = (p.comp_mask & TV_COMP_C128) ? p.vis128[i] : 0;
  uint32_t extra_mask = 0;
  for (int u = 0; u < p.D; ++u) {
    if ((an >> u) & 1ull) {
      const int dep = __popcll(an & ((1ull << u) - 1ull));
      if (L + dep >= raw_lo) extra_mask |= 1u << u;
    }
    if ((v4 >> u) & 1ull) extra_mask |= 1u << (kDp + u);
    if ((v128 >> u) & 1ull) extra_mask |= 1u << (2 * kDp + u);
  }
  return ((uint64_t)(uint32_t)raw_lo << 32) | extra_mask;
}

template <bool kOverlap>
__device__ void softmax_s(const Params& p, Smem& sm, uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int ch = (warp - 2) >> 2;
  const int row = 32 * quad + lane;
  const uint32_t tmem = sm.h.tmem;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const float sl2 = p.scale_log2;
  const uint32_t partner = rank + 2;
  // this row's line in the P staging buffers (panel ch, 128-byte swizzle: 16-byte chunk c of the
  // row at chunk c ^ (row & 7)); the signal warp copies each staged buffer to the row partner
  // (the CTA of pair O with the same rows)
  uint8_t* const p_line = sm.buf + kSSlots * kSlotBytes + ch * 16384 + (row >> 3) * 1024 +
                          (row & 7) * 128;
  int g = 0, q = 0;
  bool ok = true;
  bool waited = !kOverlap;   // this thread has waited for the kernel it depends on
  Item it;
  for (int k = 0; ok && item_at(p, sm, k, rank & 1u, it); ++k) {
    const int n = it.te - it.tb;
    if (n <= 0) continue;
    const int b = it.b;
    const int grow = 128 * it.rt + row;
    const bool row_ok = grow < p.DH;
    const Layout& y = it.y;
    // Q: the producer's TMA put this item's Q rows in the ring as eight slices of 128 rows x 64
    // dims (128-byte swizzle), slices 2j and 2j+1 in the j-th slot after the ring position the
    // item started at (2 slots per earlier tile, 4 per earlier item); this thread moves dims
    // 256ch .. 256ch+255 of its row (slices 4ch .. 4ch+3) into TMEM columns 256 + 128ch .., where
    // column c holds dims 2c (low half) and 2c + 1, the A-operand layout of a kind::f16 MMA
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.h.q_tma, q & 1, &sm.h.abort, p.timeout_ns))) {
      fail(sm, p.status);
      ok = false;   // the first tile's exchange lets the row's other warp leave too
    }
    const int q_slot0 = (kQSlots * q + 2 * g) % kSSlots;   // ring position at the item's start
#pragma unroll 1
    for (int sl = 0; sl < 4 && ok; ++sl) {
      const int s = 4 * ch + sl;
      const uint8_t* line = sm.buf + ((q_slot0 + (s >> 1)) % kSSlots) * kSlotBytes +
                            (s & 1) * 16384 + (row >> 3) * 1024 + (row & 7) * 128;
      uint32_t qv[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(line + ((c ^ (row & 7)) << 4));
        qv[4 * c] = v.x;
        qv[4 * c + 1] = v.y;
        qv[4 * c + 2] = v.z;
        qv[4 * c + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + kTmemQ + 128 * ch + 32 * sl, qv);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(&sm.h.q_local);
    ++q;

    // per-row visibility of the raw tail and of the extra tile, from the plan's masks; read at
    // the item's first raw or extra tile, after the wait for the round's earlier kernels (the
    // prefix tiles before it need no mask); at the item's start once this thread has waited
    int raw_lo = 0;
    uint32_t extra_mask = 0;   // bit j: entry j of the extra tile is visible
    bool masks = false;
    auto load_masks = [&]() {
      const uint64_t rm = row_masks(p, b, row_ok ? grow : -1, y.L, !waited);
      waited = true;
      masks = true;
      raw_lo = (int)(rm >> 32);
      extra_mask = (uint32_t)rm;
    };
    if (waited) load_masks();

    float m_ref = -INFINITY, l_run = 0.f;
    // The two warps of a row (column halves) meet at one named barrier per tile.  A warp whose
    // bounded wait ran out still takes each barrier until both warps leave the tile loop together
    // (each tile's exchange carries both warps' flags), so neither waits on the other forever.
    for (int i = 0; i < n; ++i, ++g) {
      const Tile x = tile_of(y, it.tb + i);
      const int sb = g & 1;
      const int c0 = 64 * ch;   // first S column of this thread
      if (ok && !__all_sync(0xffffffffu, mbar_wait(&sm.h.s_full[sb], (g >> 1) & 1, &sm.h.abort,
                                                   p.timeout_ns))) {
        fail(sm, p.status);
        ok = false;
      }
      float s[64];
      float raw_max = -INFINITY;
      if (ok) {
        tc_fence_after();
        {
          uint32_t* sr = reinterpret_cast<uint32_t*>(s);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            if (c0 + 32 * c < x.nqk)
              tmem_ld32(tmem + lane_base + 128 * sb + c0 + 32 * c,
                        *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
          tmem_wait_ld();
        }
        // S_t is in registers: its buffer may take S_{t+2}
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.h.s_read[sb]);
        // visible columns of this thread as a 64-bit mask: a range [lo, hi) of the tile's
        // entries (prefix tiles: all valid entries; raw tiles: positions >= raw_lo), or the
        // extra tile's per-node bits.  One code path for every tile kind.
        if (kOverlap && x.kind >= kRaw && !masks) load_masks();
        uint64_t vmask;
        if (x.kind == kExtra) {
          vmask = c0 == 0 ? (uint64_t)extra_mask : 0ull;
        } else {
          const int hi = min(64, max(0, x.valid - c0));
          const int lo = x.kind == kRaw ? min(hi, max(0, raw_lo - x.row0 - c0)) : 0;
          vmask = (hi == 64 ? ~0ull : ((1ull << hi) - 1ull)) & ~((1ull << lo) - 1ull);
        }
        const uint32_t vlo = (uint32_t)vmask, vhi = (uint32_t)(vmask >> 32);
        // row maximum of the visible raw logits (scale > 0, so the scaled maximum follows); the
        // softmax warps' instructions compete with the MMA issuer for the SM's issue slots, so a
        // fully visible half-row (most tiles) takes a three-input maximum tree
        if (vmask == ~0ull) {
          float t[22];
#pragma unroll
          for (int j = 0; j < 21; ++j) t[j] = max3f(s[3 * j], s[3 * j + 1], s[3 * j + 2]);
          t[21] = s[63];
          float u[8];
#pragma unroll
          for (int j = 0; j < 7; ++j) u[j] = max3f(t[3 * j], t[3 * j + 1], t[3 * j + 2]);
          u[7] = t[21];
          raw_max = max3f(max3f(u[0], u[1], u[2]), max3f(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
        } else {
          float mx[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) mx[j] = -INFINITY;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const bool vis = ((j < 32 ? vlo : vhi) >> (j & 31)) & 1u;
            s[j] = vis ? s[j] : -INFINITY;
            mx[j & 7] = fmaxf(mx[j & 7], s[j]);
          }
          raw_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                          fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        }
      }
      sm.h.xmax[sb][ch][row] = raw_max;
      if (lane == 0) sm.h.xok[sb][ch][quad] = ok ? 1 : 0;
      pair_sync(quad);
      raw_max = fmaxf(raw_max, sm.h.xmax[sb][ch ^ 1][row]);
      if (ok && !sm.h.xok[sb][ch ^ 1][quad]) {   // the row's other warp gave up
        fail(sm, p.status);
        ok = false;
      }
      if (!ok) break;
      const float mt = raw_max * sl2;
      const bool grow_max = mt > m_ref + kRescaleThreshold;
      const float m_new = grow_max ? mt : m_ref;
      // exactly 1 unless the maximum grows past a finite reference: pair O rescales O by it
      const float alpha = (grow_max && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
      const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
      // exponent arguments and partial sums two at a time (packed fp32 pairs)
      const uint64_t scale2 = pack_f32x2(sl2, sl2), shift2 = pack_f32x2(neg_m, neg_m);
      uint64_t sum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float a0, a1;
        unpack_f32x2(fma_f32x2(pack_f32x2(s[2 * j], s[2 * j + 1]), scale2, shift2), a0, a1);
        const float p0 = ex2_approx(a0);
        const float p1 = ex2_approx(a1);
        sum2[j & 1] = add_f32x2(sum2[j & 1], pack_f32x2(p0, p1));
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        pk[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      float s0, s1, s2, s3;
      unpack_f32x2(sum2[0], s0, s1);
      unpack_f32x2(sum2[1], s2, s3);
      const float tsum = (s0 + s1) + (s2 + s3);
      l_run = l_run * alpha + tsum;
      m_ref = m_new;
      // the copy of P_{g-1} has read the staging buffer
      if (g >= 1 && !__all_sync(0xffffffffu, mbar_wait(&sm.h.stage_free, (g - 1) & 1,
                                                       &sm.h.abort, p.timeout_ns))) {
        fail(sm, p.status);
        ok = false;
        continue;   // the next tile's exchange lets the row's other warp leave too
      }
      uint8_t* const line = p_line;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(line + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (ch == 0)
        reinterpret_cast<float*>(sm.buf + kSSlots * kSlotBytes + kPBytes)[row] = alpha;
      // the copy reads the staging buffer through the async proxy
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.h.p_staged[sb]);
    }
    // combine the two partial row sums (both threads of a row share m_ref); both warps of a row
    // take this barrier, whatever happened in the tile loop
    sm.h.xsum[ch][row] = l_run;
    if (lane == 0) sm.h.xok_end[ch][quad] = ok ? 1 : 0;
    pair_sync(quad);
    const float l_tot = l_run + sm.h.xsum[ch ^ 1][row];
    ok = ok && sm.h.xok_end[ch ^ 1][quad];   // both warps of the row leave together
    pair_sync(quad);   // both have read xsum before the next item overwrites it
    if (!ok) break;
    if (ch == 0) {
      const int mb = (q - 1) & 1;
      st_async_v2(mapa_cluster(smem_u32(&sm.h.ml[mb][row][0]), partner), __float_as_uint(m_ref),
                  __float_as_uint(l_tot), mapa_cluster(smem_u32(&sm.h.ml_full[mb]), partner));
      if (kOverlap) pdl_wait_once(waited);   // no write before the kernel depended on completed
      if (row_ok && p.n_chunks == 1)
        p.lse[(int64_t)b * p.DH + grow] =
            l_tot > 0.f ? (m_ref + log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

// ---- pair O role warps: per-tile rescale, then each item's epilogue ------------------------------
// Warp w (2..9) serves lane quadrant w % 4 and O columns 256ch .. 256ch+255, ch = (w-2)/4.
template <bool kOverlap>
__device__ void rescale_epilogue_o(const Params& p, Smem& sm, uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int ch = (warp - 2) >> 2;
  const int row = 32 * quad + lane;
  const uint32_t tmem = sm.h.tmem;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const bool arms = row == 0 && ch == 0;   // the thread that arms the receiving barriers
  const int d = 512;
  int g = 0, q = 0;
  bool waited = !kOverlap;   // (without the overlap the prologue waited)
  Item it;
  for (int k = 0; item_at(p, sm, k, rank & 1u, it); ++k) {
    const int n = it.te - it.tb;
    const int b = it.b;
    const int grow = 128 * it.rt + row;
    const bool row_ok = grow < p.DH;
    if (n <= 0) {
      if (it.y.T > 0 && p.n_chunks > 1 && row_ok) {   // an empty KV chunk: l = 0
        if (kOverlap) pdl_wait_once(waited);   // no write before the kernel depended on completed
        float* prow = p.part + part_row(p, b, grow, it.chunk) * (d + 4);
        for (int c = 0; c < 256; c += 4)
          *reinterpret_cast<float4*>(prow + 256 * ch + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ch == 0) {
          prow[d] = -INFINITY;
          prow[d + 1] = 0.f;
        }
      }
      continue;
    }
    const int mb = q & 1;
    if (arms) mbar_arrive_expect_tx(&sm.h.ml_full[mb], 128 * 8);
    for (int i = 0; i < n; ++i, ++g) {
      const int sb = g & 1;
      if (arms) mbar_arrive_expect_tx(&sm.h.p_in[sb], kPMsg);
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&sm.h.p_in[sb], (g >> 1) & 1, &sm.h.abort, p.timeout_ns))) {
        fail(sm, p.status);
        return;
      }
      const float alpha = reinterpret_cast<const float*>(sm.buf + sb * kPBuf + kPBytes)[row];
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        // O must hold every earlier PV of the item before it is rescaled (an item's first tile
        // always sends 1)
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sm.h.pv_done, (g - 1) & 1, &sm.h.abort, p.timeout_ns))) {
          fail(sm, p.status);
          return;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t r[32];
          const uint32_t col = tmem + lane_base + 256 * ch + 32 * c;
          tmem_ld32(col, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st32(col, r);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.h.p_local[sb]);
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.h.o_full, q & 1, &sm.h.abort, p.timeout_ns)) ||
        !__all_sync(0xffffffffu,
                    mbar_wait(&sm.h.ml_full[mb], (q >> 1) & 1, &sm.h.abort, p.timeout_ns))) {
      fail(sm, p.status);
      return;
    }
    ++q;
    tc_fence_after();
    // no write before the kernel this one depends on has completed (at once here: the item's
    // extra tile was loaded after that wait)
    if (kOverlap) pdl_wait_once(waited);
    const float m = sm.h.ml[mb][row][0], l = sm.h.ml[mb][row][1];
    if (p.n_chunks == 1) {
      // O leaves through shared memory and TMA stores: the V ring (idle from o_full until this
      // CTA's producer sees o_free) takes this CTA's 128 rows x 512 columns as eight 64-column
      // boxes with the 128-byte swizzle (16-byte chunk c of a row at c ^ (row & 7)); rows past
      // D*H fall outside the map and are not stored
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* stage = sm.buf + 2 * kPBuf;
      for (int c = 0; c < 256 / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + 256 * ch + 32 * c, r);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * inv,
                                                         __uint_as_float(r[2 * j + 1]) * inv);
          w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const int col = 256 * ch + 32 * c;   // O column of w[0]
        uint8_t* line = stage + (col >> 6) * 16384 + row * 128;
        const int cc0 = (col & 63) >> 3;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(line + (((cc0 + j) ^ (row & 7)) << 4)) =
              make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      }
      fence_proxy_async_smem();
      // O is out of TMEM (the next item's PV may start) and staged
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.h.o_free);
        mbar_arrive(&sm.h.stage_full);
      }
      // one thread stores the boxes once every warp has staged its rows (a bounded wait, not a
      // CTA barrier: a warp that gave up never arrives), then frees the V ring
      if (warp == 2 && lane == 0) {
        if (!mbar_wait(&sm.h.stage_full, (q - 1) & 1, &sm.h.abort, p.timeout_ns)) {
          fail(sm, p.status);
          return;
        }
        if (tv_in_range(b, 0, p.B, p.status, 3) && tv_in_range(128 * it.rt, 0, p.DH, p.status, 3))
          for (int j = 0; j < 8; ++j)
            asm volatile(
                "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::
                    "l"(reinterpret_cast<uint64_t>(&p.mO)),
                "r"(64 * j), "r"(128 * it.rt), "r"(b), "r"(smem_u32(stage + j * 16384))
                : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        mbar_arrive(&sm.h.v_free);
      }
      continue;
    } else {
      float* prow = p.part + part_row(p, b, grow, it.chunk) * (d + 4);
      for (int c = 0; c < 256 / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + 256 * ch + 32 * c, r);
        tmem_wait_ld();
        if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(prow + 256 * ch + 32 * c);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
      if (row_ok && ch == 0) {
        prow[d] = m;
        prow[d + 1] = l;
      }
    }
    // O is out of TMEM: the next item's PV may start; the V ring was not used
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.h.o_free);
    if (warp == 2 && lane == 0) mbar_arrive(&sm.h.v_free);
  }
}

// kPaged: the persistent cache is in page pools (C4 tiles through the page table, C128 entries
// and the raw tail from gathered copies); a separate instantiation keeps the contiguous path's
// producer free of the page-table work.  kOverlap: the launch chain's overlap with the kernel
// before this one (the kernel ranks the requests itself and waits late); without it, the
// instantiation waits in its prologue and keeps the late-wait checks out of its tile loops.
template <bool kPaged, bool kOverlap>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // the swizzled operand tiles need 1 KB alignment; the dynamic window starts 1 KB aligned
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    pdl_wait();
    if (threadIdx.x == 0) record_error(p.status, TV_ERR_CUDA);
    return;
  }
  pdl_launch_dependents();   // the acceptance walk reads nothing this kernel writes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (kOverlap && warp >= 2) {
    // the requests' lengths and tile counts for the ranking below, read through L2 (there is no
    // dependency wait before this read; the kernel before this one does not write L) by the
    // role warps while warps 0 and 1 set up the barriers and TMEM
    for (int j = (int)threadIdx.x - 64; j < p.B; j += (int)blockDim.x - 64) {
      const int L = __ldcg(p.L + j);
      sm.h.len[j] = L;
      sm.h.tiles[j] = (uint16_t)min(layout_for(p, L).T, 65535);
    }
  }
  // clusters of 4 consecutive CTAs; rank = 2 * (0: pair S, 1: pair O) + (row tile & 1)
  const uint32_t rank = blockIdx.x & 3;
  const bool role_s = rank < 2;
  const uint32_t sub = rank & 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSSlots; ++i) {
      mbar_init(&sm.h.full[i], 1);
      mbar_init(&sm.h.empty[i], 1);
    }
    mbar_init(&sm.h.q_full, 1);
    mbar_init(&sm.h.q_local, kSmxWarps);
    mbar_init(&sm.h.q_tma, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.h.s_full[i], 1);
      mbar_init(&sm.h.s_read[i], kSmxWarps);
      mbar_init(&sm.h.s_free[i], 1);
      mbar_init(&sm.h.p_staged[i], kSmxWarps);
      mbar_init(&sm.h.p_free[i], 1);
      mbar_init(&sm.h.p_in[i], 1);
      mbar_init(&sm.h.p_local[i], kSmxWarps);
      mbar_init(&sm.h.p_full[i], 1);
      mbar_init(&sm.h.ml_full[i], 1);
    }
    mbar_init(&sm.h.pv_done, 1);
    mbar_init(&sm.h.o_full, 1);
    mbar_init(&sm.h.o_free, kSmxWarps);
    mbar_init(&sm.h.stage_free, 1);
    mbar_init(&sm.h.stage_full, kSmxWarps);
    mbar_init(&sm.h.v_free, 1);
    mbar_init(&sm.h.drain, 1);
    sm.h.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(role_s ? &p.mQ : &p.mC4V);
    prefetch_tmap(role_s ? &p.mC4K : &p.mRawV);
  }
  if (warp == 1) {
    tmem_alloc2(&sm.h.tmem, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync();   // every CTA's barriers exist before any remote arrive, store or pair MMA
  tc_fence_after();
  if (kOverlap) {
    // rank the requests here (longest first, ties by index; the same order as order_kernel);
    // the cluster barrier above made every thread's tile counts visible
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int tb = sm.h.tiles[b];
      int r = 0;
      for (int j = 0; j < p.B; ++j) {
        const int tj = sm.h.tiles[j];
        r += (tj > tb || (tj == tb && j < b)) ? 1 : 0;
      }
      sm.h.order[r] = (uint16_t)b;
    }
    __syncthreads();
  } else {
    // a programmatic dependent of the ranking kernel: the set-up above overlaps it; every read
    // of the round's inputs comes after it has completed
    pdl_wait();
  }

  if (warp == 0) {
    producer<kPaged, kOverlap>(p, sm, role_s, sub);
  } else if (warp == 1) {
    if (lane == 0 && sub == 0) {
      if (role_s)
        mma_s(p, sm);
      else
        mma_o(p, sm);
    }
    __syncwarp();
  } else if (warp == kSigWarp) {
    if (lane == 0) {
      if (role_s)
        signal_s(p, sm, rank);
      else
        signal_o(p, sm, rank);
    }
    __syncwarp();
  } else if (role_s) {
    softmax_s<kOverlap>(p, sm, rank);
  } else {
    rescale_epilogue_o<kOverlap>(p, sm, rank);
  }

  if (kOverlap) pdl_wait();   // this kernel completes only after the one it depends on
  tc_fence_before();
  cluster_sync();   // the leaders' MMAs are drained; every awaited remote store has landed
  // after that barrier all four CTAs see the same abort flag (fail() sets the others' flags
  // before its CTA arrives), so all take the same branch
  if (*reinterpret_cast<volatile int*>(&sm.h.abort)) {
    // a wait ran out in this cluster: give the copies and stores another CTA issued before it
    // stopped (asynchronous ones included) time to land while all four CTAs are still resident
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 50000) {
    }
    cluster_sync();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(sm.h.tmem, 512);
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

// Per device, once: the kernels' shared-memory attribute and the number of 4-CTA clusters that
// can be resident at a time (a plain host call that also stays out of any stream being captured).
// Returns 0 on a CUDA error.
int cluster_slots() {
  static std::mutex mu;
  static int slots[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (slots[dev] == 0) {
    using namespace tv::tc;
    const int smem = (int)sizeof(Smem);
    if (cudaFuncSetAttribute(attn_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(attn_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(attn_kernel<true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<false, false>, &cfg) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
      }
      n = sms / kClusterCtas > 0 ? sms / kClusterCtas : 1;
    }
    slots[dev] = n;
  }
  return slots[dev];
}

// Number of KV chunks per request.  Clusters of 4 CTAs run one per resident cluster slot; a
// cluster costs about (its tiles + 4) tile-times (Q into TMEM, the first K and V fills, the O
// epilogue).  With T the largest tile count the capacities allow, pick the chunk count that
// minimises waves x (ceil(T / n) + 4); a larger count must win by more than 10 % (splitting adds
// fp32 partials and a merge pass).
int tc_chunks(const tv_shape* s) {
  int slots = cluster_slots();
  if (slots <= 0) slots = 36;
  int64_t max_tiles = 1 + (s->tail_mode == TV_TAIL_WINDOW ? (s->W + 127) / 128 : 1);
  if (s->comp_mask & TV_COMP_C4) max_tiles += ((s->n_sel > 0 ? s->n_sel : s->c4_cap) + 127) / 128;
  if (s->comp_mask & TV_COMP_C128) max_tiles += (s->c128_cap + 127) / 128;
  const int64_t clusters1 = (int64_t)s->B * n_pairs_of(s);
  // makespan in tile periods: waves of items x (tiles per chunk + an item's fill and drain, about
  // kItemTiles tile periods); the fewest chunks within 10 % of the best (every chunk adds a
  // partial row per query row to write and merge)
  constexpr int64_t kItemTiles = 12;
  int64_t cost[65];
  int64_t best_cost = -1;
  const int n_max = (int)(max_tiles < 64 ? max_tiles : 64);
  for (int n = 1; n <= n_max; ++n) {
    const int64_t waves = (clusters1 * n + slots - 1) / slots;
    cost[n] = waves * ((max_tiles + n - 1) / n + kItemTiles);
    if (best_cost < 0 || cost[n] < best_cost) best_cost = cost[n];
  }
  for (int n = 1; n <= n_max; ++n)
    if (10 * cost[n] <= 11 * best_cost) return n;
  return 1;
}

// Test aid (tv_debug_attn_timeout): the bound of every wait and one KV tile whose K copies the
// producers withhold.
std::atomic<int64_t> g_timeout_ns{(int64_t)tv::tc::kTimeoutNs};
std::atomic<int32_t> g_withhold_tile{-1};

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
  p.rows_c4 = (int64_t)c4rows;
  p.rows_c128 = (int64_t)c128rows;
  p.rows_raw = (int64_t)rawrows;
  bool ok = make_map(&p.mQ, a.Q, 3, DH, B, 128) && make_map(&p.mO, a.O, 3, DH, B, 128);
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
  // null: ranked in the kernel's prologue, which then overlaps the kernel before it (the
  // contiguous dense path; a gather of selected or paged rows comes first otherwise)
  p.order = (s->B <= kRankMax && !gathered && !paged) ? nullptr : order;
  p.part = reinterpret_cast<float*>(ws + pre_partial_bytes(s));
  p.status = a.status;
  p.timeout_ns = (uint64_t)g_timeout_ns.load();
  p.withhold_tile = g_withhold_tile.load();
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
  // larger batches: one CTA ranks all requests (B <= 12288 fits its default shared memory)
  if (p.order != nullptr) {
    if (tv::launch_pdl(order_kernel, dim3(1), dim3(1024), (size_t)s->B * sizeof(int), stream, p,
                       order) != cudaSuccess)
      return tv_check_launch("tv_tree_verify_attn (tcgen05 schedule launch)");
    if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05 schedule)")) return rc;
  }
  if (cluster_slots() <= 0)
    return tv_check_launch("tv_tree_verify_attn (tcgen05 kernel attributes)");
  const size_t smem = sizeof(Smem);
  // persistent clusters: one per resident cluster slot, at most one per work item
  const int64_t items = (int64_t)s->B * p.n_chunks * p.n_pairs;
  const int64_t clusters = items < cluster_slots() ? items : cluster_slots();
  const unsigned grid = (unsigned)(clusters * kClusterCtas);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see the launch chain
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t le = paged                ? cudaLaunchKernelEx(&cfg, attn_kernel<true, false>, p)
                         : p.order == nullptr ? cudaLaunchKernelEx(&cfg, attn_kernel<false, true>, p)
                                              : cudaLaunchKernelEx(&cfg, attn_kernel<false, false>, p);
  if (le != cudaSuccess)
    return tv_check_launch("tv_tree_verify_attn (tcgen05 cluster launch)");
  if (int rc = tv_check_launch("tv_tree_verify_attn (tcgen05)")) return rc;
  if (p.n_chunks > 1)
    return tv_launch_merge<__nv_bfloat16>(s->B, DH, 512, p.n_chunks, p.part, a.O, a.lse, stream);
  return TV_OK;
}

extern "C" int tv_debug_attn_timeout(int64_t timeout_ns, int32_t withhold_tile) {
  if (timeout_ns <= 0 || withhold_tile < -1)
    return tv_set_error(TV_ERR_ARG, "tv_debug_attn_timeout: timeout_ns must be > 0 and "
                                    "withhold_tile >= -1");
  g_timeout_ns.store(timeout_ns);
  g_withhold_tile.store(withhold_tile);
  return TV_OK;
}
