/*
 * treeverify.h -- C ABI of libtreeverify.so: the target-verify hot path of tree-structured
 * speculative decoding over online-compressed (C4 / C128) attention, for NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
 * Efficient Inference" (arXiv 2609.24698), cited as [TSD-V4] with inferred section numbers
 * (§2.2 CSA/HCA compression, §3.1 branch-aware causality, §3.2 isolation, §4.1 three-stage
 * forward and verification plan, §4.2 scratch pad and refresh, §4.3 optimisations, §5.1 naming).
 *
 * One verify round is five calls on one stream, with no host synchronisation in between:
 *   tv_build_ancestor_mask -> tv_branch_compress -> tv_tree_verify_attn -> tv_accept_walk
 *   -> tv_refresh_commit
 * plus tv_prefill_compress, which builds the persistent compressed prefix of a fresh batch.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller (unless stated otherwise).
 *   The library allocates nothing; scratch space for the attention is the caller's workspace.
 * - Every call is asynchronous on the cudaStream_t it is given (0 = legacy default stream) and
 *   returns TV_OK once its kernels are enqueued, or a negative TV_ERR_* code, without launching
 *   anything, when the host-side arguments are invalid (null pointer, bad shape).  The reason of
 *   the last host-side error of the calling thread is available from tv_last_error_string().
 * - Stream order holds as for ordinary launches.  Inside the library, kernels are launched as
 *   programmatic dependents of the kernel before them and start early only after one of this
 *   library's own kernels that allows it; each waits before it reads that kernel's results or
 *   writes anything, and before it completes.  A caller's kernel placed just before a call and
 *   itself allowing early starts (griddepcontrol.launch_dependents) must not write the call's
 *   inputs after that point.
 * - Errors found on the device (a malformed tree, a capacity overflow, a bad selection index,
 *   a wait that ran out) are written to the caller's int32 *status word with first-error-wins
 *   semantics (the word is only ever changed from 0 to a negative code); read it after the
 *   stream has been synchronised.  The affected request's outputs are then unspecified, the
 *   other requests' outputs are valid.  Kernels never trap and every wait is bounded.
 * - Tree: node 0 is the root, the last accepted token, whose K/V and query are produced in this
 *   pass; parents[b][0] == -1 and 0 <= parents[b][v] < v (topological numbering); D counts the
 *   root ([TSD-V4] §5.1: s4_k1_d5 verifies 4 draft tokens plus the root with budget 5).
 *   Node v of request b sits at position L[b] + depth[b][v].
 * - Persistent state of request b (row-major, row length d elements, dtype of the shape):
 *     rawK/rawV  [B][raw_cap][d]   raw per-token K/V, rows 0 .. L[b]-1 committed
 *     c4K/c4V    [B][c4_cap][d]    C4 entries, rows 0 .. L[b]/4 - 1 valid
 *     c128K/V    [B][c128_cap][d]  C128 entries, rows 0 .. L[b]/128 - 1 valid
 *     L          [B] int32         committed length
 *   The number of valid compressed entries is always floor(L / m): there is no separate count.
 *   Rows beyond the valid ones are never read for their values but may be loaded; they must hold
 *   finite numbers (allocate the buffers zero-filled).
 * - Scratch pad ([TSD-V4] §4.2): scrK4/scrV4 and scrK128/scrV128 [B][D][d], one row per tree
 *   node; row v holds the compressed entry of the block that node v's token closes, or zeros.
 *   It is separate from the persistent state, which only tv_refresh_commit writes (with
 *   tv_shape.stage_chain, tv_branch_compress also stages rows past the committed length, which no
 *   call reads before tv_refresh_commit has made them part of the state).
 * - Compressor m (4 = C4, 128 = C128): block j covers positions m*j .. m*j+m-1; gate logit of
 *   token t is z_t = K_t . g_m (no scale); w = softmax(z) over the block; the entry is
 *   (sum_t w_t K_t, sum_t w_t V_t), computed in fp32 and stored in the cache dtype (round to
 *   nearest even).  [TSD-V4] §2.2 gives no formula; this gated block sum is the fixed stand-in.
 * - Visibility ([TSD-V4] §3.1, §3.2): a query at position p sees compressed entry (m, j) iff
 *   m*j+m-1 <= p-1, and raw tokens at positions raw_lo(p) .. p; a tree node sees only its own
 *   ancestors (and itself) among the tree tokens and only its proper ancestors' scratch entries.
 *   raw_lo(p) = max(0, p - W) (TV_TAIL_WINDOW) or m_min * floor(p / m_min) (TV_TAIL_REMAINDER,
 *   m_min = 4 if C4 is active, else 128).
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tv_stream_t; /* the same handle type as cudaStream_t */

/* status codes */
#define TV_OK 0
#define TV_ERR_ARG (-1)        /* null pointer, unknown enum value or inconsistent argument */
#define TV_ERR_SHAPE (-2)      /* unsupported shape (D > 64, d not a multiple of 8, ...) */
#define TV_ERR_BAD_TREE (-3)   /* parents[b][0] != -1 or parents[b][v] not in [0, v) */
#define TV_ERR_CAPACITY (-4)   /* a length or entry count exceeds the buffer capacity */
#define TV_ERR_DTYPE (-5)      /* dtype not supported by the requested kernel */
#define TV_ERR_CUDA (-6)       /* a CUDA runtime call failed (launch, tensor-map encoding) */
#define TV_ERR_WORKSPACE (-7)  /* workspace too small (see tv_workspace_size) */
#define TV_ERR_TIMEOUT (-8)    /* a bounded device-side wait ran out (kernel returned early) */
#define TV_ERR_SELECTION (-9)  /* a selection index is outside the request's C4 entries */
#define TV_ERR_BOUNDS (-10)    /* bounds-checked build only: a global index failed its range
                                  check (the access was skipped; the site is printed once) */

/* tv_shape.tail_mode */
#define TV_TAIL_WINDOW 0
#define TV_TAIL_REMAINDER 1
/* tv_shape.comp_mask bits */
#define TV_COMP_C4 1
#define TV_COMP_C128 2
/* tv_shape.dtype */
#define TV_F32 0
#define TV_BF16 1
/* tv_shape.attn_kernel */
#define TV_ATTN_AUTO 0    /* tensor-core kernel where supported, else the SIMT kernel */
#define TV_ATTN_SIMT 1    /* CUDA-core fp32 kernel: any supported shape, fp32 or bf16 */
#define TV_ATTN_TCGEN05 2 /* tcgen05 tensor-core kernel: bf16, d == 512 */

typedef struct tv_shape {
  int32_t B;           /* requests (>= 0; B == 0 turns every call into a no-op) */
  int32_t D;           /* tree nodes per request including the root, 1..64 */
  int32_t H;           /* query heads sharing the single K/V head, 1..1024 */
  int32_t d;           /* head dimension of Q, K, V and O: multiple of 8, 8..512 */
  int32_t W;           /* raw window for TV_TAIL_WINDOW, 0..1024 (ignored otherwise) */
  int32_t tail_mode;   /* TV_TAIL_WINDOW | TV_TAIL_REMAINDER */
  int32_t comp_mask;   /* non-empty subset of TV_COMP_C4 | TV_COMP_C128 */
  int32_t dtype;       /* TV_F32 | TV_BF16: storage of Q, K, V, O, raw and compressed rows */
  int32_t n_sel;       /* 0: all persistent C4 entries visible; > 0: only the n_sel listed ones */
  int32_t attn_kernel; /* TV_ATTN_* */
  int64_t raw_cap;     /* rows per request of rawK / rawV */
  int64_t c4_cap;      /* rows per request of c4K / c4V (ignored without C4) */
  int64_t c128_cap;    /* rows per request of c128K / c128V (ignored without C128) */
  /* Page-based persistent cache ([TSD-V4] §4.2: one logical layer over three physical layers
   * with shared page pointers).  page_tokens == 0: rawK/rawV, c4K/c4V, c128K/c128V are
   * contiguous [B][cap][d] arrays.  page_tokens == P > 0 (a multiple of 512): they are page pools
   * of n_pool_pages pages -- rawK [n_pool_pages][P][d], c4K [n_pool_pages][P/4][d],
   * c128K [n_pool_pages][P/128][d] (V alike) -- and logical page g of request b (tokens
   * g*P .. g*P+P-1, with their C4 and C128 entries) lives in page page_table[b][g] of all three;
   * raw_cap, c4_cap and c128_cap must then be max_pages * P, * P/4 and * P/128.  A page id outside
   * 0 .. n_pool_pages-1 is reported as TV_ERR_ARG on the device (and page 0 is read instead). */
  int32_t page_tokens;
  int32_t max_pages;           /* logical pages per request (columns of page_table) */
  int32_t n_pool_pages;        /* pages in each pool */
  /* Refresh skip ([TSD-V4] §4.3: the refresh can be skipped when there is a single candidate
   * chain or the accepted chain is the latest cached one) and the two refresh schedules of §4.2
   * (C4 promptly, C128 delayed until the accepted path is known).  0: off.  1: tv_branch_compress
   * writes the round's cached chain -- the root, its lowest-numbered child, that node's
   * lowest-numbered child, ... -- into the persistent raw rows L[b] + depth and the C4 entries
   * those positions close (rows and entries past the committed length: invisible to every call
   * until tv_refresh_commit advances L), and tv_refresh_commit copies only the accepted nodes off
   * that chain and the accepted C128 entries.  A single-chain tree then commits by advancing L. */
  int32_t stage_chain;
  const int32_t* page_table;   /* device [B][max_pages] int32 (page_tokens > 0 only) */
} tv_shape;

/* Library version string (static storage). */
const char* tv_version(void);

/* Human-readable name of a TV_* status code (static storage). */
const char* tv_status_string(int code);

/* Description of the calling thread's last host-side error (thread-local storage, valid until
 * the thread's next call into the library). */
const char* tv_last_error_string(void);

/* Bytes of device workspace tv_tree_verify_attn needs for this shape (0 for B == 0).  The
 * workspace holds the split-KV partial results and the work counters; the caller allocates it
 * (any 256-byte-aligned device buffer) and may reuse it across calls on the same stream. */
size_t tv_workspace_size(const tv_shape* shape);

/* The attention kernel tv_tree_verify_attn runs for this shape on the current device:
 * TV_ATTN_SIMT or TV_ATTN_TCGEN05, or a negative TV_ERR_* code for an invalid shape. */
int tv_attn_kernel_for(const tv_shape* shape);

/*
 * Verify preprocess: the verification plan ([TSD-V4] §4.1 -- the candidate tree becomes the
 * metadata that guides attention and compression; §4.3 -- built on the device).
 *   parents  [B][D] int32   in   tree topology
 *   L        [B]    int32   in   committed lengths
 *   anc      [B][D] uint64  out  bit u of anc[b][v] set iff u is on the path root -> v
 *   depth    [B][D] int32   out  depth of v (root 0); position = L[b] + depth
 *   raw_lo   [B][D] int32   out  lowest raw position visible from v (see raw_lo(p) above)
 *   scr_vis4 [B][D] uint64  out  proper ancestors of v whose token closes a C4 block
 *                                 (nullable when C4 is inactive)
 *   scr_vis128 [B][D] uint64 out same for C128 (nullable when C128 is inactive)
 * Device errors: TV_ERR_BAD_TREE (that request's outputs are zero), TV_ERR_ARG for L < 0.
 */
int tv_build_ancestor_mask(const tv_shape* shape, const int32_t* parents, const int32_t* L,
                           uint64_t* anc, int32_t* depth, int32_t* raw_lo, uint64_t* scr_vis4,
                           uint64_t* scr_vis128, int32_t* status, tv_stream_t stream);

/*
 * Prefill compression ([TSD-V4] §2.2): writes every complete block of each request's committed
 * prefix, entries 0 .. floor(L[b]/m) - 1 of each active compressor, from the raw rows.
 *   rawK, rawV [B][raw_cap][d] in; L [B] in; g4, g128 [d] fp32 gate vectors (nullable when the
 *   compressor is inactive); c4K, c4V, c128K, c128V out.
 * Device errors: TV_ERR_CAPACITY when L > raw_cap or floor(L/m) > cap_m (request skipped).
 */
int tv_prefill_compress(const tv_shape* shape, const void* rawK, const void* rawV,
                        const int32_t* L, const float* g4, const float* g128, void* c4K,
                        void* c4V, void* c128K, void* c128V, int32_t* status,
                        tv_stream_t stream);

/*
 * Scratch-pad branch compression ([TSD-V4] §3.2, §4.1, §4.2: a chain that closes a block after
 * branching is compressed on its own, into temporary storage).  For every node v and active
 * compressor m with (L[b] + depth(v) + 1) % m == 0, row v of the m scratch pad becomes the gated
 * sum of the m positions ending at v's position, read from the sequence prefix + path(v):
 * positions < L[b] from rawK/rawV, the others from treeK/treeV of v's ancestors.  Every other
 * row is set to zero.
 * With shape->stage_chain == 1 it also stages the cached chain (see tv_shape): for every node c
 * of that chain, rawK/rawV row L[b] + depth(c) <- treeK/treeV row c, and when c closes a C4
 * block, C4 entry (L[b] + depth(c) + 1)/4 - 1 <- c's C4 scratch row; positions or entries past
 * raw_cap / c4_cap are not staged.  Nothing at or below L[b] - 1 and no C128 entry is written.
 *   rawK, rawV [B][raw_cap][d] in (and out past L[b] when staging); L [B] in; treeK, treeV
 *   [B][D][d] in (K/V of the tree tokens); parents [B][D] in; g4, g128 [d] fp32 in;
 *   scrK4, scrV4, scrK128, scrV128 [B][D][d] out (the pair of an inactive compressor is
 *   nullable); c4K, c4V [B][c4_cap][d] out past L[b]/4 when staging with C4 active (else
 *   nullable).
 * Device errors: TV_ERR_BAD_TREE, TV_ERR_CAPACITY (L > raw_cap).
 */
int tv_branch_compress(const tv_shape* shape, void* rawK, void* rawV, void* c4K, void* c4V,
                       const int32_t* L, const void* treeK, const void* treeV,
                       const int32_t* parents, const float* g4, const float* g128, void* scrK4,
                       void* scrV4, void* scrK128, void* scrV128, int32_t* status,
                       tv_stream_t stream);

/*
 * Branch-aware causal tree-verify attention ([TSD-V4] §3.1, §4.1, §4.4), split-KV.
 * Every (node v, head h) row attends, with logit scale `scale` (normally 1/sqrt(d)), to
 *   - the persistent C4 entries 0 .. L/4-1 (or, with n_sel > 0, the listed ones sel[b][i]),
 *   - the persistent C128 entries 0 .. L/128-1,
 *   - the raw rows at positions raw_lo[b][v] .. L-1,
 *   - the tree tokens u with anc bit u set and position L + depth(u) >= raw_lo[b][v],
 *   - the scratch entries of the nodes flagged in scr_vis4 / scr_vis128.
 * The compressed prefix is read once per request and shared by all D*H rows.
 *   Q    [B][D][H][d] in (dtype);  sel [B][n_sel] int32 (nullable when n_sel == 0)
 *   anc, raw_lo, scr_vis4, scr_vis128: the plan of tv_build_ancestor_mask
 *   O    [B][D][H][d] out (dtype); lse [B][D][H] fp32 out: natural-log sum of exp(logits)
 *   (Q and O 16-byte aligned)
 *   workspace: device buffer of ws_bytes >= tv_workspace_size(shape)
 * Host errors: TV_ERR_ARG (also a misaligned Q or O), TV_ERR_WORKSPACE, TV_ERR_DTYPE
 * (TV_ATTN_TCGEN05 asked for an unsupported shape).
 * Device errors: TV_ERR_SELECTION, TV_ERR_CAPACITY, TV_ERR_TIMEOUT.
 */
int tv_tree_verify_attn(const tv_shape* shape, const void* Q, const void* c4K, const void* c4V,
                        const int32_t* sel, const void* c128K, const void* c128V,
                        const void* rawK, const void* rawV, const int32_t* L,
                        const void* treeK, const void* treeV, const uint64_t* anc,
                        const int32_t* raw_lo, const uint64_t* scr_vis4,
                        const uint64_t* scr_vis128, const void* scrK4, const void* scrV4,
                        const void* scrK128, const void* scrV128, float scale, void* O,
                        float* lse, void* workspace, size_t ws_bytes, int32_t* status,
                        tv_stream_t stream);

/*
 * tv_tree_verify_attn without a workspace argument, for callers that cannot allocate device
 * memory (an engine that reserved all free memory for its own page pool, a decode loop that must
 * not pay cudaMalloc's implicit synchronisation, a plug-in host without an allocator).  The report
 * has no counterpart: this is a convenience of the library.  Same arguments, semantics and
 * outputs as tv_tree_verify_attn, minus workspace / ws_bytes.  The split-KV partial results live
 * in a 32 MiB array inside the library image, held by every GPU that loads the library's device
 * code until the process exits; a shape whose tv_workspace_size exceeds it is rejected with
 * TV_ERR_WORKSPACE.  Under CUDA's lazy module loading (the default) the device code, and with it
 * the 32 MiB, is loaded on a device at the first call there that resolves the array: call
 * tv_noalloc_prepare once per device at start-up, before reserving a memory pool and before any
 * stream capture; later calls take no device memory.  The array's address is looked up in the
 * caller's current context on every call.  All calls share the array: calls that overlap on the
 * GPU race on it (its previous contents are never read, nothing needs clearing).  Host errors name
 * tv_tree_verify_attn_noalloc.  It allocates nothing, neither on the device nor through any
 * library.
 */
int tv_tree_verify_attn_noalloc(const tv_shape* shape, const void* Q, const void* c4K,
                                const void* c4V, const int32_t* sel, const void* c128K,
                                const void* c128V, const void* rawK, const void* rawV,
                                const int32_t* L, const void* treeK, const void* treeV,
                                const uint64_t* anc, const int32_t* raw_lo,
                                const uint64_t* scr_vis4, const uint64_t* scr_vis128,
                                const void* scrK4, const void* scrV4, const void* scrK128,
                                const void* scrV128, float scale, void* O, float* lse,
                                int32_t* status, tv_stream_t stream);

/*
 * Loads the library's device code on the current device, with the built-in scratch of
 * tv_tree_verify_attn_noalloc (32 MiB), so that later calls take no device memory.  Call it once
 * per device before handing the free memory to a pool.  Returns TV_OK, or TV_ERR_CUDA if the
 * device code cannot be loaded (for instance when less than 32 MiB is free).
 */
int tv_noalloc_prepare(void);

/*
 * Accepted-path selection ([TSD-V4] §3.2, §4.1): greedy walk from the root; at each node take
 * the lowest-numbered child whose draft token equals the node's target token; stop when none.
 *   parents, draft, target [B][D] int32 in
 *   accept_len [B] out: path length including the root (>= 1)
 *   path [B][D] out: accepted node ids in order, -1 padded
 *   bonus [B] out: target token of the last accepted node
 * Device errors: TV_ERR_BAD_TREE.
 */
int tv_accept_walk(const tv_shape* shape, const int32_t* parents, const int32_t* draft,
                   const int32_t* target, int32_t* accept_len, int32_t* path, int32_t* bonus,
                   int32_t* status, tv_stream_t stream);

/*
 * Accepted-path state refresh ([TSD-V4] §3.2, §4.2: only the accepted path's token, KV and
 * compressed states reach the persistent context; rejected branches are dropped).
 * With n = accept_len[b] and path = path[b]:
 *   rawK/rawV row L+i <- treeK/treeV row path[i] (exact copy), i < n;
 *   for every active m and position e in [L, L+n-1] with (e+1) % m == 0: entry (e+1)/m - 1 <-
 *   scratch row path[e-L] of compressor m (that row is the gated sum of exactly the committed
 *   block, so the copy equals recompressing it); L[b] <- L + n;
 *   committed_pos[b][i] = old L + i for i < n, -1 otherwise.
 * The scratch pad must come from tv_branch_compress of the same round.
 * With shape->stage_chain == 1 the writes tv_branch_compress already staged are skipped: the
 * accepted nodes path[i] that are the i-th node of the cached chain (computed from parents, which
 * must then be given) keep their staged raw row and C4 entry; every other accepted raw row and C4
 * entry, and every C128 entry the accepted path closes, are copied as above.
 *   parents [B][D] in (stage_chain == 1 only, else nullable)
 * Device errors: TV_ERR_CAPACITY (L+n > raw_cap or an entry beyond cap_m; request untouched),
 * TV_ERR_ARG (accept_len outside 1..D or a path id outside 0..D-1; request untouched).
 */
int tv_refresh_commit(const tv_shape* shape, const int32_t* parents, const int32_t* accept_len,
                      const int32_t* path, const void* treeK, const void* treeV, const void* scrK4,
                      const void* scrV4, const void* scrK128, const void* scrV128, void* rawK,
                      void* rawV, void* c4K, void* c4V, void* c128K, void* c128V, int32_t* L,
                      int32_t* committed_pos, int32_t* status, tv_stream_t stream);

/*
 * Indexer top-k selection of the persistent C4 entries for the sparse prefix path ([TSD-V4] §2.2:
 * CSA is compressed *sparse* attention; the report gives no selection rule, so the rule here is
 * the stand-in of the long-context workload).  For every request b with n4 = L[b]/4 C4 entries:
 *   score[j] = q_idx[b] . k_idx[b][j], j < n4, computed in fp32 as products of the bf16 inputs
 *   (exact) added in index order 0 .. d_idx-1, one round-to-nearest-even per addition, no fused
 *   multiply-add;
 *   sel[b] = the n_sel entries of largest score (equal scores: lower j first), ascending in j --
 *   the selection list tv_tree_verify_attn takes.
 * Uses shape->B, c4_cap (rows of k_idx per request), n_sel (> 0) and needs C4 in comp_mask.
 *   d_idx: indexer dimension, a multiple of 8 in 8..256
 *   q_idx [B][d_idx] bf16 in; k_idx [B][c4_cap][d_idx] bf16 in (16-byte aligned); L [B] in
 *   sel [B][n_sel] int32 out
 *   workspace: device buffer of ws_bytes >= tv_indexer_workspace_size(shape) (the fp32 scores)
 * Host errors: TV_ERR_ARG, TV_ERR_SHAPE, TV_ERR_WORKSPACE.
 * Device errors: TV_ERR_SELECTION (n4 < n_sel), TV_ERR_CAPACITY (n4 > c4_cap); that request's
 * sel row is set to -1.
 */
size_t tv_indexer_workspace_size(const tv_shape* shape);
int tv_indexer_topk(const tv_shape* shape, int d_idx, const void* q_idx, const void* k_idx,
                    const int32_t* L, int32_t* sel, void* workspace, size_t ws_bytes,
                    int32_t* status, tv_stream_t stream);

/*
 * Testing aid for the failure path of the tensor-core attention (the report has no counterpart).
 * Sets, for every later tv_tree_verify_attn launch of the tcgen05 kernel in this process:
 *   timeout_ns     the bound of every device-side wait (default 2000000000 = 2 s; > 0);
 *   withhold_tile  one KV tile index (within each work item's tile range) whose K copies the
 *                  producers never issue, or -1 for none (the default).
 * With a tile withheld, the MMA issuer's wait for that tile runs out after timeout_ns; the kernel
 * then records TV_ERR_TIMEOUT in the status word, stops every CTA of the affected clusters,
 * drains the copies and MMAs it did issue and returns, leaving the context usable.  Restore
 * (2000000000, -1) afterwards.  Host errors: TV_ERR_ARG (timeout_ns <= 0 or withhold_tile < -1).
 */
int tv_debug_attn_timeout(int64_t timeout_ns, int32_t withhold_tile);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
