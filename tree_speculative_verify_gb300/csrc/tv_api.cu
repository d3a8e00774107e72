// Host entry points of libtreeverify.so: argument validation, workspace sizing, dispatch.
// The operations and their citations are documented in include/treeverify.h.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <string>

#include "tv_attn_common.cuh"
#include "tv_attn_tc.cuh"

// ---- error reporting --------------------------------------------------------------------------
static thread_local std::string g_last_error;

int tv_set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int tv_check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return tv_set_error(TV_ERR_CUDA, "%s: kernel launch failed: %s", what, cudaGetErrorString(e));
  return TV_OK;
}

extern "C" const char* tv_version(void) { return "treeverify 0.1 (sm_103a)"; }

extern "C" const char* tv_status_string(int code) {
  switch (code) {
    case TV_OK: return "TV_OK";
    case TV_ERR_ARG: return "TV_ERR_ARG";
    case TV_ERR_SHAPE: return "TV_ERR_SHAPE";
    case TV_ERR_BAD_TREE: return "TV_ERR_BAD_TREE";
    case TV_ERR_CAPACITY: return "TV_ERR_CAPACITY";
    case TV_ERR_DTYPE: return "TV_ERR_DTYPE";
    case TV_ERR_CUDA: return "TV_ERR_CUDA";
    case TV_ERR_WORKSPACE: return "TV_ERR_WORKSPACE";
    case TV_ERR_TIMEOUT: return "TV_ERR_TIMEOUT";
    case TV_ERR_SELECTION: return "TV_ERR_SELECTION";
    case TV_ERR_BOUNDS: return "TV_ERR_BOUNDS";
    default: return "TV_ERR_UNKNOWN";
  }
}

extern "C" const char* tv_last_error_string(void) { return g_last_error.c_str(); }

// ---- shape validation -------------------------------------------------------------------------
static int check_shape(const tv_shape* s, const char* fn) {
  g_last_error.clear();
  if (s == nullptr) return tv_set_error(TV_ERR_ARG, "%s: shape is null", fn);
  if (s->B < 0) return tv_set_error(TV_ERR_SHAPE, "%s: B = %d < 0", fn, s->B);
  if (s->D < 1 || s->D > tv::kMaxD)
    return tv_set_error(TV_ERR_SHAPE, "%s: D = %d outside 1..64", fn, s->D);
  if (s->H < 1 || s->H > 1024) return tv_set_error(TV_ERR_SHAPE, "%s: H = %d outside 1..1024", fn, s->H);
  if (s->d < 8 || s->d > tv::kMaxHeadDim || s->d % 8 != 0)
    return tv_set_error(TV_ERR_SHAPE, "%s: d = %d is not a multiple of 8 in 8..512", fn, s->d);
  if (s->tail_mode != TV_TAIL_WINDOW && s->tail_mode != TV_TAIL_REMAINDER)
    return tv_set_error(TV_ERR_ARG, "%s: unknown tail_mode %d", fn, s->tail_mode);
  if (s->tail_mode == TV_TAIL_WINDOW && (s->W < 0 || s->W > 1024))
    return tv_set_error(TV_ERR_SHAPE, "%s: W = %d outside 0..1024", fn, s->W);
  if (s->comp_mask < 1 || s->comp_mask > 3)
    return tv_set_error(TV_ERR_ARG, "%s: comp_mask %d is not a non-empty subset of C4|C128", fn,
                        s->comp_mask);
  if (s->dtype != TV_F32 && s->dtype != TV_BF16)
    return tv_set_error(TV_ERR_ARG, "%s: unknown dtype %d", fn, s->dtype);
  if (s->n_sel < 0 || (s->n_sel > 0 && !(s->comp_mask & TV_COMP_C4)))
    return tv_set_error(TV_ERR_ARG, "%s: n_sel = %d needs C4 and must be >= 0", fn, s->n_sel);
  if (s->attn_kernel < TV_ATTN_AUTO || s->attn_kernel > TV_ATTN_TCGEN05)
    return tv_set_error(TV_ERR_ARG, "%s: unknown attn_kernel %d", fn, s->attn_kernel);
  if (s->raw_cap < 0 || s->c4_cap < 0 || s->c128_cap < 0 || s->raw_cap > (int64_t)1 << 30 ||
      s->c4_cap > (int64_t)1 << 30 || s->c128_cap > (int64_t)1 << 30)
    return tv_set_error(TV_ERR_SHAPE, "%s: capacities must be in 0..2^30", fn);
  if ((int64_t)s->B * s->D * s->H > ((int64_t)1 << 31) / 1024)
    return tv_set_error(TV_ERR_SHAPE, "%s: B*D*H too large", fn);
  if (s->stage_chain != 0 && s->stage_chain != 1)
    return tv_set_error(TV_ERR_ARG, "%s: stage_chain must be 0 or 1", fn);
  if (s->page_tokens != 0) {
    const int64_t P = s->page_tokens, G = s->max_pages;
    if (P < 0 || P % 512 != 0 || P > (1 << 20))
      return tv_set_error(TV_ERR_SHAPE, "%s: page_tokens = %d is not a multiple of 512", fn,
                          s->page_tokens);
    if (G < 1 || s->n_pool_pages < 1 || (int64_t)s->n_pool_pages * P > ((int64_t)1 << 31))
      return tv_set_error(TV_ERR_SHAPE, "%s: max_pages = %d / n_pool_pages = %d out of range", fn,
                          s->max_pages, s->n_pool_pages);
    if (s->raw_cap != G * P || s->c4_cap != G * P / 4 || s->c128_cap != G * P / 128)
      return tv_set_error(TV_ERR_SHAPE,
                          "%s: with pages, raw_cap / c4_cap / c128_cap must be max_pages * P, "
                          "* P/4, * P/128",
                          fn);
    if (s->B > 0 && s->page_table == nullptr)
      return tv_set_error(TV_ERR_ARG, "%s: page_table is null", fn);
  }
  return TV_OK;
}

#define TV_REQUIRE(ptr, fn) \
  if ((ptr) == nullptr) return tv_set_error(TV_ERR_ARG, "%s: %s is null", fn, #ptr)

static inline bool has_c4(const tv_shape* s) { return s->comp_mask & TV_COMP_C4; }
static inline bool has_c128(const tv_shape* s) { return s->comp_mask & TV_COMP_C128; }

// ---- launchers implemented in the kernel files ------------------------------------------------
int tv_launch_plan(const tv_shape* s, const int32_t* parents, const int32_t* L, uint64_t* anc,
                   int32_t* depth, int32_t* raw_lo, uint64_t* scr_vis4, uint64_t* scr_vis128,
                   int32_t* status, cudaStream_t stream);
int tv_launch_prefill(const tv_shape* s, const void* rawK, const void* rawV, const int32_t* L,
                      const float* g4, const float* g128, void* c4K, void* c4V, void* c128K,
                      void* c128V, int32_t* status, cudaStream_t stream);
int tv_launch_branch(const tv_shape* s, void* rawK, void* rawV, void* c4K, void* c4V,
                     const int32_t* L,
                     const void* treeK, const void* treeV, const int32_t* parents,
                     const float* g4, const float* g128, void* scrK4, void* scrV4,
                     void* scrK128, void* scrV128, int32_t* status, cudaStream_t stream);
int tv_launch_accept(const tv_shape* s, const int32_t* parents, const int32_t* draft,
                     const int32_t* target, int32_t* accept_len, int32_t* path, int32_t* bonus,
                     int32_t* status, cudaStream_t stream);
int tv_launch_refresh(const tv_shape* s, const int32_t* parents, const int32_t* accept_len,
                      const int32_t* path,
                      const void* treeK, const void* treeV, const void* scrK4, const void* scrV4,
                      const void* scrK128, const void* scrV128, void* rawK, void* rawV,
                      void* c4K, void* c4V, void* c128K, void* c128V, int32_t* L,
                      int32_t* committed, int32_t* status, cudaStream_t stream);

int tv_launch_indexer(const tv_shape* s, int d_idx, const void* q_idx, const void* k_idx,
                      const int32_t* L, int32_t* sel, void* workspace, int32_t* status,
                      cudaStream_t stream);

// ---- split-KV geometry of the SIMT kernel -----------------------------------------------------
struct SimtPlan {
  int n_chunks;
  int chunk;
  size_t part_bytes;
};

static int64_t max_entries(const tv_shape* s) {
  int64_t n = 0;
  if (has_c4(s)) n += (s->n_sel > 0 ? s->n_sel : s->c4_cap) + s->D;
  if (has_c128(s)) n += s->c128_cap + s->D;
  n += (s->tail_mode == TV_TAIL_WINDOW ? s->W : tv::m_min_of(s->comp_mask) - 1) + s->D;
  return n;
}

static SimtPlan simt_plan(const tv_shape* s) {
  SimtPlan p;
  const int64_t DH = (int64_t)s->D * s->H;
  const int64_t row_groups = (DH + 7) / 8;
  const int64_t base_ctas = (int64_t)s->B * row_groups;
  const int64_t ne = max_entries(s);
  int64_t n_chunks = base_ctas > 0 ? (4 * 152 + base_ctas - 1) / base_ctas : 1;
  const int64_t max_chunks = (ne + 63) / 64;
  if (n_chunks > max_chunks) n_chunks = max_chunks;
  if (n_chunks < 1) n_chunks = 1;
  if (n_chunks > 256) n_chunks = 256;
  int64_t chunk = (ne + n_chunks - 1) / n_chunks;
  chunk = (chunk + 7) / 8 * 8;
  p.n_chunks = (int)n_chunks;
  p.chunk = (int)chunk;
  p.part_bytes = (size_t)s->B * DH * n_chunks * (s->d + 4) * sizeof(float);
  return p;
}

static bool tc_supported(const tv_shape* s) {
  return tv_tc_shape_ok(s) && tv_tc_available();
}

static bool use_tc(const tv_shape* s) {
  if (s->attn_kernel == TV_ATTN_SIMT) return false;
  if (s->attn_kernel == TV_ATTN_TCGEN05) return true;
  return tc_supported(s);
}

static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

extern "C" size_t tv_workspace_size(const tv_shape* s) {
  if (check_shape(s, "tv_workspace_size") != TV_OK || s->B == 0) return 0;
  if (use_tc(s)) return align256(tv_tc_workspace_size(s));
  return align256(simt_plan(s).part_bytes);
}

extern "C" int tv_attn_kernel_for(const tv_shape* s) {
  if (int rc = check_shape(s, "tv_attn_kernel_for")) return rc;
  if (!use_tc(s)) return TV_ATTN_SIMT;
  if (!tc_supported(s))
    return tv_set_error(TV_ERR_DTYPE, "tv_attn_kernel_for: the tcgen05 kernel needs bf16, d = 512, D <= 8, "
                        "and an sm_103 device");
  return TV_ATTN_TCGEN05;
}

// ---- entry points -----------------------------------------------------------------------------
extern "C" int tv_build_ancestor_mask(const tv_shape* s, const int32_t* parents, const int32_t* L,
                                      uint64_t* anc, int32_t* depth, int32_t* raw_lo,
                                      uint64_t* scr_vis4, uint64_t* scr_vis128, int32_t* status,
                                      tv_stream_t stream) {
  const char* fn = "tv_build_ancestor_mask";
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(parents, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(anc, fn);
  TV_REQUIRE(depth, fn);
  TV_REQUIRE(raw_lo, fn);
  TV_REQUIRE(status, fn);
  if (has_c4(s)) TV_REQUIRE(scr_vis4, fn);
  if (has_c128(s)) TV_REQUIRE(scr_vis128, fn);
  return tv_launch_plan(s, parents, L, anc, depth, raw_lo, scr_vis4, scr_vis128, status,
                        (cudaStream_t)stream);
}

extern "C" int tv_prefill_compress(const tv_shape* s, const void* rawK, const void* rawV,
                                   const int32_t* L, const float* g4, const float* g128,
                                   void* c4K, void* c4V, void* c128K, void* c128V,
                                   int32_t* status, tv_stream_t stream) {
  const char* fn = "tv_prefill_compress";
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(rawK, fn);
  TV_REQUIRE(rawV, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(status, fn);
  if (has_c4(s)) {
    TV_REQUIRE(g4, fn);
    TV_REQUIRE(c4K, fn);
    TV_REQUIRE(c4V, fn);
  }
  if (has_c128(s)) {
    TV_REQUIRE(g128, fn);
    TV_REQUIRE(c128K, fn);
    TV_REQUIRE(c128V, fn);
  }
  return tv_launch_prefill(s, rawK, rawV, L, g4, g128, c4K, c4V, c128K, c128V, status,
                           (cudaStream_t)stream);
}

extern "C" int tv_branch_compress(const tv_shape* s, void* rawK, void* rawV, void* c4K, void* c4V,
                                  const int32_t* L, const void* treeK, const void* treeV,
                                  const int32_t* parents, const float* g4, const float* g128,
                                  void* scrK4, void* scrV4, void* scrK128, void* scrV128,
                                  int32_t* status, tv_stream_t stream) {
  const char* fn = "tv_branch_compress";
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(rawK, fn);
  TV_REQUIRE(rawV, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(treeK, fn);
  TV_REQUIRE(treeV, fn);
  TV_REQUIRE(parents, fn);
  TV_REQUIRE(status, fn);
  if (has_c4(s)) {
    TV_REQUIRE(g4, fn);
    TV_REQUIRE(scrK4, fn);
    TV_REQUIRE(scrV4, fn);
  }
  if (has_c128(s)) {
    TV_REQUIRE(g128, fn);
    TV_REQUIRE(scrK128, fn);
    TV_REQUIRE(scrV128, fn);
  }
  if (s->stage_chain && has_c4(s)) {
    TV_REQUIRE(c4K, fn);
    TV_REQUIRE(c4V, fn);
  }
  return tv_launch_branch(s, rawK, rawV, c4K, c4V, L, treeK, treeV, parents, g4, g128, scrK4,
                          scrV4, scrK128, scrV128, status, (cudaStream_t)stream);
}

template <typename T>
static tv::AttnParams<T> make_params(const tv_shape* s, const void* Q, const void* c4K,
                                     const void* c4V, const int32_t* sel, const void* c128K,
                                     const void* c128V, const void* rawK, const void* rawV,
                                     const int32_t* L, const void* treeK, const void* treeV,
                                     const uint64_t* anc, const int32_t* raw_lo,
                                     const uint64_t* scr_vis4, const uint64_t* scr_vis128,
                                     const void* scrK4, const void* scrV4, const void* scrK128,
                                     const void* scrV128, float scale, void* O, float* lse,
                                     int32_t* status) {
  tv::AttnParams<T> p;
  p.B = s->B;
  p.D = s->D;
  p.H = s->H;
  p.d = s->d;
  p.W = s->W;
  p.tail_mode = s->tail_mode;
  p.comp_mask = s->comp_mask;
  p.n_sel = s->n_sel;
  p.raw_cap = s->raw_cap;
  p.c4_cap = s->c4_cap;
  p.c128_cap = s->c128_cap;
  p.pg = tv::paging_of(s);
  p.Q = (const T*)Q;
  p.c4K = (const T*)c4K;
  p.c4V = (const T*)c4V;
  p.c128K = (const T*)c128K;
  p.c128V = (const T*)c128V;
  p.rawK = (const T*)rawK;
  p.rawV = (const T*)rawV;
  p.treeK = (const T*)treeK;
  p.treeV = (const T*)treeV;
  p.scrK4 = (const T*)scrK4;
  p.scrV4 = (const T*)scrV4;
  p.scrK128 = (const T*)scrK128;
  p.scrV128 = (const T*)scrV128;
  p.sel = sel;
  p.L = L;
  p.raw_lo = raw_lo;
  p.anc = anc;
  p.scr_vis4 = scr_vis4;
  p.scr_vis128 = scr_vis128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.n_chunks = 1;
  p.chunk = 0;
  p.part = nullptr;
  p.O = (T*)O;
  p.lse = lse;
  p.status = status;
  return p;
}

// The attention behind both entry points; fn names the caller's entry point in error messages.
int tv_attn_entry(const char* fn, const tv_shape* s, const void* Q, const void* c4K,
                  const void* c4V, const int32_t* sel, const void* c128K, const void* c128V,
                  const void* rawK, const void* rawV, const int32_t* L, const void* treeK,
                  const void* treeV, const uint64_t* anc, const int32_t* raw_lo,
                  const uint64_t* scr_vis4, const uint64_t* scr_vis128, const void* scrK4,
                  const void* scrV4, const void* scrK128, const void* scrV128, float scale,
                  void* O, float* lse, void* workspace, size_t ws_bytes, int32_t* status,
                  tv_stream_t stream) {
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(Q, fn);
  TV_REQUIRE(rawK, fn);
  TV_REQUIRE(rawV, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(treeK, fn);
  TV_REQUIRE(treeV, fn);
  TV_REQUIRE(anc, fn);
  TV_REQUIRE(raw_lo, fn);
  TV_REQUIRE(O, fn);
  TV_REQUIRE(lse, fn);
  TV_REQUIRE(workspace, fn);
  TV_REQUIRE(status, fn);
  if (has_c4(s)) {
    TV_REQUIRE(c4K, fn);
    TV_REQUIRE(c4V, fn);
    TV_REQUIRE(scr_vis4, fn);
    TV_REQUIRE(scrK4, fn);
    TV_REQUIRE(scrV4, fn);
  }
  if (has_c128(s)) {
    TV_REQUIRE(c128K, fn);
    TV_REQUIRE(c128V, fn);
    TV_REQUIRE(scr_vis128, fn);
    TV_REQUIRE(scrK128, fn);
    TV_REQUIRE(scrV128, fn);
  }
  if (s->n_sel > 0) TV_REQUIRE(sel, fn);
  if (!(scale > 0.f) || !(scale < 1e30f))
    return tv_set_error(TV_ERR_ARG, "%s: scale must be a positive finite number", fn);
  if (((uintptr_t)workspace) % 256 != 0)
    return tv_set_error(TV_ERR_ARG, "%s: workspace must be 256-byte aligned", fn);
  // rows of Q and O are read and written 16 bytes at a time
  if (((uintptr_t)Q | (uintptr_t)O) & 15u)
    return tv_set_error(TV_ERR_ARG, "%s: Q and O must be 16-byte aligned", fn);
  const size_t need = tv_workspace_size(s);
  if (ws_bytes < need)
    return tv_set_error(TV_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes,
                        need);
  if (use_tc(s)) {
    if (!tc_supported(s))
      return tv_set_error(TV_ERR_DTYPE,
                          "%s: the tcgen05 kernel needs bf16, d = 512, D <= 8 and an sm_103 device", fn);
    auto p = make_params<__nv_bfloat16>(s, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK,
                                        treeV, anc, raw_lo, scr_vis4, scr_vis128, scrK4, scrV4,
                                        scrK128, scrV128, scale, O, lse, status);
    return tv_launch_attn_tc(s, p, workspace, (cudaStream_t)stream);
  }
  const SimtPlan sp = simt_plan(s);
  if (s->dtype == TV_BF16) {
    auto p = make_params<__nv_bfloat16>(s, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK,
                                        treeV, anc, raw_lo, scr_vis4, scr_vis128, scrK4, scrV4,
                                        scrK128, scrV128, scale, O, lse, status);
    p.n_chunks = sp.n_chunks;
    p.chunk = sp.chunk;
    p.part = (float*)workspace;
    return tv_launch_attn_simt_bf16(p, (cudaStream_t)stream);
  }
  auto p = make_params<float>(s, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK, treeV,
                              anc, raw_lo, scr_vis4, scr_vis128, scrK4, scrV4, scrK128, scrV128,
                              scale, O, lse, status);
  p.n_chunks = sp.n_chunks;
  p.chunk = sp.chunk;
  p.part = (float*)workspace;
  return tv_launch_attn_simt_f32(p, (cudaStream_t)stream);
}

extern "C" int tv_tree_verify_attn(const tv_shape* s, const void* Q, const void* c4K,
                                   const void* c4V, const int32_t* sel, const void* c128K,
                                   const void* c128V, const void* rawK, const void* rawV,
                                   const int32_t* L, const void* treeK, const void* treeV,
                                   const uint64_t* anc, const int32_t* raw_lo,
                                   const uint64_t* scr_vis4, const uint64_t* scr_vis128,
                                   const void* scrK4, const void* scrV4, const void* scrK128,
                                   const void* scrV128, float scale, void* O, float* lse,
                                   void* workspace, size_t ws_bytes, int32_t* status,
                                   tv_stream_t stream) {
  return tv_attn_entry("tv_tree_verify_attn", s, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L,
                       treeK, treeV, anc, raw_lo, scr_vis4, scr_vis128, scrK4, scrV4, scrK128,
                       scrV128, scale, O, lse, workspace, ws_bytes, status, stream);
}

extern "C" int tv_accept_walk(const tv_shape* s, const int32_t* parents, const int32_t* draft,
                              const int32_t* target, int32_t* accept_len, int32_t* path,
                              int32_t* bonus, int32_t* status, tv_stream_t stream) {
  const char* fn = "tv_accept_walk";
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(parents, fn);
  TV_REQUIRE(draft, fn);
  TV_REQUIRE(target, fn);
  TV_REQUIRE(accept_len, fn);
  TV_REQUIRE(path, fn);
  TV_REQUIRE(bonus, fn);
  TV_REQUIRE(status, fn);
  return tv_launch_accept(s, parents, draft, target, accept_len, path, bonus, status,
                          (cudaStream_t)stream);
}

extern "C" int tv_refresh_commit(const tv_shape* s, const int32_t* parents,
                                 const int32_t* accept_len, const int32_t* path,
                                 const void* treeK, const void* treeV,
                                 const void* scrK4, const void* scrV4, const void* scrK128,
                                 const void* scrV128, void* rawK, void* rawV, void* c4K,
                                 void* c4V, void* c128K, void* c128V, int32_t* L,
                                 int32_t* committed_pos, int32_t* status, tv_stream_t stream) {
  const char* fn = "tv_refresh_commit";
  if (int rc = check_shape(s, fn)) return rc;
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(accept_len, fn);
  TV_REQUIRE(path, fn);
  TV_REQUIRE(treeK, fn);
  TV_REQUIRE(treeV, fn);
  TV_REQUIRE(rawK, fn);
  TV_REQUIRE(rawV, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(committed_pos, fn);
  TV_REQUIRE(status, fn);
  if (s->stage_chain) TV_REQUIRE(parents, fn);
  if (has_c4(s)) {
    TV_REQUIRE(scrK4, fn);
    TV_REQUIRE(scrV4, fn);
    TV_REQUIRE(c4K, fn);
    TV_REQUIRE(c4V, fn);
  }
  if (has_c128(s)) {
    TV_REQUIRE(scrK128, fn);
    TV_REQUIRE(scrV128, fn);
    TV_REQUIRE(c128K, fn);
    TV_REQUIRE(c128V, fn);
  }
  return tv_launch_refresh(s, parents, accept_len, path, treeK, treeV, scrK4, scrV4, scrK128,
                           scrV128, rawK, rawV, c4K, c4V, c128K, c128V, L, committed_pos, status,
                           (cudaStream_t)stream);
}

// ---- indexer top-k ------------------------------------------------------------------------------
static size_t indexer_ws(const tv_shape* s) {
  return ((size_t)s->B * (size_t)s->c4_cap * sizeof(float) + 255) / 256 * 256;
}

extern "C" size_t tv_indexer_workspace_size(const tv_shape* s) {
  if (check_shape(s, "tv_indexer_workspace_size") != TV_OK || s->B == 0) return 0;
  return indexer_ws(s);
}

extern "C" int tv_indexer_topk(const tv_shape* s, int d_idx, const void* q_idx, const void* k_idx,
                               const int32_t* L, int32_t* sel, void* workspace, size_t ws_bytes,
                               int32_t* status, tv_stream_t stream) {
  const char* fn = "tv_indexer_topk";
  if (int rc = check_shape(s, fn)) return rc;
  if (!has_c4(s) || s->n_sel <= 0)
    return tv_set_error(TV_ERR_ARG, "%s: needs C4 in comp_mask and n_sel > 0 (n_sel = %d)", fn,
                        s->n_sel);
  if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0)
    return tv_set_error(TV_ERR_SHAPE, "%s: d_idx = %d is not a multiple of 8 in 8..256", fn, d_idx);
  if (s->B == 0) return TV_OK;
  TV_REQUIRE(q_idx, fn);
  TV_REQUIRE(k_idx, fn);
  TV_REQUIRE(L, fn);
  TV_REQUIRE(sel, fn);
  TV_REQUIRE(status, fn);
  if (((uintptr_t)q_idx | (uintptr_t)k_idx) & 15u)
    return tv_set_error(TV_ERR_ARG, "%s: q_idx and k_idx must be 16-byte aligned", fn);
  const size_t need = indexer_ws(s);
  if (workspace == nullptr || ws_bytes < need)
    return tv_set_error(TV_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes,
                        need);
  return tv_launch_indexer(s, d_idx, q_idx, k_idx, L, sel, workspace, status,
                           (cudaStream_t)stream);
}
