// C ABI of the gdnbeam library: argument checks, workspace layout, call
// sequencing, and the dispatch of each stage to its kernels.
#include <atomic>
#include <new>
#include <stdio.h>
#include <string.h>
#include <vector>

#include "common.cuh"
#include "launchers.h"

using namespace gdnbeam;

namespace gdnbeam {
static std::atomic<long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace gdnbeam

namespace {

__device__ unsigned int g_dev_error_word;

// Device address of the error word per device, resolved once with that
// device current (atomic: concurrent first calls store the same value).
constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_err_ptr[kMaxDevices] = {};

unsigned* err_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* e = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (!e) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error_word) != cudaSuccess) return nullptr;
    e = (unsigned*)p;
    g_err_ptr[dev].store(e, std::memory_order_relaxed);
  }
  return e;
}

inline size_t elem_size(int dtype) { return dtype == GDNBEAM_BF16 ? 2 : 4; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline int n_proj(const gdnbeam_config& c) { return 2 * key_heads(c) * c.d_k + c.H * c.d_v + 2 * c.H; }
inline int feat_dim(const gdnbeam_config& c) { return c.residual ? c.d_model : c.H * c.d_v; }
inline bool key_width_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }
inline bool value_width_ok(int d) { return key_width_ok(d) || d == 512; }

int validate(const gdnbeam_config* c) {
  if (!c) return GDNBEAM_EINVAL;
  if (c->R < 1 || c->layers < 1 || c->H < 1 || c->d_model < 1 || c->V < 2 || c->T < 1 ||
      c->W_max < 1 || c->L_max < 1)
    return GDNBEAM_EINVAL;
  if (c->T > GDNBEAM_MAX_T || !key_width_ok(c->d_k) || !value_width_ok(c->d_v))
    return GDNBEAM_EUNSUPPORTED;
  // the state-path baselines keep a whole d_v x d_k state per block
  if (c->state_path != 0 && (c->d_k > 128 || c->d_v > 128)) return GDNBEAM_EUNSUPPORTED;
  if (c->dtype != GDNBEAM_F32 && c->dtype != GDNBEAM_BF16) return GDNBEAM_EUNSUPPORTED;
  if (c->V > 16384 || c->W_max > 4096) return GDNBEAM_EUNSUPPORTED;
  if (!c->residual && c->layers != 1) return GDNBEAM_EUNSUPPORTED;
  if (c->residual && c->H * c->d_v != c->d_model) return GDNBEAM_EUNSUPPORTED;
  if ((long long)c->W_max * c->V >= (1ll << 31)) return GDNBEAM_EUNSUPPORTED;
  if (c->state_path < 0 || c->state_path > 2) return GDNBEAM_EUNSUPPORTED;
  if (c->H_k < 0 || (c->H_k > 0 && c->H % c->H_k != 0)) return GDNBEAM_EINVAL;
  if ((long long)c->R * c->L_max >= (1ll << 31) || (long long)c->R * c->W_max * c->V >= (1ll << 40))
    return GDNBEAM_EUNSUPPORTED;
  return GDNBEAM_OK;
}

}  // namespace

unsigned* gdnbeam::error_word() { return err_ptr(); }

struct gdnbeam_ctx {
  gdnbeam_config c;
  gdnbeam_weights w;
  char* ws;
  size_t ws_bytes;
  bool tc_gemm, tc_replay;
  char variant[96];
  // persistent state
  void* sctx;        // [R][layers][H][d_v][d_k]
  void* gtr_k;       // [layers][T-1][R*W_max][H_k*d_k]
  void* gtr_delta;   // [layers][T-1][R*W_max][H*d_v]
  float* gtr_alpha;  // [layers][T-1][R*W_max][H]
  int32_t* anc[2];   // [R*W_max][T]
  int32_t* sid[2];   // [R*W_max][T]
  // transients of one decode call
  void* u;      // [R*W_max][d_model]
  float* x;     // [R*W_max][d_model] residual stream (residual only)
  void* q;      // [R*W_max][H*d_k]
  void* v;      // [R*W_max][H*d_v]
  float* beta;  // [R*W_max][H]
  void* o;      // [R*W_max][H*d_v]
  void* sel;    // selection scratch
  size_t sel_bytes;
  void* gemm;   // CUDA-core GEMM scratch (fp32 raw outputs)
  size_t gemm_bytes;
  float2* tstats;  // [R*W_max][ceil(V/256)]: per (row, 256-code tile) max logit and
                   // sum of exp(z - max), left by the logits stage
  const void* last_logits;  // logits buffer the last logits stage wrote
  int last_rows;
  void* states[2];  // FullState baseline: [R*W_max][layers][H][d_v][d_k] per buffer
  void* sctx_store; // FullState baseline: S_ctx in the storage type (t = 0 parent)
  // prefill buffers for R*L_max rows
  void *pf_u, *pf_q, *pf_k, *pf_v, *pf_feat;
  float *pf_x, *pf_alpha, *pf_beta;
  void* pf_scr;  // stacked layers on the chunked prefill: chunk states and records
  size_t pf_scr_bytes;
  // sequencing: prefilled is set while every request holds a prefilled
  // context (live[r]); a per-request reset clears some of them
  int prefilled;
  std::vector<unsigned char> live;
  int last_step;
  int W_hist[GDNBEAM_MAX_T];
  // per-stage timing
  bool timing = false;
  std::vector<cudaEvent_t> ev_pool;
  std::vector<int> ev_stage;   // stage of each recorded pair
  size_t ev_used = 0;          // pairs recorded since the last read

  ~gdnbeam_ctx() {
    for (cudaEvent_t e : ev_pool) cudaEventDestroy(e);
  }
  // Brackets one stage with events when timing is on; returns the pair index.
  int tic(int stage, cudaStream_t s) {
    if (!timing) return -1;
    if (2 * (ev_used + 1) > ev_pool.size()) {
      for (int i = 0; i < 2; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        ev_pool.push_back(e);
      }
    }
    int idx = (int)ev_used++;
    if ((int)ev_stage.size() <= idx) ev_stage.resize(idx + 1);
    ev_stage[idx] = stage;
    cudaEventRecord(ev_pool[2 * idx], s);
    return idx;
  }
  void toc(int idx, cudaStream_t s) {
    if (idx >= 0) cudaEventRecord(ev_pool[2 * idx + 1], s);
  }

  size_t rec_rows() const { return (size_t)c.R * c.W_max; }
  char* gk(int layer, int j) const {
    return (char*)gtr_k + ((size_t)layer * (c.T - 1) + j) * rec_rows() * key_heads(c) * c.d_k * elem_size(c.dtype);
  }
  char* gd(int layer, int j) const {
    return (char*)gtr_delta + ((size_t)layer * (c.T - 1) + j) * rec_rows() * c.H * c.d_v * elem_size(c.dtype);
  }
  float* ga(int layer, int j) const {
    return gtr_alpha + ((size_t)layer * (c.T - 1) + j) * rec_rows() * c.H;
  }
};

namespace {

// Lays the workspace out from base (nullptr = dry run) and returns its size.
size_t carve(const gdnbeam_config& c, bool tc_gemm, char* base, gdnbeam_ctx* x,
             gdnbeam_footprint* fp) {
  const size_t es = elem_size(c.dtype);
  const size_t rows = (size_t)c.R * c.W_max;
  const size_t pf_rows = (size_t)c.R * c.L_max;
  const int depths = c.T > 1 ? c.T - 1 : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  // S_ctx is kept in fp32 whatever the storage type: it is read once per
  // (request, head) tile and shared by every beam, so its width costs little.
  size_t sctx_b = (size_t)c.R * c.layers * c.H * c.d_v * c.d_k * sizeof(float);
  size_t gk_b = (size_t)c.layers * depths * rows * key_heads(c) * c.d_k * es;
  size_t gd_b = (size_t)c.layers * depths * rows * c.H * c.d_v * es;
  size_t ga_b = (size_t)c.layers * depths * rows * c.H * sizeof(float);
  size_t anc_b = rows * c.T * sizeof(int32_t);
  char* p_sctx = take(sctx_b);
  char* p_gk = take(gk_b);
  char* p_gd = take(gd_b);
  char* p_ga = take(ga_b);
  char* p_anc0 = take(anc_b);
  char* p_anc1 = take(anc_b);
  char* p_sid0 = take(anc_b);
  char* p_sid1 = take(anc_b);
  char* p_u = take(rows * c.d_model * es);
  char* p_x = take(c.residual ? rows * c.d_model * sizeof(float) : 0);
  char* p_q = take(rows * key_heads(c) * c.d_k * es);
  char* p_v = take(rows * c.H * c.d_v * es);
  char* p_beta = take(rows * c.H * sizeof(float));
  char* p_o = take(rows * c.H * c.d_v * es);
  // the widest selection reads W_max rows per request and keeps W_max beams
  size_t sel_b = select_scratch_bytes(c.R, c.W_max, c.W_max, c.V);
  char* p_sel = take(sel_b);
  size_t gemm_b;
  if (tc_gemm) {
    gemm_b = 0;  // the tensor-core GEMMs need no scratch; logits partials go to tstats
  } else {
    size_t a = rows * (size_t)n_proj(c) * 4, b = rows * (size_t)c.V * 4;
    size_t p = pf_rows * (size_t)n_proj(c) * 4, r = (size_t)c.R * c.V * 4;
    gemm_b = a > b ? a : b;
    if (p > gemm_b) gemm_b = p;
    if (r > gemm_b) gemm_b = r;
  }
  char* p_gemm = take(gemm_b);
  const int n_hint_tiles = (c.V + kHintTile - 1) / kHintTile;
  char* p_tst = take((rows > (size_t)c.R ? rows : (size_t)c.R) * n_hint_tiles * sizeof(float2));
  const size_t st_b = c.state_path == 1 ? rows * c.layers * c.H * c.d_v * c.d_k * es : 0;
  char* p_st0 = take(st_b);
  char* p_st1 = take(st_b);
  char* p_sst = take(c.state_path ? (size_t)c.R * c.layers * c.H * c.d_v * c.d_k * es : 0);
  char* p_pfu = take(pf_rows * c.d_model * es);
  char* p_pfx = take(c.residual ? pf_rows * c.d_model * sizeof(float) : 0);
  char* p_pfq = take(pf_rows * key_heads(c) * c.d_k * es);
  char* p_pfk = take(pf_rows * key_heads(c) * c.d_k * es);
  char* p_pfv = take(pf_rows * c.H * c.d_v * es);
  char* p_pfa = take(pf_rows * c.H * sizeof(float));
  char* p_pfb = take(pf_rows * c.H * sizeof(float));
  char* p_pff = take((size_t)c.R * feat_dim(c) * es);
  const size_t pscr_b =
      (c.residual && tc_gemm && tc_prefill_supported(c)) ? prefill_out_scratch_bytes(c, c.L_max) : 0;
  char* p_pscr = take(pscr_b);
  if (x) {
    x->sctx = p_sctx; x->gtr_k = p_gk; x->gtr_delta = p_gd; x->gtr_alpha = (float*)p_ga;
    x->anc[0] = (int32_t*)p_anc0; x->anc[1] = (int32_t*)p_anc1;
    x->sid[0] = (int32_t*)p_sid0; x->sid[1] = (int32_t*)p_sid1;
    x->u = p_u; x->x = (float*)p_x; x->q = p_q; x->v = p_v; x->beta = (float*)p_beta;
    x->o = p_o; x->sel = p_sel; x->sel_bytes = sel_b; x->gemm = p_gemm; x->gemm_bytes = gemm_b;
    x->tstats = (float2*)p_tst; x->last_logits = nullptr; x->last_rows = 0;
    x->states[0] = p_st0; x->states[1] = p_st1; x->sctx_store = p_sst;
    x->pf_u = p_pfu; x->pf_x = (float*)p_pfx; x->pf_q = p_pfq; x->pf_k = p_pfk;
    x->pf_v = p_pfv; x->pf_alpha = (float*)p_pfa; x->pf_beta = (float*)p_pfb; x->pf_feat = p_pff;
    x->pf_scr = p_pscr; x->pf_scr_bytes = pscr_b;
  }
  if (fp) {
    fp->sctx_bytes = sctx_b;
    fp->record_elements = 1 + (size_t)c.d_v + c.d_k;
    fp->records_bytes = gk_b + gd_b + ga_b;
    fp->ancestry_bytes = 4 * anc_b;
    fp->fullstate_bytes = (size_t)c.R * c.layers * c.H * c.W_max * c.d_v * c.d_k * es;
    fp->workspace_bytes = off;
  }
  return off;
}

// Embedding rows of n tokens: u = E[tok] without a residual stream; with
// one, x = E[tok] (fp32) and, when the fused pass supports the width, u =
// the first layer's RMS-normalised rows in the same pass (*normed set).
int embed_rows(const gdnbeam_config& c, int n, const int32_t* tok, const void* E, void* u,
               float* x, unsigned* err, cudaStream_t s, bool* normed) {
  *normed = false;
  if (c.residual) {
    const int st = launch_gather_norm_rows(c.dtype, n, c.d_model, tok, c.V, E, x, u, err, s);
    if (st != GDNBEAM_EINVAL) {
      *normed = st == GDNBEAM_OK;
      return st;
    }
  }
  return launch_gather_rows(c.dtype, n, c.d_model, tok, c.V, E, u, c.residual ? x : nullptr, err,
                            s);
}

int project_any(const gdnbeam_config& c, bool tc, int n, const void* u, const void* Wp, void* q,
                void* k, void* v, float* alpha, float* beta, void* scratch, size_t scratch_bytes,
                const gdnbeam_dumps* d, cudaStream_t s) {
  if (tc) return launch_tc_project(c, n, u, Wp, q, k, v, alpha, beta, d, s);
  const int Np = n_proj(c);
  if (!scratch || scratch_bytes < (size_t)n * Np * 4) return GDNBEAM_EWORKSPACE;
  int st = launch_simt_gemm_nt(c.dtype, n, Np, c.d_model, u, c.d_model, Wp, c.d_model,
                               (float*)scratch, Np, s);
  if (st) return st;
  return launch_proj_epilogue(c, n, (const float*)scratch, q, k, v, alpha, beta, d, s);
}

// Logits for n rows. tstats (may be NULL on the CUDA-core path) receives the
// per (row, 256-code tile) maximum and sum of exp; the tensor-core path
// needs it as its partial buffer.
int logits_any(const gdnbeam_config& c, bool tc, int n, const void* feat, const void* Wo,
               void* z, float* lse, void* scratch, size_t scratch_bytes, float2* tstats,
               const gdnbeam_dumps* d, cudaStream_t s) {
  if (tc) {
    if (!tstats) return GDNBEAM_EWORKSPACE;
    return launch_tc_logits(c, n, feat, Wo, z, lse, tstats, d, s);
  }
  const int F = feat_dim(c);
  if (!scratch || scratch_bytes < (size_t)n * c.V * 4) return GDNBEAM_EWORKSPACE;
  int st = launch_simt_gemm_nt(c.dtype, n, c.V, F, feat, F, Wo, F, (float*)scratch, c.V, s);
  if (st) return st;
  st = launch_logits_rows(c.dtype, n, c.V, (const float*)scratch, z, lse,
                          d ? d->logits : nullptr, s);
  if (st || !tstats) return st;
  return launch_tile_max(c.dtype, n, c.V, z, tstats, error_word(), s);
}

gdnbeam_dumps layer_dumps(const gdnbeam_dumps* d, const gdnbeam_config& c, int layer, size_t n) {
  gdnbeam_dumps o{};
  if (!d) return o;
  auto sh = [&](float* p, size_t per) { return p ? p + (size_t)layer * n * per : nullptr; };
  o.q = sh(d->q, (size_t)key_heads(c) * c.d_k);
  o.k = sh(d->k, (size_t)key_heads(c) * c.d_k);
  o.v = sh(d->v, (size_t)c.H * c.d_v);
  o.alpha = sh(d->alpha, c.H);
  o.beta = sh(d->beta, c.H);
  o.delta = sh(d->delta, (size_t)c.H * c.d_v);
  o.o = sh(d->o, (size_t)c.H * c.d_v);
  o.logits = d->logits;
  return o;
}

}  // namespace

extern "C" {

const char* gdnbeam_strerror(int st) {
  switch (st) {
    case GDNBEAM_OK: return "ok";
    case GDNBEAM_EINVAL: return "invalid argument";
    case GDNBEAM_EUNSUPPORTED: return "unsupported shape or dtype";
    case GDNBEAM_EWORKSPACE: return "workspace or scratch too small";
    case GDNBEAM_ESTATE: return "call out of sequence";
    case GDNBEAM_ECUDA: return "CUDA error";
    case GDNBEAM_EDEVICE: return "device-side error";
    case GDNBEAM_ENOMEM: return "host allocation failed";
    default: return "unknown status";
  }
}

int gdnbeam_footprint_of(const gdnbeam_config* cfg, gdnbeam_footprint* out) {
  int st = validate(cfg);
  if (st) return st;
  if (!out) return GDNBEAM_EINVAL;
  carve(*cfg, tc_gemm_supported(*cfg), nullptr, nullptr, out);
  return GDNBEAM_OK;
}

int gdnbeam_create(const gdnbeam_config* cfg, const gdnbeam_weights* w, void* workspace,
                   size_t workspace_bytes, gdnbeam_ctx** out) {
  if (!out) return GDNBEAM_EINVAL;
  *out = nullptr;
  int st = validate(cfg);
  if (st) return st;
  if (!w || !w->E || !w->W_proj || !w->W_o || !workspace) return GDNBEAM_EINVAL;
  if (((uintptr_t)workspace & 255) != 0) return GDNBEAM_EINVAL;
  const bool tc = tc_gemm_supported(*cfg);
  if (workspace_bytes < carve(*cfg, tc, nullptr, nullptr, nullptr)) return GDNBEAM_EWORKSPACE;
  gdnbeam_ctx* x = new (std::nothrow) gdnbeam_ctx();
  if (!x) return GDNBEAM_ENOMEM;
  x->c = *cfg;
  x->w = *w;
  x->ws = (char*)workspace;
  x->ws_bytes = workspace_bytes;
  x->tc_gemm = tc;
  x->tc_replay = tc_replay_supported(cfg->dtype, cfg->d_k, cfg->d_v);
  carve(*cfg, tc, (char*)workspace, x, nullptr);
  if (cfg->state_path)
    snprintf(x->variant, sizeof(x->variant), "proj=%s state=%s logits=%s select=bound",
             tc ? "tc" : "simt", cfg->state_path == 1 ? "fullstate" : "replayssm",
             tc ? "tc" : "simt");
  else
    snprintf(x->variant, sizeof(x->variant), "proj=%s replay=%s logits=%s select=bound",
             tc ? "tc" : "simt", x->tc_replay ? "tc" : "simt", tc ? "tc" : "simt");
  x->prefilled = 0;
  x->live.assign(cfg->R, 0);
  x->last_step = -1;
  *out = x;
  return GDNBEAM_OK;
}

void gdnbeam_destroy(gdnbeam_ctx* ctx) { delete ctx; }

const char* gdnbeam_variant(const gdnbeam_ctx* ctx) { return ctx ? ctx->variant : ""; }

int gdnbeam_reset(gdnbeam_ctx* ctx, const int32_t* request_mask) {
  if (!ctx) return GDNBEAM_EINVAL;
  const int R = ctx->c.R;
  for (int r = 0; r < R; ++r)
    if (!request_mask || request_mask[r]) ctx->live[r] = 0;
  ctx->prefilled = 0;
  ctx->last_step = -1;
  return GDNBEAM_OK;
}

}  // extern "C"

namespace {

// Prefill of cp.R requests whose prompts are packed [cp.R][L] at prompt:
// S_ctx of request i goes to sctx_base + i * (layers*H*d_v*d_k), its root
// row's logits and lse to root_logits / root_lse row i, and (baselines) the
// storage copy of S_ctx to sctx_store_base. cp is the context's
// configuration with R set to the requests of this pass.
int prefill_pass(gdnbeam_ctx* ctx, const gdnbeam_config& c, const int32_t* prompt, int L,
                 float* sctx_base, void* sctx_store_base, void* root_logits, float* root_lse,
                 cudaStream_t s) {
  unsigned* err = err_ptr();
  const int n = c.R * L;
  const size_t es = elem_size(c.dtype);
  const int Np = n_proj(c);
  const long long rstride = (long long)c.layers * c.H * c.d_v * c.d_k;
  int ev = ctx->tic(GDNBEAM_STAGE_EMBED, s);
  bool normed = false;  // pf_u already holds layer 0's normalised rows
  int st = embed_rows(c, n, prompt, ctx->w.E, ctx->pf_u, ctx->pf_x, err, s, &normed);
  ctx->toc(ev, s);
  if (st) return st;
  for (int layer = 0; layer < c.layers; ++layer) {
    if (c.residual && !(layer == 0 && normed)) {
      ev = ctx->tic(GDNBEAM_STAGE_EMBED, s);
      st = launch_rmsnorm_rows(c.dtype, n, c.d_model, ctx->pf_x, c.d_model, ctx->pf_u, s);
      ctx->toc(ev, s);
      if (st) return st;
    }
    const char* Wp = (const char*)ctx->w.W_proj + (size_t)layer * Np * c.d_model * es;
    float* sc = sctx_base + (size_t)layer * c.H * c.d_v * c.d_k;
    if (ctx->tc_gemm && tc_prefill_supported(c) && !c.residual) {
      // The chunked prefill reads the query only at each request's last
      // token: the projection over all prompt rows skips the query columns,
      // and a second one forms the last rows' queries (into rows 0 .. R-1
      // of the query buffer).
      ev = ctx->tic(GDNBEAM_STAGE_PROJECT, s);
      st = launch_tc_project(c, n, ctx->pf_u, Wp, ctx->pf_q, ctx->pf_k, ctx->pf_v, ctx->pf_alpha,
                             ctx->pf_beta, nullptr, s, PROJ_NO_Q);
      if (!st)
        st = launch_tc_project(c, c.R, (const char*)ctx->pf_u + (size_t)(L - 1) * c.d_model * es, Wp,
                               ctx->pf_q, nullptr, nullptr, nullptr, nullptr, nullptr, s,
                               PROJ_Q_ONLY, (long long)L * c.d_model);
      ctx->toc(ev, s);
      if (st) return st;
      ev = ctx->tic(GDNBEAM_STAGE_PREFILL, s);
      st = launch_prefill_tc(c, L, ctx->pf_q, (long long)key_heads(c) * c.d_k, ctx->pf_k, ctx->pf_v,
                             ctx->pf_alpha, ctx->pf_beta, sc, rstride, ctx->pf_feat, s);
      ctx->toc(ev, s);
      if (st) return st;
      continue;
    }
    ev = ctx->tic(GDNBEAM_STAGE_PROJECT, s);
    st = project_any(c, ctx->tc_gemm, n, ctx->pf_u, Wp, ctx->pf_q, ctx->pf_k, ctx->pf_v,
                     ctx->pf_alpha, ctx->pf_beta, ctx->gemm, ctx->gemm_bytes, nullptr, s);
    ctx->toc(ev, s);
    if (st) return st;
    ev = ctx->tic(GDNBEAM_STAGE_PREFILL, s);
    // (stacked layers with tensor cores: the chunked prefill, every
    // position's o added to the stream through pf_scr)
    st = launch_prefill_scan(c, L, ctx->pf_q, ctx->pf_k, ctx->pf_v, ctx->pf_alpha, ctx->pf_beta,
                             sc, rstride, c.residual ? nullptr : ctx->pf_feat,
                             c.residual ? ctx->pf_x : nullptr, s, ctx->pf_scr, ctx->pf_scr_bytes);
    ctx->toc(ev, s);
    if (st) return st;
  }
  if (c.state_path) {  // the baselines read S_ctx in the storage type
    st = launch_to_storage(c.dtype, (size_t)c.R * rstride, sctx_base, sctx_store_base, s);
    if (st) return st;
  }
  if (c.residual) {
    st = launch_rmsnorm_rows(c.dtype, c.R, c.d_model, ctx->pf_x + (size_t)(L - 1) * c.d_model,
                             (long long)L * c.d_model, ctx->pf_feat, s);
    if (st) return st;
  }
  ev = ctx->tic(GDNBEAM_STAGE_LOGITS, s);
  st = logits_any(c, ctx->tc_gemm, c.R, ctx->pf_feat, ctx->w.W_o, root_logits, root_lse,
                  ctx->gemm, ctx->gemm_bytes, ctx->tstats, nullptr, s);
  ctx->toc(ev, s);
  return st;
}

}  // namespace

extern "C" {

int gdnbeam_prefill_state(gdnbeam_ctx* ctx, const int32_t* prompt, int L, void* root_logits,
                          float* root_lse, gdnbeam_stream_t stream) {
  if (!ctx || !prompt || !root_logits || !root_lse) return GDNBEAM_EINVAL;
  const gdnbeam_config& c = ctx->c;
  if (L < 1 || L > c.L_max) return GDNBEAM_EINVAL;
  ctx->prefilled = 0;
  ctx->live.assign(c.R, 0);
  ctx->last_logits = nullptr;
  int st = prefill_pass(ctx, c, prompt, L, (float*)ctx->sctx, ctx->sctx_store, root_logits,
                        root_lse, (cudaStream_t)stream);
  if (st) return st;
  ctx->last_logits = root_logits;
  ctx->last_rows = c.R;
  ctx->live.assign(c.R, 1);
  ctx->prefilled = 1;
  ctx->last_step = -1;
  return GDNBEAM_OK;
}

int gdnbeam_prefill_requests(gdnbeam_ctx* ctx, const int32_t* request_ids, int count,
                             const int32_t* prompts, int L, void* root_logits, float* root_lse,
                             gdnbeam_stream_t stream) {
  if (!ctx || count < 0) return GDNBEAM_EINVAL;
  const gdnbeam_config& c = ctx->c;
  if (count == 0) return GDNBEAM_OK;
  if (!request_ids || !prompts || !root_logits || !root_lse) return GDNBEAM_EINVAL;
  if (L < 1 || L > c.L_max || count > c.R) return GDNBEAM_EINVAL;
  std::vector<unsigned char> seen(c.R, 0);
  for (int i = 0; i < count; ++i) {
    const int r = request_ids[i];
    if (r < 0 || r >= c.R || seen[r]) return GDNBEAM_EINVAL;
    seen[r] = 1;
  }
  const size_t es = elem_size(c.dtype);
  const size_t rstride = (size_t)c.layers * c.H * c.d_v * c.d_k;
  gdnbeam_config one = c;
  one.R = 1;
  // The root rows written here are not the rows a selection would find the
  // logits stage's tile maxima for: the selection computes its own.
  ctx->last_logits = nullptr;
  ctx->last_rows = 0;
  ctx->last_step = -1;
  for (int i = 0; i < count; ++i) {
    const int r = request_ids[i];
    ctx->live[r] = 0;
    ctx->prefilled = 0;
    int st = prefill_pass(ctx, one, prompts + (size_t)i * L, L, (float*)ctx->sctx + r * rstride,
                          ctx->sctx_store ? (char*)ctx->sctx_store + r * rstride * es : nullptr,
                          (char*)root_logits + (size_t)r * c.V * es, root_lse + r,
                          (cudaStream_t)stream);
    if (st) return st;
    ctx->live[r] = 1;
  }
  bool all = true;
  for (int r = 0; r < c.R; ++r) all = all && ctx->live[r];
  ctx->prefilled = all ? 1 : 0;
  return GDNBEAM_OK;
}

int gdnbeam_step(gdnbeam_ctx* ctx, int t, int W_t, const int32_t* parents, const int32_t* tokens,
                 void* logits, float* lse, const gdnbeam_dumps* dumps, gdnbeam_stream_t stream) {
  if (!ctx || !tokens || !logits || !lse) return GDNBEAM_EINVAL;
  const gdnbeam_config& c = ctx->c;
  if (t < 0 || t > c.T - 2 || W_t < 1 || W_t > c.W_max) return GDNBEAM_EINVAL;
  if (t > 0 && !parents) return GDNBEAM_EINVAL;
  if (!ctx->prefilled) return GDNBEAM_ESTATE;
  if (t > 0 && ctx->last_step != t - 1) return GDNBEAM_ESTATE;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned* err = err_ptr();
  const int n = c.R * W_t;
  const size_t es = elem_size(c.dtype);
  const int Np = n_proj(c);
  const int W_prev = t > 0 ? ctx->W_hist[t - 1] : 1;
  const int cur = t & 1;
  ctx->last_step = -2;  // invalid until this call succeeds
  int ev = ctx->tic(GDNBEAM_STAGE_ANCESTRY, s);
  int st = launch_ancestry(c.R, t, c.T, c.V, W_prev, W_t, parents, tokens, ctx->anc[cur ^ 1],
                           ctx->sid[cur ^ 1], ctx->anc[cur], ctx->sid[cur], err, s);
  ctx->toc(ev, s);
  if (st) return st;
  ev = ctx->tic(GDNBEAM_STAGE_EMBED, s);
  bool normed = false;  // u already holds layer 0's normalised rows
  st = embed_rows(c, n, tokens, ctx->w.E, ctx->u, ctx->x, err, s, &normed);
  ctx->toc(ev, s);
  if (st) return st;
  for (int layer = 0; layer < c.layers; ++layer) {
    if (c.residual && !(layer == 0 && normed)) {
      ev = ctx->tic(GDNBEAM_STAGE_EMBED, s);
      st = launch_rmsnorm_rows(c.dtype, n, c.d_model, ctx->x, c.d_model, ctx->u, s);
      ctx->toc(ev, s);
      if (st) return st;
    }
    gdnbeam_dumps ld = layer_dumps(dumps, c, layer, n);
    const char* Wp = (const char*)ctx->w.W_proj + (size_t)layer * Np * c.d_model * es;
    ev = ctx->tic(GDNBEAM_STAGE_PROJECT, s);
    st = project_any(c, ctx->tc_gemm, n, ctx->u, Wp, ctx->q, ctx->gk(layer, t), ctx->v,
                     ctx->ga(layer, t), ctx->beta, ctx->gemm, ctx->gemm_bytes, &ld, s);
    ctx->toc(ev, s);
    if (st) return st;
    ReplayArgs a{};
    a.R = c.R; a.H = c.H; a.d_k = c.d_k; a.d_v = c.d_v; a.t = t; a.W_t = W_t; a.Hk = key_heads(c);
    a.sctx = (const float*)ctx->sctx + (size_t)layer * c.H * c.d_v * c.d_k;
    a.sctx_rstride = (long long)c.layers * c.H * c.d_v * c.d_k;
    a.q = ctx->q; a.k = ctx->gk(layer, t); a.v = ctx->v;
    a.alpha = ctx->ga(layer, t); a.beta = ctx->beta;
    for (int j = 0; j < t; ++j) {
      a.depth[j].k = ctx->gk(layer, j);
      a.depth[j].delta = ctx->gd(layer, j);
      a.depth[j].alpha = ctx->ga(layer, j);
      a.depth[j].W_j = ctx->W_hist[j];
    }
    a.anc = ctx->anc[cur]; a.anc_stride = c.T;
    // with a residual stream o_t is only added to it (the features read x)
    a.delta_out = ctx->gd(layer, t); a.o_out = c.residual ? nullptr : ctx->o;
    a.x_inout = c.residual ? ctx->x : nullptr;
    a.delta_dump = ld.delta; a.o_dump = ld.o;
    a.err = err;
    ev = ctx->tic(GDNBEAM_STAGE_REPLAY, s);
    if (c.state_path == 2) {
      ReplaySsmArgs g{};
      g.R = c.R; g.H = c.H; g.d_k = c.d_k; g.d_v = c.d_v; g.t = t; g.W_t = W_t; g.Hk = key_heads(c);
      g.sctx_store = (const char*)ctx->sctx_store + (size_t)layer * c.H * c.d_v * c.d_k * es;
      g.sctx_rstride = a.sctx_rstride;
      g.q = a.q; g.k = a.k; g.v = a.v; g.alpha = a.alpha; g.beta = a.beta;
      for (int j = 0; j < t; ++j) g.depth[j] = a.depth[j];
      g.anc = a.anc; g.anc_stride = a.anc_stride;
      g.delta_out = a.delta_out; g.o_out = a.o_out; g.x_inout = a.x_inout;
      g.delta_dump = a.delta_dump; g.o_dump = a.o_dump; g.err = err;
      st = launch_replayssm(c.dtype, g, s);
    } else if (c.state_path) {
      FullStateArgs f{};
      f.R = c.R; f.H = c.H; f.d_k = c.d_k; f.d_v = c.d_v; f.t = t; f.W_t = W_t; f.Hk = key_heads(c);
      f.W_prev = W_prev; f.layers = c.layers; f.layer = layer;
      f.sctx_store = (const char*)ctx->sctx_store + (size_t)layer * c.H * c.d_v * c.d_k * es;
      f.sctx_rstride = a.sctx_rstride;
      f.states_prev = ctx->states[cur ^ 1]; f.states_cur = ctx->states[cur];
      f.parents = parents;
      f.q = a.q; f.k = a.k; f.v = a.v; f.alpha = a.alpha; f.beta = a.beta;
      f.delta_out = a.delta_out; f.o_out = a.o_out; f.x_inout = a.x_inout;
      f.delta_dump = a.delta_dump; f.o_dump = a.o_dump; f.err = err;
      st = launch_fullstate(c.dtype, f, s);
    } else {
      st = ctx->tc_replay ? launch_tc_replay(a, s) : launch_replay(c.dtype, a, s);
    }
    ctx->toc(ev, s);
    if (st) return st;
  }
  const void* feat = ctx->o;
  if (c.residual) {
    ev = ctx->tic(GDNBEAM_STAGE_EMBED, s);
    st = launch_rmsnorm_rows(c.dtype, n, c.d_model, ctx->x, c.d_model, ctx->u, s);
    ctx->toc(ev, s);
    if (st) return st;
    feat = ctx->u;
  }
  gdnbeam_dumps zd{};
  if (dumps) zd.logits = dumps->logits;
  ev = ctx->tic(GDNBEAM_STAGE_LOGITS, s);
  st = logits_any(c, ctx->tc_gemm, n, feat, ctx->w.W_o, logits, lse, ctx->gemm, ctx->gemm_bytes,
                  ctx->tstats, &zd, s);
  ctx->last_logits = logits;
  ctx->last_rows = n;
  ctx->toc(ev, s);
  if (st) return st;
  ctx->W_hist[t] = W_t;
  ctx->last_step = t;
  return GDNBEAM_OK;
}

int gdnbeam_select(gdnbeam_ctx* ctx, int t, int W_t, int W_next, const void* logits,
                   const float* lse, const float* cum, const float* bias, int32_t* parents,
                   int32_t* tokens, float* cum_next, gdnbeam_stream_t stream) {
  if (!ctx) return GDNBEAM_EINVAL;
  const gdnbeam_config& c = ctx->c;
  if (t < -1 || t > c.T - 2) return GDNBEAM_EINVAL;
  if (t == -1 && W_t != 1) return GDNBEAM_EINVAL;
  if (W_t < 1 || W_t > c.W_max || W_next < 1 || W_next > c.W_max) return GDNBEAM_EINVAL;
  if (!logits || !lse || !parents || !tokens || !cum_next) return GDNBEAM_EINVAL;
  if ((long long)W_next > (long long)W_t * c.V) return GDNBEAM_EINVAL;
  // The tile maxima the logits stage left behind bound the selection when
  // these are the logits it wrote; the result is exact either way.
  const float2* hint =
      (logits == ctx->last_logits && ctx->last_rows == c.R * W_t) ? ctx->tstats : nullptr;
  int ev = ctx->tic(GDNBEAM_STAGE_SELECT, (cudaStream_t)stream);
  int st = launch_select(c.R, W_t, W_next, c.V, c.dtype, logits, lse, cum, bias, hint, parents,
                         tokens, cum_next, ctx->sel, err_ptr(), (cudaStream_t)stream);
  ctx->toc(ev, (cudaStream_t)stream);
  return st;
}

int gdnbeam_get_paths(gdnbeam_ctx* ctx, int W_final, const int32_t* parents,
                      const int32_t* tokens, int32_t* sid, gdnbeam_stream_t stream) {
  if (!ctx || !tokens || !sid) return GDNBEAM_EINVAL;
  const gdnbeam_config& c = ctx->c;
  if (W_final < 1 || W_final > c.W_max) return GDNBEAM_EINVAL;
  const int t = c.T - 1;
  if (t > 0) {
    if (!parents) return GDNBEAM_EINVAL;
    if (ctx->last_step != c.T - 2) return GDNBEAM_ESTATE;
  }
  const int W_prev = t > 0 ? ctx->W_hist[t - 1] : 1;
  const int prev = (t - 1) & 1;
  return launch_ancestry(c.R, t, c.T, c.V, W_prev, W_final, parents, tokens, nullptr,
                         t > 0 ? ctx->sid[prev] : nullptr, nullptr, sid, err_ptr(),
                         (cudaStream_t)stream);
}

int gdnbeam_timing(gdnbeam_ctx* ctx, int enable) {
  if (!ctx) return GDNBEAM_EINVAL;
  ctx->timing = enable != 0;
  ctx->ev_used = 0;
  return GDNBEAM_OK;
}

int gdnbeam_stage_times(gdnbeam_ctx* ctx, float* ms, int* count) {
  if (!ctx || !ms) return GDNBEAM_EINVAL;
  for (int i = 0; i < GDNBEAM_NSTAGES; ++i) {
    ms[i] = 0.0f;
    if (count) count[i] = 0;
  }
  for (size_t i = 0; i < ctx->ev_used; ++i) {
    GDN_CUDA(cudaEventSynchronize(ctx->ev_pool[2 * i + 1]));
    float t = 0.0f;
    GDN_CUDA(cudaEventElapsedTime(&t, ctx->ev_pool[2 * i], ctx->ev_pool[2 * i + 1]));
    ms[ctx->ev_stage[i]] += t;
    if (count) count[ctx->ev_stage[i]] += 1;
  }
  ctx->ev_used = 0;
  return GDNBEAM_OK;
}

long long gdnbeam_launches(int clear) {
  return clear ? g_launches.exchange(0) : g_launches.load();
}

int gdnbeam_read_sctx(gdnbeam_ctx* ctx, float* out, gdnbeam_stream_t stream) {
  if (!ctx || !out) return GDNBEAM_EINVAL;
  if (!ctx->prefilled) return GDNBEAM_ESTATE;
  const gdnbeam_config& c = ctx->c;
  size_t bytes = (size_t)c.R * c.layers * c.H * c.d_v * c.d_k * sizeof(float);
  GDN_CUDA(cudaMemcpyAsync(out, ctx->sctx, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
  return GDNBEAM_OK;
}

int gdnbeam_device_status(int clear) {
  unsigned* p = err_ptr();
  if (!p) return GDNBEAM_ECUDA;
  unsigned v = 0;
  GDN_CUDA(cudaDeviceSynchronize());
  GDN_CUDA(cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost));
  if (clear && v) {
    unsigned z = 0;
    GDN_CUDA(cudaMemcpy(p, &z, sizeof(z), cudaMemcpyHostToDevice));
  }
  return (int)v;
}

int gdnbeam_status(gdnbeam_ctx* ctx, gdnbeam_stream_t stream) {
  if (!ctx) return GDNBEAM_EINVAL;
  GDN_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  GDN_CUDA(cudaGetLastError());
  int v = gdnbeam_device_status(1);
  if (v < 0) return v;
  return v ? GDNBEAM_EDEVICE : GDNBEAM_OK;
}

// ---------------------------------------------------------------------------
// Tensor-level calls
// ---------------------------------------------------------------------------

size_t gdnbeam_project_scratch_bytes(const gdnbeam_config* cfg, int n) {
  if (validate(cfg) || n < 0) return 0;
  if (tc_gemm_supported(*cfg)) return 0;
  return (size_t)n * n_proj(*cfg) * 4;
}

int gdnbeam_project(const gdnbeam_config* cfg, int n, const void* u, const void* W_proj, void* q,
                    void* k, void* v, float* alpha, float* beta, void* scratch,
                    size_t scratch_bytes, const gdnbeam_dumps* dumps, gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  if (n < 0 || !u || !W_proj || !q || !k || !v || !alpha || !beta) return GDNBEAM_EINVAL;
  if (n == 0) return GDNBEAM_OK;
  return project_any(*cfg, tc_gemm_supported(*cfg), n, u, W_proj, q, k, v, alpha, beta, scratch,
                     scratch_bytes, dumps, (cudaStream_t)stream);
}

int gdnbeam_replay(const gdnbeam_config* cfg, int t, int W_t, const float* sctx,
                   long long sctx_rstride, const void* q, const void* k, const void* v,
                   const float* alpha, const float* beta, const gdnbeam_records* depth,
                   const int32_t* anc, int anc_stride, void* delta_out, void* o_out,
                   float* x_inout, const gdnbeam_dumps* dumps, gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  const gdnbeam_config& c = *cfg;
  if (t < 0 || t >= GDNBEAM_MAX_T || W_t < 1 || !sctx || !q || !k || !v || !alpha || !beta ||
      !delta_out || !o_out)
    return GDNBEAM_EINVAL;
  if (t > 0 && (!depth || !anc || anc_stride < t)) return GDNBEAM_EINVAL;
  ReplayArgs a{};
  a.R = c.R; a.H = c.H; a.d_k = c.d_k; a.d_v = c.d_v; a.t = t; a.W_t = W_t; a.Hk = key_heads(c);
  a.sctx = sctx; a.sctx_rstride = sctx_rstride;
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  for (int j = 0; j < t; ++j) {
    if (!depth[j].k || !depth[j].delta || !depth[j].alpha || depth[j].W_j < 1) return GDNBEAM_EINVAL;
    a.depth[j] = depth[j];
  }
  a.anc = anc; a.anc_stride = anc_stride;
  a.delta_out = delta_out; a.o_out = o_out; a.x_inout = x_inout;
  a.delta_dump = dumps ? dumps->delta : nullptr;
  a.o_dump = dumps ? dumps->o : nullptr;
  a.err = err_ptr();
  if (tc_replay_supported(c.dtype, c.d_k, c.d_v)) return launch_tc_replay(a, (cudaStream_t)stream);
  return launch_replay(c.dtype, a, (cudaStream_t)stream);
}

int gdnbeam_fullstate_step(const gdnbeam_config* cfg, int t, int W_t, int W_prev,
                           const void* sctx_store, long long sctx_rstride,
                           const void* states_prev, void* states_cur, const int32_t* parents,
                           const void* q, const void* k, const void* v, const float* alpha,
                           const float* beta, void* delta_out, void* o_out,
                           gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  const gdnbeam_config& c = *cfg;
  if (c.d_k > 128 || c.d_v > 128) return GDNBEAM_EUNSUPPORTED;
  if (t < 0 || t >= GDNBEAM_MAX_T || W_t < 1 || !sctx_store || !states_cur || !q || !k || !v ||
      !alpha || !beta || !delta_out || !o_out)
    return GDNBEAM_EINVAL;
  if (t > 0 && (!states_prev || !parents || W_prev < 1)) return GDNBEAM_EINVAL;
  FullStateArgs f{};
  f.R = c.R; f.H = c.H; f.d_k = c.d_k; f.d_v = c.d_v; f.t = t; f.W_t = W_t; f.Hk = key_heads(c);
  f.W_prev = t > 0 ? W_prev : 1; f.layers = 1; f.layer = 0;
  f.sctx_store = sctx_store; f.sctx_rstride = sctx_rstride;
  f.states_prev = states_prev; f.states_cur = states_cur; f.parents = parents;
  f.q = q; f.k = k; f.v = v; f.alpha = alpha; f.beta = beta;
  f.delta_out = delta_out; f.o_out = o_out;
  f.err = err_ptr();
  return launch_fullstate(c.dtype, f, (cudaStream_t)stream);
}

int gdnbeam_replayssm_step(const gdnbeam_config* cfg, int t, int W_t, const void* sctx_store,
                           long long sctx_rstride, const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, const gdnbeam_records* depth,
                           const int32_t* anc, int anc_stride, void* delta_out, void* o_out,
                           gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  const gdnbeam_config& c = *cfg;
  if (c.d_k > 128 || c.d_v > 128) return GDNBEAM_EUNSUPPORTED;
  if (t < 0 || t >= GDNBEAM_MAX_T || W_t < 1 || !sctx_store || !q || !k || !v || !alpha ||
      !beta || !delta_out || !o_out)
    return GDNBEAM_EINVAL;
  if (t > 0 && (!depth || !anc || anc_stride < t)) return GDNBEAM_EINVAL;
  ReplaySsmArgs g{};
  g.R = c.R; g.H = c.H; g.d_k = c.d_k; g.d_v = c.d_v; g.t = t; g.W_t = W_t; g.Hk = key_heads(c);
  g.sctx_store = sctx_store; g.sctx_rstride = sctx_rstride;
  g.q = q; g.k = k; g.v = v; g.alpha = alpha; g.beta = beta;
  for (int j = 0; j < t; ++j) {
    if (!depth[j].k || !depth[j].delta || !depth[j].alpha || depth[j].W_j < 1) return GDNBEAM_EINVAL;
    g.depth[j] = depth[j];
  }
  g.anc = anc; g.anc_stride = anc_stride;
  g.delta_out = delta_out; g.o_out = o_out;
  g.err = err_ptr();
  return launch_replayssm(c.dtype, g, (cudaStream_t)stream);
}

size_t gdnbeam_logits_scratch_bytes(const gdnbeam_config* cfg, int n) {
  if (validate(cfg) || n < 0) return 0;
  if (tc_gemm_supported(*cfg)) return tc_logits_scratch_bytes(*cfg, n);
  return (size_t)n * cfg->V * 4;
}

int gdnbeam_logits(const gdnbeam_config* cfg, int n, const void* feat, const void* W_o, void* z,
                   float* lse, void* scratch, size_t scratch_bytes, const gdnbeam_dumps* dumps,
                   gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  if (n < 0 || !feat || !W_o || !z || !lse) return GDNBEAM_EINVAL;
  if (n == 0) return GDNBEAM_OK;
  const bool tc = tc_gemm_supported(*cfg);
  if (tc && scratch_bytes < tc_logits_scratch_bytes(*cfg, n)) return GDNBEAM_EWORKSPACE;
  return logits_any(*cfg, tc, n, feat, W_o, z, lse, scratch, scratch_bytes,
                    tc ? (float2*)scratch : nullptr, dumps, (cudaStream_t)stream);
}

size_t gdnbeam_select_scratch_bytes(int R, int W_t, int W_next, int V) {
  if (R < 1 || W_t < 1 || W_next < 1 || V < 1) return 0;
  return select_scratch_bytes(R, W_t, W_next, V);
}

int gdnbeam_select_topw(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                        const float* lse, const float* cum, const float* bias, int32_t* parents,
                        int32_t* tokens, float* cum_next, void* scratch, size_t scratch_bytes,
                        gdnbeam_stream_t stream) {
  if (R < 1 || W_t < 1 || W_next < 1 || V < 2 || !logits || !lse || !parents || !tokens ||
      !cum_next || !scratch)
    return GDNBEAM_EINVAL;
  if (dtype != GDNBEAM_F32 && dtype != GDNBEAM_BF16) return GDNBEAM_EUNSUPPORTED;
  if ((long long)W_t * V >= (1ll << 31) || (long long)W_next > (long long)W_t * V)
    return GDNBEAM_EINVAL;
  if (scratch_bytes < select_scratch_bytes(R, W_t, W_next, V)) return GDNBEAM_EWORKSPACE;
  return launch_select(R, W_t, W_next, V, dtype, logits, lse, cum, bias, nullptr, parents, tokens,
                       cum_next, scratch, err_ptr(), (cudaStream_t)stream);
}

int gdnbeam_ancestry(int R, int t, int T, int V, int W_prev, int W_t, const int32_t* parents,
                     const int32_t* tokens, const int32_t* anc_prev, const int32_t* sid_prev,
                     int32_t* anc_out, int32_t* sid_out, gdnbeam_stream_t stream) {
  if (R < 1 || t < 0 || t >= T || T > GDNBEAM_MAX_T || W_t < 1 || W_prev < 1 || !tokens ||
      !sid_out)
    return GDNBEAM_EINVAL;
  if (t > 0 && (!parents || !sid_prev)) return GDNBEAM_EINVAL;
  if (t > 1 && anc_out && !anc_prev) return GDNBEAM_EINVAL;
  return launch_ancestry(R, t, T, V, W_prev, W_t, parents, tokens, anc_prev, sid_prev, anc_out,
                         sid_out, err_ptr(), (cudaStream_t)stream);
}

size_t gdnbeam_prefill_scan_scratch_bytes(const gdnbeam_config* cfg, int L, int with_residual) {
  if (validate(cfg) || L < 1 || !with_residual) return 0;
  return tc_prefill_supported(*cfg) ? prefill_out_scratch_bytes(*cfg, L) : 0;
}

int gdnbeam_prefill_scan(const gdnbeam_config* cfg, int L, const void* q, const void* k,
                         const void* v, const float* alpha, const float* beta, float* sctx_out,
                         long long sctx_rstride, void* o_last, float* x_inout, void* scratch,
                         size_t scratch_bytes, gdnbeam_stream_t stream) {
  int st = validate(cfg);
  if (st) return st;
  if (L < 1 || !q || !k || !v || !alpha || !beta || !sctx_out) return GDNBEAM_EINVAL;
  if (x_inout && scratch_bytes < gdnbeam_prefill_scan_scratch_bytes(cfg, L, 1)) return GDNBEAM_EWORKSPACE;
  return launch_prefill_scan(*cfg, L, q, k, v, alpha, beta, sctx_out, sctx_rstride, o_last,
                             x_inout, (cudaStream_t)stream, scratch, scratch_bytes);
}

}  // extern "C"
