/*
 * gdnbeam — large-beam Gated DeltaNet decoding with a shared context state,
 * append-only transition records, an ancestry index and projection replay.
 *
 * Sources, named by page title:
 *   OneLA   "OneLA: Scaling Linear-Attention Decoding to Large Beams in
 *            Generative Recommendation" (review page)
 *   RecoGEM "RecoGEM: A Serving System for Production-Scale Generative
 *            Recommendation"
 *
 * Conventions for every call below.
 *   - Pointers are DEVICE pointers owned by the caller unless marked (host).
 *     The library never allocates device memory: the context carves all it
 *     needs out of one caller-allocated workspace.
 *   - Calls are asynchronous on the given stream. They return a status:
 *     0 on success or a negative GDNBEAM_E* code. Argument errors are found
 *     on the host before anything is launched. Errors found on the device
 *     (an out-of-range token, parent or slot index; a non-finite score) set a
 *     device error word, skip the offending access and are reported by
 *     gdnbeam_status()/gdnbeam_device_status(); the device never traps.
 *   - Storage type is fp32 (GDNBEAM_F32) or bf16 (GDNBEAM_BF16) for every
 *     tensor marked "storage"; accumulation is always fp32.
 *   - Per-beam tensors of one decode call are packed [R][W_t][...]: request
 *     r's beam b is row r*W_t + b.
 *   - Decode call t (0 <= t <= T-2) runs on the beams kept by selection t
 *     and feeds selection t+1; selection 0 reads the prefill row. A beam's
 *     slot at depth j is its ancestor's row index at decode call j.
 *   - gdnbeam_step, gdnbeam_select and gdnbeam_get_paths only enqueue kernels
 *     on the given stream, with every size and pointer fixed at the call; none
 *     of them synchronises or allocates. A sequence of them (one decode step)
 *     can therefore be captured on a non-default stream into a CUDA graph and
 *     replayed, on the same buffers, with stage timing off (gdnbeam_timing):
 *     a replay stores the same bits as the calls. The context's call-order
 *     checks run at capture, not at replay.
 */
#ifndef GDNBEAM_H_
#define GDNBEAM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdnbeam_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  GDNBEAM_OK = 0,
  GDNBEAM_EINVAL = -1,       /* null pointer, size out of range, bad index argument */
  GDNBEAM_EUNSUPPORTED = -2, /* shape or dtype this library does not handle */
  GDNBEAM_EWORKSPACE = -3,   /* workspace or scratch smaller than required */
  GDNBEAM_ESTATE = -4,       /* call out of order (step before prefill, t out of sequence) */
  GDNBEAM_ECUDA = -5,        /* a CUDA runtime/driver call or a launch failed */
  GDNBEAM_EDEVICE = -6,      /* the device error word was set */
  GDNBEAM_ENOMEM = -7        /* host allocation of the context failed */
};

enum { GDNBEAM_F32 = 0, GDNBEAM_BF16 = 1 };

/* Device error word bits (gdnbeam_device_status). */
enum {
  GDNBEAM_DERR_TOKEN = 1,     /* token id outside [0, V) */
  GDNBEAM_DERR_PARENT = 2,    /* parent index outside [0, W_{t-1}) */
  GDNBEAM_DERR_SLOT = 4,      /* ancestry slot outside its depth's beam count */
  GDNBEAM_DERR_NONFINITE = 8, /* a NaN or infinite logit, lse or cumulative score reached
                               * selection (when the logits stage's tile maxima are
                               * reused, a NaN or +inf logit shows through its row's
                               * lse; a -inf logit then scores -inf unflagged) */
  GDNBEAM_DERR_TIMEOUT = 16,  /* a bounded on-chip wait gave up */
  GDNBEAM_DERR_SELECT = 32    /* selection bookkeeping inconsistency */
};

#define GDNBEAM_MAX_T 8        /* longest SID (selections) supported */

/* Shape of one decode job. d_k in {16, 32, 64, 128, 256}, d_v in {16, 32, 64,
 * 128, 256, 512} (the state-path baselines: both at most 128); 1 <= T <= GDNBEAM_MAX_T;
 * V <= 16384; W_max <= 4096. residual = 0 requires layers = 1 and reads the
 * codebook logits off concat_h(o) (OneLA §1.2 eq. 3 output); residual = 1 runs
 * a residual stream with unit-gain RMSNorm (eps 1e-6) before each layer and
 * before the codebook head, which requires H*d_v == d_model. */
typedef struct gdnbeam_config {
  int R;        /* requests decoded together */
  int layers;   /* stacked GDN layers */
  int H;        /* (value) heads per layer */
  int d_k;      /* key / query width per head */
  int d_v;      /* value width per head */
  int d_model;  /* embedding width */
  int V;        /* codebook size (candidates per beam) */
  int T;        /* SID length = number of selections */
  int W_max;    /* largest beam count of any selection */
  int L_max;    /* longest prompt gdnbeam_prefill_state accepts */
  int dtype;    /* GDNBEAM_F32 or GDNBEAM_BF16 storage */
  int residual; /* 0: single layer; 1: residual stream + RMSNorm glue */
  int state_path; /* 0: shared context + records + projection replay (OneLA);
                     1: FullState baseline, one d_v x d_k state per beam copied
                        on reorder (OneLA §3 "Controlled FullState"): same
                        pipeline, only the state path swapped;
                     2: ReplaySSM baseline (OneLA §1, Fig. 2): no per-beam
                        state; every step rebuilds each beam's parent state
                        from the stored S_ctx by replaying its ancestors'
                        records, then applies the current token */
  int H_k;      /* query/key heads (0: H). H must be a multiple of H_k; value
                   head h reads key head h / (H / H_k), consecutive value
                   heads sharing one (grouped query attention, OneLA §4's
                   H_K != H_V geometries). q, k and the records' keys hold
                   H_k heads; v, gates, states, delta and o hold H. */
} gdnbeam_config;

/* Weights, storage type, row-major, owned by the caller and kept alive for
 * the life of the context.
 *   E       [V][d_model]                      token embedding
 *   W_proj  [layers][N_proj][d_model]         N_proj = 2*H_k*d_k + H*d_v + 2*H rows:
 *             H_k*d_k query rows, H_k*d_k key rows, H*d_v value rows, then the H
 *             decay-gate vectors w_alpha and the H write-gate vectors w_beta
 *   W_o     [V][F]                            codebook head; F = H*d_v (single
 *             layer) or d_model (residual) */
typedef struct gdnbeam_weights {
  const void* E;
  const void* W_proj;
  const void* W_o;
} gdnbeam_weights;

/* Optional fp32 copies of intermediate values before storage rounding, for
 * parity checks. Any member may be NULL. Shapes for a call on n = R*W_t rows:
 *   q, k [layers][n][H_k*d_k]; v, delta, o [layers][n][H*d_v];
 *   alpha, beta [layers][n][H]; logits [n][V]. */
typedef struct gdnbeam_dumps {
  float* q;
  float* k;
  float* v;
  float* alpha;
  float* beta;
  float* delta;
  float* o;
  float* logits;
} gdnbeam_dumps;

/* Memory accounting of a configuration (host only, no CUDA call). */
typedef struct gdnbeam_footprint {
  size_t sctx_bytes;          /* shared context states: R*layers*H*d_v*d_k fp32 */
  size_t record_elements;     /* elements of one transition record: 1 + d_v + d_k (OneLA §2.2 eq. 5) */
  size_t records_bytes;       /* all record slots: R*layers*H*(T-1)*W_max*(d_v + d_k) storage + alpha fp32 */
  size_t ancestry_bytes;      /* ancestry index and token paths (int32) */
  size_t fullstate_bytes;     /* one per-beam full state per beam: R*layers*H*W_max*d_v*d_k (storage) */
  size_t workspace_bytes;     /* everything gdnbeam_create needs */
} gdnbeam_footprint;

typedef struct gdnbeam_ctx gdnbeam_ctx;

/* ---------------------------------------------------------------------------
 * Context-level calls (the decode loop)
 * ------------------------------------------------------------------------- */

/* Validates cfg and fills *out (host). Returns GDNBEAM_EINVAL/EUNSUPPORTED on
 * a configuration this library rejects. */
int gdnbeam_footprint_of(const gdnbeam_config* cfg, gdnbeam_footprint* out);

/* Creates a context over a caller-allocated workspace of at least
 * footprint.workspace_bytes, 256-byte aligned. The host-side context struct is
 * the only thing the library allocates; weights and workspace stay owned by
 * the caller. *out is set on success, NULL otherwise. */
int gdnbeam_create(const gdnbeam_config* cfg, const gdnbeam_weights* w,
                   void* workspace, size_t workspace_bytes, gdnbeam_ctx** out);
void gdnbeam_destroy(gdnbeam_ctx* ctx);

/* Prefill (OneLA §1.1, §2.1): runs the GDN recurrence (eq. 3) from S = 0 over
 * every request's prompt, keeps S_ctx per (request, layer, head) in the
 * workspace and writes the root row's logits and log-normaliser.
 *   prompt      [R][L] int32 token ids, 1 <= L <= L_max
 *   root_logits [R][V] storage
 *   root_lse    [R] fp32, lse = log sum_v exp(z_v) */
int gdnbeam_prefill_state(gdnbeam_ctx* ctx, const int32_t* prompt, int L,
                          void* root_logits, float* root_lse, gdnbeam_stream_t stream);

/* One decode call t on W_t beams per request (OneLA §2.3-2.5):
 *   1. ancestry update (eq. 9) from parents (ignored at t = 0) and token paths;
 *   2. projections of the beams' tokens -> q, k, v, alpha, beta; k and alpha
 *      go straight into the depth-t record slot;
 *   3. fused replay: u_q, u_k from S_ctx, folded along the ancestors' records
 *      (eqs. 6-7), then delta_t and o_t (eq. 8); delta_t fills the record;
 *   4. codebook logits and their log-normaliser.
 *   parents [R][W_t] int32 rows of the previous call (t >= 1)
 *   tokens  [R][W_t] int32 token ids chosen by the selection that made the beams
 *   logits  [R*W_t][V] storage (out);  lse [R*W_t] fp32 (out)
 *   dumps   optional (host struct of device pointers), may be NULL
 * Calls must come in order t = 0, 1, ..., T-2 after a prefill; t = 0 may be
 * issued again at any time to restart decoding from the same prefill. */
int gdnbeam_step(gdnbeam_ctx* ctx, int t, int W_t, const int32_t* parents,
                 const int32_t* tokens, void* logits, float* lse,
                 const gdnbeam_dumps* dumps, gdnbeam_stream_t stream);

/* Global top-W_next over the W_t x V candidates of every request (OneLA §1.1;
 * RecoGEM §4.3 exact selection: the result is the exact top-W_next, whatever
 * path computes it). Score of candidate (b, v):
 *   s = fl32(cum'_b + fl32(z_bv - lse_b)),  cum'_b = fl32(cum_b + bias_b)
 * in IEEE fp32 without contraction; order by s descending, then flat index
 * b*V + v ascending. t = -1 selects from the prefill row (W_t must be 1).
 *   logits [R*W_t][V] storage; lse [R*W_t]; cum [R*W_t] or NULL (= 0);
 *   bias [R*W_t] or NULL; outputs parents, tokens [R][W_next] int32 and
 *   cum_next [R][W_next] fp32, in selection order.
 * Requires W_next <= min(W_max, W_t*V). */
int gdnbeam_select(gdnbeam_ctx* ctx, int t, int W_t, int W_next, const void* logits,
                   const float* lse, const float* cum, const float* bias,
                   int32_t* parents, int32_t* tokens, float* cum_next,
                   gdnbeam_stream_t stream);

/* Final SID paths after the last selection: sid [R][W_final][T] int32. */
int gdnbeam_get_paths(gdnbeam_ctx* ctx, int W_final, const int32_t* parents,
                      const int32_t* tokens, int32_t* sid, gdnbeam_stream_t stream);

/* Copies S_ctx, fp32 [R][layers][H][d_v][d_k], into out. S_ctx is kept in
 * fp32 for every storage type: one copy per (request, layer, head) is shared
 * by all beams, so its width is amortised over the beam width. */
int gdnbeam_read_sctx(gdnbeam_ctx* ctx, float* out, gdnbeam_stream_t stream);

/* Releases requests' contexts (OneLA §2.1: S_ctx is the one persistent state
 * of a request; §2.4: records stay in their slots until the request ends,
 * nothing moves). request_mask (host) is [R] int32: requests with a non-zero
 * entry are released; NULL releases every request. Decoding restarts at
 * t = 0 and gdnbeam_step returns GDNBEAM_ESTATE until every request holds a
 * context again: gdnbeam_prefill_state (all requests) or
 * gdnbeam_prefill_requests (some). Requests not released keep their S_ctx
 * and the root rows the caller holds for them. Host only; no CUDA call. */
int gdnbeam_reset(gdnbeam_ctx* ctx, const int32_t* request_mask);

/* Prefill of some requests only (OneLA §1.1, §2.1), the others keeping their
 * S_ctx: for i < count, request request_ids[i] (host array, distinct ids in
 * [0, R)) gets the context of prompt row i.
 *   prompts     [count][L] int32 token ids, 1 <= L <= L_max
 *   root_logits [R][V] storage and root_lse [R] fp32: only the listed
 *               requests' rows are written.
 * The listed requests then hold a context again (see gdnbeam_reset); their
 * S_ctx and root rows equal those a full gdnbeam_prefill_state with the same
 * prompt rows would give. Each request runs as its own pass through the same
 * kernels, in order on the stream. Errors as gdnbeam_prefill_state;
 * GDNBEAM_EINVAL for an id out of range or listed twice (nothing launched). */
int gdnbeam_prefill_requests(gdnbeam_ctx* ctx, const int32_t* request_ids, int count,
                             const int32_t* prompts, int L, void* root_logits, float* root_lse,
                             gdnbeam_stream_t stream);

/* Synchronises the stream, then returns GDNBEAM_EDEVICE if the device error
 * word is set (and clears it), GDNBEAM_ECUDA on a CUDA error, else 0. */
int gdnbeam_status(gdnbeam_ctx* ctx, gdnbeam_stream_t stream);

/* Reads and optionally clears the device error word of the current device
 * (synchronous). Returns a GDNBEAM_DERR_* bit set, or a negative status. */
int gdnbeam_device_status(int clear);

/* Name of the kernel variant the context uses for each stage
 * ("tc" = tcgen05 tensor cores, "simt" = CUDA cores), as a static string such
 * as "proj=tc replay=tc logits=tc select=bound". */
const char* gdnbeam_variant(const gdnbeam_ctx* ctx);

const char* gdnbeam_strerror(int status);

/* Stages a context times when timing is on (gdnbeam_stage_times). */
enum {
  GDNBEAM_STAGE_ANCESTRY = 0, /* eq. 9 update and token paths */
  GDNBEAM_STAGE_EMBED = 1,    /* embedding gather, RMSNorm glue */
  GDNBEAM_STAGE_PROJECT = 2,  /* q, k, v, alpha, beta projections */
  GDNBEAM_STAGE_REPLAY = 3,   /* fused shared-context replay */
  GDNBEAM_STAGE_LOGITS = 4,   /* codebook logits and log-normaliser */
  GDNBEAM_STAGE_SELECT = 5,   /* exact global top-W selection */
  GDNBEAM_STAGE_PREFILL = 6,  /* prefill recurrence */
  GDNBEAM_NSTAGES = 7
};

/* Turns per-stage timing on or off (host). While on, every stage the
 * context launches is bracketed by two CUDA events on its stream; nothing
 * else changes. Turning it on clears earlier records. */
int gdnbeam_timing(gdnbeam_ctx* ctx, int enable);

/* Synchronises the recorded events and writes, per stage, the summed
 * milliseconds (ms[GDNBEAM_NSTAGES]) and the number of timed launches
 * (count[GDNBEAM_NSTAGES], may be NULL); then clears the records. */
int gdnbeam_stage_times(gdnbeam_ctx* ctx, float* ms, int* count);

/* Kernel launches this library has issued in this process (all contexts and
 * tensor-level calls); clear != 0 resets the counter after reading. */
long long gdnbeam_launches(int clear);

/* ---------------------------------------------------------------------------
 * Tensor-level calls: each stage on explicit buffers (same kernels the
 * context runs). cfg gives dims and dtype; only the fields named matter.
 * ------------------------------------------------------------------------- */

/* Projections for n rows of one layer (OneLA §1.2 eq. 3 inputs).
 *   u [n][d_model] storage, W_proj [N_proj][d_model] storage (one layer);
 *   q [n][H_k*d_k], k [n][H_k*d_k], v [n][H*d_v] storage; alpha, beta [n][H] fp32.
 *   q and k are L2-normalised per head (eps 1e-6 inside the root);
 *   alpha = exp(-softplus(w_alpha.u)), beta = sigmoid(w_beta.u).
 * scratch: device buffer of gdnbeam_project_scratch_bytes(cfg, n) bytes
 * (0 for the tensor-core path; may then be NULL). dumps: optional fp32 copies
 * (layer 0 slots of gdnbeam_dumps). */
size_t gdnbeam_project_scratch_bytes(const gdnbeam_config* cfg, int n);
int gdnbeam_project(const gdnbeam_config* cfg, int n, const void* u, const void* W_proj,
                    void* q, void* k, void* v, float* alpha, float* beta,
                    void* scratch, size_t scratch_bytes, const gdnbeam_dumps* dumps,
                    gdnbeam_stream_t stream);

/* Records of one depth (OneLA §2.2 eq. 5), rows packed [R][W_j][H]. */
typedef struct gdnbeam_records {
  const void* k;       /* [R*W_j][H_k*d_k] storage */
  const void* delta;   /* [R*W_j][H*d_v] storage */
  const float* alpha;  /* [R*W_j][H] */
  int W_j;             /* beams per request at that depth */
} gdnbeam_records;

/* Fused shared-context replay for one layer at decode call t (OneLA §2.3
 * eqs. 6-8, §2.5): for every request r, beam b < W_t and head h,
 *   u_q = S_ctx q_b, u_k = S_ctx k_b, folded over j < t with the record at
 *   slot anc[r*W_t+b][j] of depth j; delta = beta (v - alpha u_k);
 *   o = alpha u_q + delta (k_b . q_b).
 *   sctx [R][H][d_v][d_k] fp32 (stride between requests: sctx_rstride elements)
 *   q, k [R*W_t][H_k*d_k], v [R*W_t][H*d_v] storage; alpha, beta [R*W_t][H]
 *   depth: host array of t record descriptors; anc [R*W_t][anc_stride] int32
 *   delta_out, o_out [R*W_t][H*d_v] storage; x_inout optional fp32
 *   [R*W_t][H*d_v] residual stream to which o is added (NULL: none).
 *   dumps: optional fp32 delta / o (layer 0 slots). */
int gdnbeam_replay(const gdnbeam_config* cfg, int t, int W_t, const float* sctx,
                   long long sctx_rstride, const void* q, const void* k, const void* v,
                   const float* alpha, const float* beta, const gdnbeam_records* depth,
                   const int32_t* anc, int anc_stride, void* delta_out, void* o_out,
                   float* x_inout, const gdnbeam_dumps* dumps, gdnbeam_stream_t stream);

/* The pages' two baselines of the same step, for one layer (gdnbeam_step runs
 * them inside the decode loop when state_path is 1 or 2). Head widths d_k, d_v
 * at most 128; storage-precision states; outputs as gdnbeam_replay.
 *
 * FullState (OneLA §3, the "Controlled FullState" path): every beam keeps its
 * own d_v x d_k state. For request r, beam b < W_t and head h, the parent
 * state S_par is sctx_store's head h of request r at t = 0, else
 * states_prev[r*W_prev + parents[r*W_t+b]]; then (eq. 3)
 *   delta = beta (v - alpha S_par k), S = alpha S_par + delta k^T, o = S q,
 * and S is stored to states_cur[r*W_t+b].
 *   sctx_store [R][H][d_v][d_k] storage, sctx_rstride elements between requests
 *   states_prev [R*W_prev][H][d_v][d_k], states_cur [R*W_t][H][d_v][d_k] storage
 *   parents [R*W_t] int32 (read when t > 0; out-of-range entries set
 *   GDNBEAM_DERR_PARENT). Returns GDNBEAM_EUNSUPPORTED for wider heads. */
int gdnbeam_fullstate_step(const gdnbeam_config* cfg, int t, int W_t, int W_prev,
                           const void* sctx_store, long long sctx_rstride,
                           const void* states_prev, void* states_cur, const int32_t* parents,
                           const void* q, const void* k, const void* v, const float* alpha,
                           const float* beta, void* delta_out, void* o_out,
                           gdnbeam_stream_t stream);

/* ReplaySSM (OneLA §1.3 and §7.2, the baseline that recomputes instead of
 * storing): no per-beam state is kept. Each (beam, head) rebuilds its parent
 * state from the request's S_ctx (sctx_store, storage precision) by applying
 * its t ancestors' records in depth order (eq. 4), then takes the step as
 * FullState does. Records, anc and the other arguments as gdnbeam_replay.
 * Returns GDNBEAM_EUNSUPPORTED for wider heads. */
int gdnbeam_replayssm_step(const gdnbeam_config* cfg, int t, int W_t, const void* sctx_store,
                           long long sctx_rstride, const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, const gdnbeam_records* depth,
                           const int32_t* anc, int anc_stride, void* delta_out, void* o_out,
                           gdnbeam_stream_t stream);

/* Codebook logits for n rows: z = W_o feat, lse = log sum exp z.
 *   feat [n][F] storage; W_o [V][F]; z [n][V] storage; lse [n] fp32. */
size_t gdnbeam_logits_scratch_bytes(const gdnbeam_config* cfg, int n);
int gdnbeam_logits(const gdnbeam_config* cfg, int n, const void* feat, const void* W_o,
                   void* z, float* lse, void* scratch, size_t scratch_bytes,
                   const gdnbeam_dumps* dumps, gdnbeam_stream_t stream);

/* Exact global top-W_next per request, as gdnbeam_select, on explicit
 * scratch of gdnbeam_select_scratch_bytes(R, W_t, W_next, V) bytes. */
size_t gdnbeam_select_scratch_bytes(int R, int W_t, int W_next, int V);
int gdnbeam_select_topw(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                        const float* lse, const float* cum, const float* bias,
                        int32_t* parents, int32_t* tokens, float* cum_next,
                        void* scratch, size_t scratch_bytes, gdnbeam_stream_t stream);

/* The same selection as gdnbeam_select_topw for callers that cannot allocate
 * device memory: a plugin that its host framework calls with only its input
 * and output tensors, or a process whose device memory another allocator has
 * fully reserved, has no way to pass the scratch buffer that call needs. This
 * variant takes no scratch and allocates nothing; it uses a fixed area of
 * gdnbeam_select_noalloc_max_bytes() bytes (16 MiB) that the library keeps on
 * every device where it is loaded, until the process exits. (The pages have no
 * counterpart: this is a deployment convenience, not part of the method.)
 *   - Selections whose scratch (gdnbeam_select_scratch_bytes) exceeds that
 *     size are refused with GDNBEAM_EWORKSPACE before anything is launched.
 *   - The first call on each device looks up the area's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the one area, and its contents persist between calls;
 *     every call writes each request's state in the area before reading it
 *     (a leftover value can cost time, never change a result). Calls whose
 *     work overlaps on the GPU (other streams, other host threads) race on
 *     the area: order them on one stream or synchronise between them.
 * Arguments, outputs and errors are those of gdnbeam_select_topw. */
size_t gdnbeam_select_noalloc_max_bytes(void);
int gdnbeam_select_topw_noalloc(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                                const float* lse, const float* cum, const float* bias,
                                int32_t* parents, int32_t* tokens, float* cum_next,
                                gdnbeam_stream_t stream);

/* Ancestry-index update of OneLA §2.4 eq. 9 for decode call t:
 *   anc_out[r*W_t+b][j] = anc_prev[r*W_prev+p][j] (j < t-1), anc_out[..][t-1] = p,
 *   with p = parents[r*W_t+b]; sid_out[..][s] = sid_prev[..p..][s] (s < t),
 *   sid_out[..][t] = tokens[r*W_t+b]. Row stride of anc and sid is T ints.
 *   At t = 0 anc is untouched and sid_out[..][0] = tokens. */
int gdnbeam_ancestry(int R, int t, int T, int V, int W_prev, int W_t, const int32_t* parents,
                     const int32_t* tokens, const int32_t* anc_prev, const int32_t* sid_prev,
                     int32_t* anc_out, int32_t* sid_out, gdnbeam_stream_t stream);

/* Prefill recurrence over L tokens for every (request, head) from S = 0
 * (OneLA §1.2 eq. 3).
 *   q, k [R*L][H_k*d_k], v [R*L][H*d_v] storage; alpha, beta [R*L][H] fp32;
 *   sctx_out [R][H][d_v][d_k] fp32 (request stride sctx_rstride elements);
 *   o_last [R][H*d_v] storage output at the last position (or NULL);
 *   x_inout optional fp32 [R*L][H*d_v]: o of every position is added to it.
 * bf16 storage with d_k = d_v = 128 runs the chunked tensor-core form (OneLA
 * §2.1 prefill, 64-token chunks); with x_inout it also needs scratch of
 * gdnbeam_prefill_scan_scratch_bytes(cfg, L, 1) bytes (every chunk's start
 * state and every token's record, fp32), else GDNBEAM_EWORKSPACE. Other
 * shapes run the recurrence on CUDA cores and need no scratch (may be NULL). */
size_t gdnbeam_prefill_scan_scratch_bytes(const gdnbeam_config* cfg, int L, int with_residual);
int gdnbeam_prefill_scan(const gdnbeam_config* cfg, int L, const void* q, const void* k,
                         const void* v, const float* alpha, const float* beta,
                         float* sctx_out, long long sctx_rstride, void* o_last,
                         float* x_inout, void* scratch, size_t scratch_bytes,
                         gdnbeam_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNBEAM_H_ */
