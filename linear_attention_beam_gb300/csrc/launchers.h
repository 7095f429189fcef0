// Host-side launchers of the gdnbeam kernels (internal to the library).
// Each returns a GDNBEAM_* status; all take the device error word pointer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdnbeam.h"

namespace gdnbeam {

// ---- CUDA-core kernels (any supported shape, fp32 or bf16 storage) -------

// u[m] = E[tokens[m]] (storage copy); if x != NULL also x[m] = fp32(E[...]).
// Rows of E into a residual stream plus its first RMS norm, one pass:
// x[m] = E[tok[m]] as fp32, u[m] = x[m] / rms(x[m]) (unit gain, eps 1e-6).
// GDNBEAM_EINVAL (nothing launched) unless d is a multiple of 128 up to 2048
// and the rows are vector-aligned.
int launch_gather_norm_rows(int dtype, int n, int d, const int32_t* tokens, int V, const void* E,
                            float* x, void* u, unsigned* err, cudaStream_t s);
int launch_gather_rows(int dtype, int n, int d_model, const int32_t* tokens, int V,
                       const void* E, void* u, float* x, unsigned* err, cudaStream_t s);

// u[m] = x[m] / sqrt(mean(x[m]^2) + 1e-6), stored in the storage type.
// Rows are x + m*x_stride (fp32) and u + m*d (storage).
int launch_rmsnorm_rows(int dtype, int n, int d, const float* x, long long x_stride, void* u,
                        cudaStream_t s);

// C[M][N] (fp32, row stride ldc) = A[M][K] . B[N][K]^T, storage inputs.
int launch_simt_gemm_nt(int dtype, int M, int N, int K, const void* A, int lda,
                        const void* B, int ldb, float* C, int ldc, cudaStream_t s);

// Raw projections P[n][N_proj] (fp32) -> q, k, v (storage), alpha, beta.
int launch_proj_epilogue(const gdnbeam_config& c, int n, const float* P, void* q, void* k,
                         void* v, float* alpha, float* beta, const gdnbeam_dumps* d,
                         cudaStream_t s);

// Raw logits Z[n][V] (fp32) -> z (storage), lse, optional fp32 dump.
int launch_logits_rows(int dtype, int n, int V, const float* Z, void* z, float* lse,
                       float* z_dump, cudaStream_t s);

// ---- tcgen05 tensor-core GEMMs (bf16, d = 128, d_model % 64 == 0) --------

bool tc_gemm_supported(const gdnbeam_config& c);
// Projection columns to compute: all of them, all but the queries (a
// prefill that needs the query only at the last token), or only the queries.
enum { PROJ_ALL = 0, PROJ_NO_Q = 1, PROJ_Q_ONLY = 2 };
// ldu: elements between consecutive rows of u (0: d_model).
int launch_tc_project(const gdnbeam_config& c, int n, const void* u, const void* W_proj,
                      void* q, void* k, void* v, float* alpha, float* beta,
                      const gdnbeam_dumps* d, cudaStream_t s, int cols = PROJ_ALL,
                      long long ldu = 0);
size_t tc_logits_scratch_bytes(const gdnbeam_config& c, int n);
int launch_tc_logits(const gdnbeam_config& c, int n, const void* feat, const void* W_o,
                     void* z, float* lse, void* scratch, const gdnbeam_dumps* d,
                     cudaStream_t s);

// ---- replay, prefill, selection, ancestry ---------------------------------

// Number of SMs of the current device (cached per device).
int sm_count();

// Query/key heads of a configuration (value head h reads key head
// h / (H / key_heads)).
inline int key_heads(const gdnbeam_config& c) { return c.H_k > 0 ? c.H_k : c.H; }

struct ReplayArgs {
  int R, H, d_k, d_v, t, W_t;
  int Hk;             // key heads: q, k and the records' keys hold Hk heads
  const float* sctx;  // fp32 [R][H][d_v][d_k], request stride sctx_rstride
  long long sctx_rstride;
  const void *q, *k, *v;
  const float *alpha, *beta;
  gdnbeam_records depth[GDNBEAM_MAX_T];
  const int32_t* anc;
  int anc_stride;
  void *delta_out, *o_out;  // o_out may be null when x_inout takes o_t
  float* x_inout;
  float *delta_dump, *o_dump;
  unsigned* err;
};
int launch_replay(int dtype, const ReplayArgs& a, cudaStream_t s);
bool tc_replay_supported(int dtype, int d_k, int d_v);
int launch_tc_replay(const ReplayArgs& a, cudaStream_t s);

// FullState baseline step for one layer (one d_v x d_k state per beam).
struct FullStateArgs {
  int R, H, d_k, d_v, t, W_t, W_prev, layers, layer;
  int Hk;                      // key heads (q, k hold Hk heads)
  const void* sctx_store;      // storage copy of S_ctx [R][...] (the t = 0 parent)
  long long sctx_rstride;      // request stride of sctx_store, elements
  const void* states_prev;     // storage [R*W_prev][layers][H][d_v][d_k]
  void* states_cur;            // storage [R*W_t][layers][H][d_v][d_k]
  const int32_t* parents;      // [R*W_t] rows of the previous call (t >= 1)
  const void *q, *k, *v;
  const float *alpha, *beta;
  void *delta_out, *o_out;     // o_out may be null when x_inout takes o_t
  float* x_inout;
  float *delta_dump, *o_dump;
  unsigned* err;
};
int launch_fullstate(int dtype, const FullStateArgs& a, cudaStream_t s);

// ReplaySSM baseline step for one layer: every (beam, head) re-applies its
// ancestors' records to the request's stored S_ctx, then the current token.
struct ReplaySsmArgs {
  int R, H, d_k, d_v, t, W_t;
  int Hk;                      // key heads (q, k and the records' keys hold Hk heads)
  const void* sctx_store;      // storage copy of S_ctx [R][...] (request stride below)
  long long sctx_rstride;      // elements
  const void *q, *k, *v;
  const float *alpha, *beta;
  gdnbeam_records depth[GDNBEAM_MAX_T];
  const int32_t* anc;
  int anc_stride;
  void *delta_out, *o_out;     // o_out may be null when x_inout takes o_t
  float* x_inout;
  float *delta_dump, *o_dump;
  unsigned* err;
};
int launch_replayssm(int dtype, const ReplaySsmArgs& a, cudaStream_t s);
// dst[i] = storage(src[i]) for n elements (S_ctx copy for the FullState path).
int launch_to_storage(int dtype, size_t n, const float* src, void* dst, cudaStream_t s);

// Chunked tensor-core prefill (bf16, d_k = d_v = 128): S_ctx and o at the
// last token, as launch_prefill_scan.
bool tc_prefill_supported(const gdnbeam_config& c);
// [R][L][width] bf16 rows as a 3-D TMA map, [64 columns][box_rows rows]
// boxes, 128-byte swizzled, rows past L read as zeros.
bool prefill_rows_map(CUtensorMap* map, const void* ptr, int R, int L, int width, int box_rows);
// The fp32 residual stream [R][L][width] as a 3-D TMA map with [128 columns]
// [64 rows] boxes, unswizzled, rows past L read as zeros.
bool prefill_stream_map(CUtensorMap* map, const float* x, int R, int L, int width);
// q_last: each request's query row at its last prompt token, q_last_ld
// elements apart. s0_out, delta_out (both or neither): every 64-token
// chunk's start state [R*H][2*ceil(L/128)][128][128] and every token's
// record [R*L][H*128], fp32, for launch_prefill_out_tc.
int launch_prefill_tc(const gdnbeam_config& c, int L, const void* q_last, long long q_last_ld,
                      const void* k, const void* v, const float* alpha, const float* beta,
                      float* sctx, long long rstride, void* o_last, cudaStream_t s,
                      float* s0_out = nullptr, float* delta_out = nullptr);
// Stacked layers: adds o of every prompt position to the residual stream x
// [R*L][H*128] from the chunk states and records launch_prefill_tc left in
// scratch (prefill_out_scratch_bytes: the records, then the chunk states).
size_t prefill_out_scratch_bytes(const gdnbeam_config& c, int L);
int launch_prefill_out_tc(const gdnbeam_config& c, int L, const void* q, const void* k,
                          const float* alpha, const float* s0, const float* delta, float* x,
                          cudaStream_t s);
// Prefill over L tokens of every request: the chunked tensor-core kernels
// when the shape allows (with a residual stream x_inout only when scratch
// holds prefill_out_scratch_bytes), else the recurrent CUDA-core scan.
int launch_prefill_scan(const gdnbeam_config& c, int L, const void* q, const void* k,
                        const void* v, const float* alpha, const float* beta, float* sctx,
                        long long sctx_rstride, void* o_last, float* x_inout, cudaStream_t s,
                        void* scratch = nullptr, size_t scratch_bytes = 0);

// Selection scratch and launch. hint (may be NULL): per (row, 256-code tile)
// the maximum logit in .x, as the logits stages leave it; NULL computes it.
size_t select_scratch_bytes(int R, int W_t, int W_next, int V);
int launch_select(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                  const float* lse, const float* cum, const float* bias, const float2* hint,
                  int32_t* parents, int32_t* tokens, float* cum_next, void* scratch,
                  unsigned* err, cudaStream_t s);
// Per (row, 256-code tile) maximum of stored logits into hint[row][tile].x.
int launch_tile_max(int dtype, int n, int V, const void* z, float2* hint, unsigned* err,
                    cudaStream_t s);
constexpr int kHintTile = 256;

// Device error word of the current device (defined with the C ABI).
unsigned* error_word();

int launch_ancestry(int R, int t, int T, int V, int W_prev, int W_t, const int32_t* parents,
                    const int32_t* tokens, const int32_t* anc_prev, const int32_t* sid_prev,
                    int32_t* anc_out, int32_t* sid_out, unsigned* err, cudaStream_t s);

}  // namespace gdnbeam
