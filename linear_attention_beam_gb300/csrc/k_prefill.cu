// Prefill recurrence: compresses each request's prompt into S_ctx.
//
// OneLA §1.1/§2.1: the shared prompt is folded into one recurrent state per
// (request, layer, head), shared by every beam. The recurrence is eq. 3 of
// §1.2 run from S = 0. One block per (request, head); the rows of S (d_k
// fp32 values each) stay in registers, split over a few threads per row, and
// the next token's k, q, v and gates are prefetched while the current token
// is applied.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

// TPR threads share row i of S, each holding DK / TPR consecutive columns;
// a dot product is a few interleaved partial sums per thread and a
// butterfly over the TPR threads. Tokens are staged CH at a time in shared
// memory (as fp32), the next chunk's loads in flight while the current one
// is applied, so the per-token loop reads only shared memory and needs no
// block barrier.
template <typename T, int DK, int TPR, int CH>
__global__ void __launch_bounds__(128 * TPR) prefill_scan_kernel(
    int L, int H, int dv, const T* __restrict__ q, const T* __restrict__ k,
    const T* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    float* __restrict__ sctx, long long rstride, T* __restrict__ o_last, float* __restrict__ x) {
  constexpr int NC = DK / TPR;            // columns per thread
  constexpr int NA = NC < 4 ? NC : 4;     // partial sums per thread
  constexpr int EPV = 16 / (int)sizeof(T);  // elements per 16-byte load
  constexpr int NT = 128 * TPR;
  constexpr int KV = DK / EPV;            // 16-byte pieces per k or q row
  constexpr int PF = (CH * (2 * KV + 128 / EPV) + NT - 1) / NT;  // loads per thread per chunk
  // a k or q row keeps each thread's NC columns as one segment, segments 16
  // bytes apart in the bank cycle so the TPR threads of a row read without
  // bank conflicts
  constexpr int PAD = TPR > 1 ? 4 : 0;
  constexpr int RS = TPR * (NC + PAD);     // floats per staged k or q row
  extern __shared__ __align__(16) float sm[];
  float* ks = sm;                          // [2][CH][RS]
  float* qs = ks + 2 * CH * RS;            // [2][CH][RS]
  float* vs = qs + 2 * CH * RS;            // [2][CH][128]
  float2* gs = reinterpret_cast<float2*>(vs + 2 * CH * 128);  // [2][CH]
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x;
  const int i = tid / TPR, part = tid % TPR, c0 = part * NC;
  const int VV = dv / EPV;                 // 16-byte pieces per v row
  const int per_chunk = CH * (2 * KV + VV);
  float S[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) S[c] = 0.0f;
  const size_t row0 = (size_t)r * L;
  const int n_chunks = (L + CH - 1) / CH;

  // piece u of a chunk: k rows, then q rows, then v rows (16 bytes each)
  auto load = [&](int chunk, uint4 (&buf)[PF], float2& g) {
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int u = tid + e * NT;
      buf[e] = make_uint4(0u, 0u, 0u, 0u);
      if (u < per_chunk) {
        int t, piece;
        const T* base;
        int width;
        if (u < CH * KV) { t = u / KV; piece = u % KV; base = k; width = DK; }
        else if (u < 2 * CH * KV) { t = (u - CH * KV) / KV; piece = (u - CH * KV) % KV; base = q; width = DK; }
        else { t = (u - 2 * CH * KV) / VV; piece = (u - 2 * CH * KV) % VV; base = v; width = dv; }
        const int pos = chunk * CH + t;
        if (pos < L)
          buf[e] = __ldg(reinterpret_cast<const uint4*>(base + ((row0 + pos) * H + h) * width) + piece);
      }
    }
    g = make_float2(0.f, 0.f);
    if (tid < CH) {
      const int pos = chunk * CH + tid;
      if (pos < L) g = make_float2(alpha[(row0 + pos) * H + h], beta[(row0 + pos) * H + h]);
    }
  };
  auto col = [&](int c) { return (c / NC) * (NC + PAD) + c % NC; };  // position of column c
  auto stash = [&](int sb, const uint4 (&buf)[PF], const float2& g) {
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int u = tid + e * NT;
      if (u < per_chunk) {
        float* dst;
        if (u < CH * KV) dst = ks + (size_t)(sb * CH + u / KV) * RS + col((u % KV) * EPV);
        else if (u < 2 * CH * KV) dst = qs + (size_t)(sb * CH + (u - CH * KV) / KV) * RS + col(((u - CH * KV) % KV) * EPV);
        else dst = vs + (size_t)(sb * CH + (u - 2 * CH * KV) / VV) * 128 + ((u - 2 * CH * KV) % VV) * EPV;
        const T* el = reinterpret_cast<const T*>(&buf[e]);
#pragma unroll
        for (int x = 0; x < EPV; ++x) dst[x] = St<T>::to_f(el[x]);
      }
    }
    if (tid < CH) gs[sb * CH + tid] = g;
  };

  {
    uint4 buf[PF];
    float2 g;
    load(0, buf, g);
    stash(0, buf, g);
  }
  __syncthreads();
  const bool active = i < dv;
  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int sb = chunk & 1;
    uint4 nxt[PF];
    float2 gn;
    if (chunk + 1 < n_chunks) load(chunk + 1, nxt, gn);
    const int steps = min(CH, L - chunk * CH);
    for (int t = 0; t < steps; ++t) {
      const float* kr = ks + (size_t)(sb * CH + t) * RS + part * (NC + PAD);
      const float* qr = qs + (size_t)(sb * CH + t) * RS + part * (NC + PAD);
      const float2 g = gs[sb * CH + t];
      float pa[NA];
#pragma unroll
      for (int u = 0; u < NA; ++u) pa[u] = 0.0f;
#pragma unroll
      for (int c = 0; c < NC; ++c) pa[c % NA] = fmaf(S[c], kr[c], pa[c % NA]);
      float p = 0.0f;
#pragma unroll
      for (int u = 0; u < NA; ++u) p += pa[u];
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      const float delta = g.y * (vs[(size_t)(sb * CH + t) * 128 + (active ? i : 0)] - g.x * p);
      float oa[NA];
#pragma unroll
      for (int u = 0; u < NA; ++u) oa[u] = 0.0f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        S[c] = fmaf(g.x, S[c], delta * kr[c]);
        oa[c % NA] = fmaf(S[c], qr[c], oa[c % NA]);
      }
      float o = 0.0f;
#pragma unroll
      for (int u = 0; u < NA; ++u) o += oa[u];
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
      if (active && part == 0) {
        const int pos = chunk * CH + t;
        const size_t row = row0 + pos;
        if (x) x[(row * H + h) * dv + i] += o;
        if (o_last && pos == L - 1) stf(o_last + ((size_t)r * H + h) * dv + i, o);
      }
    }
    // buffer sb ^ 1 was last read in the previous chunk, before its barrier
    if (chunk + 1 < n_chunks) stash(sb ^ 1, nxt, gn);
    __syncthreads();
  }
  if (active) {
    float* out = sctx + (size_t)r * rstride + ((size_t)h * dv + i) * DK + c0;
#pragma unroll
    for (int c = 0; c < NC; ++c) out[c] = S[c];
  }
}

constexpr int kScanChunk = 32;

template <typename T, int DK, int TPR>
int launch_scan(const gdnbeam_config& c, int L, const void* q, const void* k, const void* v,
                const float* alpha, const float* beta, float* sctx, long long rs, void* o_last,
                float* x, cudaStream_t s) {
  constexpr int CH = kScanChunk;
  constexpr int PAD = TPR > 1 ? 4 : 0, RS = TPR * (DK / TPR + PAD);
  const size_t smem = (size_t)(2 * CH * RS * 2 + 2 * CH * 128) * sizeof(float) + 2 * CH * sizeof(float2);
  GDN_CUDA(cudaFuncSetAttribute(prefill_scan_kernel<T, DK, TPR, CH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  prefill_scan_kernel<T, DK, TPR, CH><<<c.R * c.H, 128 * TPR, smem, s>>>(
      L, c.H, c.d_v, (const T*)q, (const T*)k, (const T*)v, alpha, beta, sctx, rs, (T*)o_last, x);
  return GDNBEAM_OK;
}

template <typename T>
int dispatch_dk(const gdnbeam_config& c, int L, const void* q, const void* k, const void* v,
                const float* alpha, const float* beta, float* sctx, long long rs, void* o_last,
                float* x, cudaStream_t s) {
  const int epv = 16 / (int)sizeof(T);
  if (c.d_v % epv != 0 || ((uintptr_t)q & 15) || ((uintptr_t)k & 15) || ((uintptr_t)v & 15) ||
      (c.H * c.d_k) % epv != 0)
    return GDNBEAM_EUNSUPPORTED;
  int st;
  switch (c.d_k) {
    case 16: st = launch_scan<T, 16, 1>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 32: st = launch_scan<T, 32, 1>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 64: st = launch_scan<T, 64, 2>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 128: st = launch_scan<T, 128, 4>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
  if (st) return st;
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

int launch_prefill_scan(const gdnbeam_config& c, int L, const void* q, const void* k,
                        const void* v, const float* alpha, const float* beta, float* sctx,
                        long long rs, void* o_last, float* x, cudaStream_t s) {
  if (L <= 0) return GDNBEAM_EINVAL;
  if (c.d_v > 128) return GDNBEAM_EUNSUPPORTED;
  if (c.dtype == GDNBEAM_BF16)
    return dispatch_dk<__nv_bfloat16>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s);
  return dispatch_dk<float>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s);
}

}  // namespace gdnbeam
