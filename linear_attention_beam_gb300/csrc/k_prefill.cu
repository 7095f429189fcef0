// Prefill recurrence: compresses each request's prompt into S_ctx.
//
// OneLA §1.1/§2.1: the shared prompt is folded into one recurrent state per
// (request, layer, head), shared by every beam. The recurrence is eq. 3 of
// §1.2 run from S = 0. One block per (request, head); thread i keeps row i
// of S (d_k fp32 values) in registers, and the next token's k, q, v and gates
// are prefetched into registers while the current token is applied.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

template <typename T, int DK>
__global__ void __launch_bounds__(128) prefill_scan_kernel(
    int L, int H, int dv, const T* __restrict__ q, const T* __restrict__ k,
    const T* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    float* __restrict__ sctx, long long rstride, T* __restrict__ o_last, float* __restrict__ x) {
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  const int i = threadIdx.x;
  __shared__ float kb[2][DK], qb[2][DK], gb[2][2];
  float S[DK];
#pragma unroll
  for (int c = 0; c < DK; ++c) S[c] = 0.0f;

  const size_t row0 = (size_t)r * L;
  auto fetch = [&](int pos, float& kr, float& qr, float& vr, float& ar, float& br) {
    size_t row = row0 + pos;
    if (i < DK) {
      kr = ldf(k + (row * H + h) * DK + i);
      qr = ldf(q + (row * H + h) * DK + i);
    }
    if (i < dv) vr = ldf(v + (row * H + h) * dv + i);
    if (i == 0) { ar = alpha[row * H + h]; br = beta[row * H + h]; }
  };
  float kr = 0.f, qr = 0.f, vr = 0.f, ar = 0.f, br = 0.f;
  fetch(0, kr, qr, vr, ar, br);
  if (i < DK) { kb[0][i] = kr; qb[0][i] = qr; }
  if (i == 0) { gb[0][0] = ar; gb[0][1] = br; }
  float v_cur = vr;
  __syncthreads();

  for (int pos = 0; pos < L; ++pos) {
    const int buf = pos & 1;
    float kn = 0.f, qn = 0.f, vn = 0.f, an = 0.f, bn = 0.f;
    if (pos + 1 < L) fetch(pos + 1, kn, qn, vn, an, bn);
    if (i < dv) {
      const float a = gb[buf][0], b = gb[buf][1];
      float p = 0.0f;
#pragma unroll
      for (int c = 0; c < DK; ++c) p = fmaf(S[c], kb[buf][c], p);
      const float delta = b * (v_cur - a * p);
      float o = 0.0f;
#pragma unroll
      for (int c = 0; c < DK; ++c) {
        S[c] = fmaf(a, S[c], delta * kb[buf][c]);
        o = fmaf(S[c], qb[buf][c], o);
      }
      size_t row = row0 + pos;
      if (x) x[(row * H + h) * dv + i] += o;
      if (o_last && pos == L - 1) stf(o_last + ((size_t)r * H + h) * dv + i, o);
    }
    if (pos + 1 < L) {
      if (i < DK) { kb[buf ^ 1][i] = kn; qb[buf ^ 1][i] = qn; }
      if (i == 0) { gb[buf ^ 1][0] = an; gb[buf ^ 1][1] = bn; }
      v_cur = vn;
    }
    __syncthreads();
  }
  if (i < dv) {
    float* out = sctx + (size_t)r * rstride + ((size_t)h * dv + i) * DK;
#pragma unroll
    for (int c = 0; c < DK; ++c) out[c] = S[c];
  }
}

template <typename T>
int dispatch_dk(const gdnbeam_config& c, int L, const void* q, const void* k, const void* v,
                const float* alpha, const float* beta, float* sctx, long long rs, void* o_last,
                float* x, cudaStream_t s) {
  dim3 grid(c.R * c.H);
  const int threads = 128;
#define GDN_SCAN(DK)                                                                         \
  prefill_scan_kernel<T, DK><<<grid, threads, 0, s>>>(L, c.H, c.d_v, (const T*)q,           \
      (const T*)k, (const T*)v, alpha, beta, sctx, rs, (T*)o_last, x)
  switch (c.d_k) {
    case 16: GDN_SCAN(16); break;
    case 32: GDN_SCAN(32); break;
    case 64: GDN_SCAN(64); break;
    case 128: GDN_SCAN(128); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
#undef GDN_SCAN
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
