// FullState baseline: one d_v x d_k state per beam, copied on reorder.
//
// The "Controlled FullState" path of OneLA §3: the same decode pipeline with
// only the state path swapped. Every beam of decode call t reads its parent's
// full state (S_ctx at t = 0), applies the GDN recurrence of OneLA §1.2 eq. 3
// and writes its own state into the next buffer, indexed by the new beam
// order. It moves 2 * H * d_v * d_k storage elements per beam-step, which is
// what the shared-context replay avoids.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

// One block per (beam row, head); thread i owns state row i (DK values in
// registers).
template <typename T, int DK>
__global__ void __launch_bounds__(128) fullstate_step_kernel(FullStateArgs a) {
  const int row = blockIdx.x;  // r * W_t + b
  const int h = blockIdx.y;
  const int r = row / a.W_t;
  const int i = threadIdx.x;
  const int H = a.H, dv = a.d_v;
  __shared__ float kq[2][DK];
  const T* q = (const T*)a.q + ((size_t)row * H + h) * DK;
  const T* k = (const T*)a.k + ((size_t)row * H + h) * DK;
  for (int c = threadIdx.x; c < DK; c += blockDim.x) {
    kq[0][c] = ldf(k + c);
    kq[1][c] = ldf(q + c);
  }
  __syncthreads();
  if (i >= dv) return;
  float S[DK];
  if (a.t == 0) {
    const float* src = a.sctx + (size_t)r * a.sctx_rstride + ((size_t)h * dv + i) * DK;
#pragma unroll
    for (int c = 0; c < DK; ++c) S[c] = src[c];
  } else {
    int par = a.parents[row];
    if (par < 0 || par >= a.W_prev) {
      if (i == 0) raise_error(a.err, GDNBEAM_DERR_PARENT);
      par = 0;
    }
    const T* src = (const T*)a.states_prev +
                   ((((size_t)r * a.W_prev + par) * a.layers + a.layer) * H + h) * (size_t)dv * DK +
                   (size_t)i * DK;
#pragma unroll
    for (int c = 0; c < DK; ++c) S[c] = ldf(src + c);
  }
  const size_t gi = ((size_t)row * H + h) * dv + i;
  const float al = a.alpha[(size_t)row * H + h], be = a.beta[(size_t)row * H + h];
  float p = 0.f;
#pragma unroll
  for (int c = 0; c < DK; ++c) p = fmaf(S[c], kq[0][c], p);
  const float delta = be * (ldf((const T*)a.v + gi) - al * p);
  float o = 0.f;
  T* dst = (T*)a.states_cur + ((((size_t)row * a.layers + a.layer) * H + h) * (size_t)dv + i) * DK;
#pragma unroll
  for (int c = 0; c < DK; ++c) {
    const float sn = fmaf(al, S[c], delta * kq[0][c]);
    dst[c] = St<T>::from_f(sn);
    o = fmaf(sn, kq[1][c], o);
  }
  stf((T*)a.delta_out + gi, delta);
  stf((T*)a.o_out + gi, o);
  if (a.delta_dump) a.delta_dump[gi] = delta;
  if (a.o_dump) a.o_dump[gi] = o;
  if (a.x_inout) a.x_inout[gi] += o;
}

template <typename T>
int dispatch(const FullStateArgs& a, cudaStream_t s) {
  dim3 grid(a.R * a.W_t, a.H);
  switch (a.d_k) {
    case 16: fullstate_step_kernel<T, 16><<<grid, 128, 0, s>>>(a); break;
    case 32: fullstate_step_kernel<T, 32><<<grid, 128, 0, s>>>(a); break;
    case 64: fullstate_step_kernel<T, 64><<<grid, 128, 0, s>>>(a); break;
    case 128: fullstate_step_kernel<T, 128><<<grid, 128, 0, s>>>(a); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

int launch_fullstate(int dtype, const FullStateArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.d_v > 128 || a.R * a.W_t > 0x7FFFFFFF) return GDNBEAM_EUNSUPPORTED;
  return dtype == GDNBEAM_BF16 ? dispatch<__nv_bfloat16>(a, s) : dispatch<float>(a, s);
}

}  // namespace gdnbeam
