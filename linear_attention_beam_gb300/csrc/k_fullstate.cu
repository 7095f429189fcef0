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
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

// One block per (beam row, head). The parent's d_v x d_k state (one
// contiguous block) arrives in shared memory by a single bulk copy; thread i
// applies eq. 3 to row i in place, visiting its 16-byte chunks in an order
// rotated by i so the threads of a warp hit different banks; the child state
// leaves by a single bulk copy.
template <typename T, int DK>
__global__ void __launch_bounds__(128) fullstate_step_kernel(FullStateArgs a) {
  extern __shared__ __align__(128) uint8_t tile[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  __shared__ float kq[2][DK];
  constexpr int EPC = 16 / (int)sizeof(T);     // elements per 16-byte chunk
  constexpr int CPR = DK / EPC;                 // chunks per row
  const int row = blockIdx.x;  // r * W_t + b
  const int h = blockIdx.y;
  const int r = row / a.W_t;
  const int i = threadIdx.x;
  const int H = a.H, dv = a.d_v;
  const uint32_t bytes = (uint32_t)(dv * DK * sizeof(T));
  const uint32_t sbar = tc::smem_u32(&bar), stile = tc::smem_u32(tile);
  if (i == 0) {
    tc::mbar_init(sbar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  const T* q = (const T*)a.q + ((size_t)row * H + h) * DK;
  const T* k = (const T*)a.k + ((size_t)row * H + h) * DK;
  for (int c = threadIdx.x; c < DK; c += blockDim.x) {
    kq[0][c] = ldf(k + c);
    kq[1][c] = ldf(q + c);
  }
  __syncthreads();
  if (i == 0) {
    // the parent's state, or the shared context state at the first decode call
    const T* src;
    if (a.t > 0) {
      int par = a.parents[row];
      if (par < 0 || par >= a.W_prev) {
        raise_error(a.err, GDNBEAM_DERR_PARENT);
        par = 0;
      }
      src = (const T*)a.states_prev +
            ((((size_t)r * a.W_prev + par) * a.layers + a.layer) * H + h) * (size_t)dv * DK;
    } else {
      src = (const T*)a.sctx_store + (size_t)r * a.sctx_rstride + (size_t)h * dv * DK;
    }
    tc::mbar_arrive_expect_tx(sbar, bytes);
    tc::bulk_load(stile, src, bytes, sbar);
  }
  const bool ok = tc::mbar_wait(sbar, 0, &s_abort, a.err);
  if (ok && i < dv) {
    T* rowp = reinterpret_cast<T*>(tile) + (size_t)i * DK;
    auto chunk_in = [&](int ch, float (&x)[EPC]) {
      const uint4 raw = *reinterpret_cast<const uint4*>(rowp + ch * EPC);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int j = 0; j < EPC; ++j) x[j] = St<T>::to_f(e[j]);
    };
    const size_t gi = ((size_t)row * H + h) * dv + i;
    const float al = a.alpha[(size_t)row * H + h], be = a.beta[(size_t)row * H + h];
    float p = 0.f;
#pragma unroll 4
    for (int c = 0; c < CPR; ++c) {
      const int ch = (c + i) % CPR;
      float x[EPC];
      chunk_in(ch, x);
#pragma unroll
      for (int j = 0; j < EPC; ++j) p = fmaf(x[j], kq[0][ch * EPC + j], p);
    }
    const float delta = be * (ldf((const T*)a.v + gi) - al * p);
    float o = 0.f;
#pragma unroll 4
    for (int c = 0; c < CPR; ++c) {
      const int ch = (c + i) % CPR;
      float x[EPC];
      chunk_in(ch, x);
      uint4 out;
      T* oe = reinterpret_cast<T*>(&out);
#pragma unroll
      for (int j = 0; j < EPC; ++j) {
        const float sn = fmaf(al, x[j], delta * kq[0][ch * EPC + j]);
        oe[j] = St<T>::from_f(sn);
        o = fmaf(sn, kq[1][ch * EPC + j], o);
      }
      *reinterpret_cast<uint4*>(rowp + ch * EPC) = out;  // each thread rewrites its own row
    }
    stf((T*)a.delta_out + gi, delta);
    stf((T*)a.o_out + gi, o);
    if (a.delta_dump) a.delta_dump[gi] = delta;
    if (a.o_dump) a.o_dump[gi] = o;
    if (a.x_inout) a.x_inout[gi] += o;
  }
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (i == 0 && ok) {
    T* dst = (T*)a.states_cur + (((size_t)row * a.layers + a.layer) * H + h) * (size_t)dv * DK;
    tc::bulk_store(dst, stile, bytes);
    tc::bulk_commit();
    tc::bulk_wait_read<0>();  // the tile is read out before the block exits
  }
}

template <typename T, int DK>
int launch_dk(const FullStateArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)a.d_v * DK * sizeof(T);
  GDN_CUDA(cudaFuncSetAttribute(fullstate_step_kernel<T, DK>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  fullstate_step_kernel<T, DK><<<dim3(a.R * a.W_t, a.H), 128, smem, s>>>(a);
  return GDNBEAM_OK;
}

template <typename T>
int dispatch(const FullStateArgs& a, cudaStream_t s) {
  int st;
  switch (a.d_k) {
    case 16: st = launch_dk<T, 16>(a, s); break;
    case 32: st = launch_dk<T, 32>(a, s); break;
    case 64: st = launch_dk<T, 64>(a, s); break;
    case 128: st = launch_dk<T, 128>(a, s); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
  if (st) return st;
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

template <typename T>
__global__ void to_storage_kernel(size_t n, const float* __restrict__ src, T* __restrict__ dst) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = St<T>::from_f(src[i]);
}

int launch_to_storage(int dtype, size_t n, const float* src, void* dst, cudaStream_t s) {
  if (n == 0) return GDNBEAM_OK;
  const unsigned blocks = (unsigned)((n + 255) / 256 < 65536 ? (n + 255) / 256 : 65536);
  if (dtype == GDNBEAM_BF16)
    to_storage_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(n, src, (__nv_bfloat16*)dst);
  else
    to_storage_kernel<float><<<blocks, 256, 0, s>>>(n, src, (float*)dst);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

int launch_fullstate(int dtype, const FullStateArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.d_v > 128 || a.R * a.W_t > 0x7FFFFFFF) return GDNBEAM_EUNSUPPORTED;
  return dtype == GDNBEAM_BF16 ? dispatch<__nv_bfloat16>(a, s) : dispatch<float>(a, s);
}

}  // namespace gdnbeam
