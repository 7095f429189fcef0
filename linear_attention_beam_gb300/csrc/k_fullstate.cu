// State-path baselines: FullState (one d_v x d_k state per beam, copied on
// reorder) and ReplaySSM (no stored per-beam state; each step rebuilds the
// parent state from the shared S_ctx and the ancestors' records).
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

constexpr int kRsDepth = GDNBEAM_MAX_T - 2;  // ancestor records a ReplaySSM step replays

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
  const int hk = h / (H / a.Hk);  // the key head this value head reads
  const uint32_t bytes = (uint32_t)(dv * DK * sizeof(T));
  const uint32_t sbar = tc::smem_u32(&bar), stile = tc::smem_u32(tile);
  if (i == 0) {
    tc::mbar_init(sbar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  const T* q = (const T*)a.q + ((size_t)row * a.Hk + hk) * DK;
  const T* k = (const T*)a.k + ((size_t)row * a.Hk + hk) * DK;
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
    if (a.o_out) stf((T*)a.o_out + gi, o);
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

// ReplaySSM: one block per (beam row, head); thread i owns value row i. Each
// element of row i of the request's stored S_ctx is brought to the beam's
// parent state by replaying the t ancestor records, x <- alpha_j x +
// delta_j[i] k_j (OneLA §2.2 eqs. 4-5: the records regenerate the states
// they came from), in fp32 registers; a first pass forms S k_t, a second
// recomputes the row and applies eq. 3 for the current token. No state is
// ever written. bf16 rows are read straight into registers (TPR threads per
// row, 64 columns each, as packed words) and every thread walks its columns
// in the same order, so the key reads are broadcasts; fp32 rows go through a
// shared tile read in rotated order.
template <typename T, int DK, int TD>  // TD: replay depth t of this call
__global__ void __launch_bounds__(256, 2) replayssm_step_kernel(ReplaySsmArgs a) {
  extern __shared__ __align__(128) uint8_t tile[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  __shared__ __align__(16) float kq[2][DK];
  __shared__ __align__(16) float kjs[kRsDepth][DK];
  __shared__ float ajs[kRsDepth];
  constexpr bool kTile = sizeof(T) == 4;
  constexpr int TPR = kTile || DK < 128 ? 1 : DK / 64;  // threads per row (bf16 path)
  constexpr int NCOL = DK / TPR;                         // columns per thread
  constexpr int EPC = 16 / (int)sizeof(T);
  constexpr int CPR = DK / EPC;
  const int row = blockIdx.x;  // r * W_t + b
  const int h = blockIdx.y;
  const int r = row / a.W_t;
  const int tid = threadIdx.x;
  const int i = tid / TPR, part = tid % TPR, c0 = part * NCOL;
  const int H = a.H, dv = a.d_v;
  const int hk = h / (H / a.Hk);  // the key head this value head reads
  const T* srow_g = (const T*)a.sctx_store + (size_t)r * a.sctx_rstride + (size_t)h * dv * DK;
  const uint32_t sbar = tc::smem_u32(&bar), stile = tc::smem_u32(tile);
  if (kTile) {
    if (i == 0) {
      tc::mbar_init(sbar, 1);
      s_abort = 0;
      tc::fence_mbar_init();
    }
    __syncthreads();
    if (i == 0) {
      const uint32_t bytes = (uint32_t)(dv * DK * sizeof(T));
      tc::mbar_arrive_expect_tx(sbar, bytes);
      tc::bulk_load(stile, srow_g, bytes, sbar);
    }
  }
  // the beam's ancestor slots; a slot outside its depth skips that record
  int slot[TD > 0 ? TD : 1];
  bool use[TD > 0 ? TD : 1];
#pragma unroll
  for (int j = 0; j < TD; ++j) {
    const int sl = a.anc[(size_t)row * a.anc_stride + j];
    use[j] = sl >= 0 && sl < a.depth[j].W_j;
    if (!use[j] && tid == 0) raise_error(a.err, GDNBEAM_DERR_SLOT);
    slot[j] = use[j] ? sl : 0;
  }
  const T* q = (const T*)a.q + ((size_t)row * a.Hk + hk) * DK;
  const T* k = (const T*)a.k + ((size_t)row * a.Hk + hk) * DK;
  for (int c = tid; c < DK; c += blockDim.x) {
    kq[0][c] = ldf(k + c);
    kq[1][c] = ldf(q + c);
#pragma unroll
    for (int j = 0; j < TD; ++j)
        kjs[j][c] = use[j] ? ldf((const T*)a.depth[j].k +
                                 (((size_t)r * a.depth[j].W_j + slot[j]) * a.Hk + hk) * DK + c)
                           : 0.f;
  }
#pragma unroll
  for (int j = 0; j < TD; ++j)
    if (tid == j)
      ajs[j] = use[j] ? a.depth[j].alpha[((size_t)r * a.depth[j].W_j + slot[j]) * H + h] : 1.f;
  float dj[TD > 0 ? TD : 1];
#pragma unroll
  for (int j = 0; j < TD; ++j)
    dj[j] = (use[j] && i < dv)
                ? ldf((const T*)a.depth[j].delta + (((size_t)r * a.depth[j].W_j + slot[j]) * H + h) * dv + i)
                : 0.f;
  uint32_t srow[kTile ? 1 : NCOL / 2];
  if constexpr (!kTile) {
    if (i < dv) {
      const uint4* src = reinterpret_cast<const uint4*>(srow_g + (size_t)i * DK + c0);
#pragma unroll
      for (int c = 0; c < NCOL / 8; ++c) {
        const uint4 w = __ldg(src + c);
        srow[4 * c] = w.x; srow[4 * c + 1] = w.y; srow[4 * c + 2] = w.z; srow[4 * c + 3] = w.w;
      }
    }
  }
  __syncthreads();
  const bool ok = kTile ? tc::mbar_wait(sbar, 0, &s_abort, a.err) : true;
  const size_t gi = ((size_t)row * H + h) * dv + i;
  const bool active = ok && i < dv;
  if (!kTile || active) {
    const float al = a.alpha[(size_t)row * H + h], be = a.beta[(size_t)row * H + h];
    float p = 0.f, o = 0.f, delta = 0.f;
    if constexpr (!kTile) {
      // (the TPR threads of a row stay together for the shuffles below,
      // inactive rows computing on zeros)
      auto parent2 = [&](int c2, float& x0, float& x1) {
        x0 = __uint_as_float(srow[c2] << 16);
        x1 = __uint_as_float(srow[c2] & 0xFFFF0000u);
#pragma unroll
        for (int j = 0; j < TD; ++j) {
          const float2 kk = *reinterpret_cast<const float2*>(&kjs[j][c0 + 2 * c2]);
          x0 = fmaf(ajs[j], x0, dj[j] * kk.x);
          x1 = fmaf(ajs[j], x1, dj[j] * kk.y);
        }
      };
      if (!active) {
#pragma unroll
        for (int c2 = 0; c2 < NCOL / 2; ++c2) srow[c2] = 0u;
      }
      float pa = 0.f, pb = 0.f;
#pragma unroll
      for (int c2 = 0; c2 < NCOL / 2; ++c2) {
        float x0, x1;
        parent2(c2, x0, x1);
        pa = fmaf(x0, kq[0][c0 + 2 * c2], pa);
        pb = fmaf(x1, kq[0][c0 + 2 * c2 + 1], pb);
      }
      p = pa + pb;
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      delta = be * ((active ? ldf((const T*)a.v + gi) : 0.f) - al * p);
      float oa = 0.f, ob = 0.f;
#pragma unroll
      for (int c2 = 0; c2 < NCOL / 2; ++c2) {
        float x0, x1;
        parent2(c2, x0, x1);
        oa = fmaf(fmaf(al, x0, delta * kq[0][c0 + 2 * c2]), kq[1][c0 + 2 * c2], oa);
        ob = fmaf(fmaf(al, x1, delta * kq[0][c0 + 2 * c2 + 1]), kq[1][c0 + 2 * c2 + 1], ob);
      }
      o = oa + ob;
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
    } else {
      const T* rowp = reinterpret_cast<const T*>(tile) + (size_t)i * DK;
      auto parent = [&](int ch, float (&x)[EPC]) {
        const uint4 raw = *reinterpret_cast<const uint4*>(rowp + ch * EPC);
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int u = 0; u < EPC; ++u) {
          float xv = St<T>::to_f(e[u]);
#pragma unroll
          for (int j = 0; j < TD; ++j) xv = fmaf(ajs[j], xv, dj[j] * kjs[j][ch * EPC + u]);
          x[u] = xv;
        }
      };
#pragma unroll 2
      for (int c = 0; c < CPR; ++c) {
        const int ch = (c + i) % CPR;
        float x[EPC];
        parent(ch, x);
#pragma unroll
        for (int u = 0; u < EPC; ++u) p = fmaf(x[u], kq[0][ch * EPC + u], p);
      }
      delta = be * (ldf((const T*)a.v + gi) - al * p);
#pragma unroll 2
      for (int c = 0; c < CPR; ++c) {
        const int ch = (c + i) % CPR;
        float x[EPC];
        parent(ch, x);
#pragma unroll
        for (int u = 0; u < EPC; ++u)
          o = fmaf(fmaf(al, x[u], delta * kq[0][ch * EPC + u]), kq[1][ch * EPC + u], o);
      }
    }
    if (active && part == 0) {
      stf((T*)a.delta_out + gi, delta);
      if (a.o_out) stf((T*)a.o_out + gi, o);
      if (a.delta_dump) a.delta_dump[gi] = delta;
      if (a.o_dump) a.o_dump[gi] = o;
      if (a.x_inout) a.x_inout[gi] += o;
    }
  }
}

template <typename T, int DK, int TD>
int launch_rs_td(const ReplaySsmArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(T) == 4 ? (size_t)a.d_v * DK * sizeof(T) : 16;
  GDN_CUDA(cudaFuncSetAttribute(replayssm_step_kernel<T, DK, TD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  constexpr int TPR = sizeof(T) == 4 || DK < 128 ? 1 : DK / 64;
  replayssm_step_kernel<T, DK, TD><<<dim3(a.R * a.W_t, a.H), 128 * TPR, smem, s>>>(a);
  return GDNBEAM_OK;
}

template <typename T, int DK>
int launch_rs_dk(const ReplaySsmArgs& a, cudaStream_t s) {
  switch (a.t) {
    case 0: return launch_rs_td<T, DK, 0>(a, s);
    case 1: return launch_rs_td<T, DK, 1>(a, s);
    case 2: return launch_rs_td<T, DK, 2>(a, s);
    case 3: return launch_rs_td<T, DK, 3>(a, s);
    case 4: return launch_rs_td<T, DK, 4>(a, s);
    case 5: return launch_rs_td<T, DK, 5>(a, s);
    case 6: return launch_rs_td<T, DK, 6>(a, s);
    default: return GDNBEAM_EUNSUPPORTED;
  }
}

template <typename T>
int dispatch_rs(const ReplaySsmArgs& a, cudaStream_t s) {
  int st;
  switch (a.d_k) {
    case 16: st = launch_rs_dk<T, 16>(a, s); break;
    case 32: st = launch_rs_dk<T, 32>(a, s); break;
    case 64: st = launch_rs_dk<T, 64>(a, s); break;
    case 128: st = launch_rs_dk<T, 128>(a, s); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
  if (st) return st;
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

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

int launch_replayssm(int dtype, const ReplaySsmArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.d_v > 128 || a.t > kRsDepth || a.R * a.W_t > 0x7FFFFFFF) return GDNBEAM_EUNSUPPORTED;
  return dtype == GDNBEAM_BF16 ? dispatch_rs<__nv_bfloat16>(a, s) : dispatch_rs<float>(a, s);
}

int launch_fullstate(int dtype, const FullStateArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.d_v > 128 || a.R * a.W_t > 0x7FFFFFFF) return GDNBEAM_EUNSUPPORTED;
  return dtype == GDNBEAM_BF16 ? dispatch<__nv_bfloat16>(a, s) : dispatch<float>(a, s);
}

}  // namespace gdnbeam
