// CUDA-core kernels for the shape-general path: embedding gather, RMSNorm,
// a tiled fp32-accumulating GEMM, and the projection / logits epilogues.
// These serve the fp32 storage runs and any shape the tensor-core kernels do
// not cover; the bf16 d = 128 hot path uses the tcgen05 kernels instead.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

// ---------------------------------------------------------------------------
// Embedding gather: u[m] = E[tok[m]]
// ---------------------------------------------------------------------------
template <typename T>
__global__ void gather_rows_kernel(int n, int d_model, const int32_t* __restrict__ tokens, int V,
                                   const T* __restrict__ E, T* __restrict__ u,
                                   float* __restrict__ x, unsigned* err) {
  int m = blockIdx.x;
  if (m >= n) return;
  int tok = tokens[m];
  bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) raise_error(err, GDNBEAM_DERR_TOKEN);
  const T* src = E + (size_t)(ok ? tok : 0) * d_model;
  for (int c = threadIdx.x; c < d_model; c += blockDim.x) {
    T val = ok ? src[c] : St<T>::from_f(0.0f);
    u[(size_t)m * d_model + c] = val;
    if (x) x[(size_t)m * d_model + c] = St<T>::to_f(val);
  }
}

// Same, one warp per row, 16-byte pieces: the row's token is read once (the
// warp's next row's token is fetched while this row is copied) and each
// lane issues up to kGatherU piece loads before storing any, so a warp keeps
// a whole 4 KB bf16 row in flight. cpr: 16-byte pieces per row.
constexpr int kGatherU = 8;
template <typename T>
__global__ void gather_rows_vec_kernel(int n, int cpr, const int32_t* __restrict__ tokens, int V,
                                       const uint4* __restrict__ E, uint4* __restrict__ u,
                                       float4* __restrict__ x, unsigned* err) {
  constexpr int EPC = 16 / (int)sizeof(T);
  const int lane = threadIdx.x & 31;
  const int step = gridDim.x * (blockDim.x >> 5);
  int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int tok = m < n ? __ldg(tokens + m) : 0;
  for (; m < n; m += step) {
    const int next = m + step < n ? __ldg(tokens + m + step) : 0;
    const bool ok = tok >= 0 && tok < V;
    if (!ok && lane == 0) raise_error(err, GDNBEAM_DERR_TOKEN);
    const uint4* src = E + (size_t)(ok ? tok : 0) * cpr;
    uint4* dst = u + (size_t)m * cpr;
    for (int p0 = 0; p0 < cpr; p0 += 32 * kGatherU) {
      uint4 val[kGatherU];
#pragma unroll
      for (int i = 0; i < kGatherU; ++i) {
        const int p = p0 + 32 * i + lane;
        val[i] = ok && p < cpr ? __ldg(src + p) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kGatherU; ++i) {
        const int p = p0 + 32 * i + lane;
        if (p >= cpr) continue;
        dst[p] = val[i];
        if (x) {
          const T* e = reinterpret_cast<const T*>(&val[i]);
          float4* xr = x + ((size_t)m * cpr + p) * (EPC / 4);
#pragma unroll
          for (int j = 0; j < EPC / 4; ++j)
            xr[j] = make_float4(St<T>::to_f(e[4 * j]), St<T>::to_f(e[4 * j + 1]),
                                St<T>::to_f(e[4 * j + 2]), St<T>::to_f(e[4 * j + 3]));
        }
      }
    }
    tok = next;
  }
}

int launch_gather_rows(int dtype, int n, int d_model, const int32_t* tokens, int V,
                       const void* E, void* u, float* x, unsigned* err, cudaStream_t s) {
  if (n <= 0) return GDNBEAM_OK;
  const int esz = dtype == GDNBEAM_BF16 ? 2 : 4;
  if ((d_model * esz) % 16 == 0 && ((uintptr_t)E & 15) == 0 && ((uintptr_t)u & 15) == 0 &&
      ((uintptr_t)x & 15) == 0) {
    const int cpr = d_model * esz / 16;
    // eight rows (warps) per block, at most eight blocks per SM
    const long long want = ((long long)n + 7) / 8;
    const int blocks = (int)(want < 8 * sm_count() ? want : 8 * sm_count());
    if (dtype == GDNBEAM_BF16)
      gather_rows_vec_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
          n, cpr, tokens, V, (const uint4*)E, (uint4*)u, (float4*)x, err);
    else
      gather_rows_vec_kernel<float><<<blocks, 256, 0, s>>>(n, cpr, tokens, V, (const uint4*)E,
                                                           (uint4*)u, (float4*)x, err);
    GDN_LAUNCH_CHECK();
    return GDNBEAM_OK;
  }
  if (dtype == GDNBEAM_BF16)
    gather_rows_kernel<__nv_bfloat16><<<n, 256, 0, s>>>(n, d_model, tokens, V,
        (const __nv_bfloat16*)E, (__nv_bfloat16*)u, x, err);
  else
    gather_rows_kernel<float><<<n, 256, 0, s>>>(n, d_model, tokens, V, (const float*)E,
                                                (float*)u, x, err);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

// ---------------------------------------------------------------------------
// RMSNorm rows (unit gain, eps 1e-6): one warp per row
// ---------------------------------------------------------------------------
template <typename T>
__global__ void rmsnorm_rows_kernel(int n, int d, const float* __restrict__ x, long long xs,
                                    T* __restrict__ u) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const float* row = x + (size_t)warp * xs;
  float ss = 0.0f;
  for (int c = lane; c < d; c += 32) ss += row[c] * row[c];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  float inv = 1.0f / sqrtf(ss / (float)d + 1e-6f);
  for (int c = lane; c < d; c += 32) stf(u + (size_t)warp * d + c, row[c] * inv);
}

// Same, for d a multiple of 128 up to 2048 on 16-byte aligned rows: each
// lane keeps its d / 32 values in registers (float4 loads), so the row is
// read once, and writes them back packed.
constexpr int kNormMaxVec = 16;  // float4 per lane: d <= 2048

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_rows_vec_kernel(int n, int nv, const float* __restrict__ x,
                                                               long long xs, T* __restrict__ u) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const float4* row = reinterpret_cast<const float4*>(x + (size_t)warp * xs);
  float4 v[kNormMaxVec];
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    if (k < nv) {
      v[k] = __ldg(row + lane + 32 * k);
      ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const int d = nv * 128;
  const float inv = 1.0f / sqrtf(ss / (float)d + 1e-6f);
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    if (k < nv) {
      const size_t c = (size_t)warp * d + 4 * (lane + 32 * k);
      if constexpr (sizeof(T) == 2) {
        const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].x * inv)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].y * inv)) << 16);
        const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].z * inv)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].w * inv)) << 16);
        *reinterpret_cast<uint2*>(u + c) = make_uint2(lo, hi);
      } else {
        *reinterpret_cast<float4*>(u + c) =
            make_float4(v[k].x * inv, v[k].y * inv, v[k].z * inv, v[k].w * inv);
      }
    }
  }
}

// Embedding rows into a residual stream and its first RMS norm in one pass:
// x[m] = E[tok[m]] (fp32) and u[m] = x[m] / rms(x[m]) in the storage type,
// one warp per row held in registers, with the chunk-to-lane layout and the
// arithmetic of rmsnorm_rows_vec_kernel (lane l holds 4-element chunks
// l + 32k, k < nv; d = 128 nv). A token outside [0, V) gives a zero row and
// is reported.
template <typename T>
__global__ void __launch_bounds__(256) gather_norm_rows_kernel(int n, int nv,
                                                               const int32_t* __restrict__ tokens,
                                                               int V, const T* __restrict__ E,
                                                               float* __restrict__ x,
                                                               T* __restrict__ u, unsigned* err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const int d = nv * 128;
  const int tok = __ldg(tokens + warp);
  const bool ok = tok >= 0 && tok < V;
  if (!ok && lane == 0) raise_error(err, GDNBEAM_DERR_TOKEN);
  const T* src = E + (size_t)(ok ? tok : 0) * d;
  float4 v[kNormMaxVec];
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    if (k < nv) {
      const int c = 4 * (lane + 32 * k);
      if constexpr (sizeof(T) == 2) {
        const uint2 w = ok ? __ldg(reinterpret_cast<const uint2*>(src + c)) : make_uint2(0u, 0u);
        v[k] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      } else {
        v[k] = ok ? __ldg(reinterpret_cast<const float4*>(src + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      reinterpret_cast<float4*>(x + (size_t)warp * d)[lane + 32 * k] = v[k];
      ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = 1.0f / sqrtf(ss / (float)d + 1e-6f);
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    if (k < nv) {
      const size_t c = (size_t)warp * d + 4 * (lane + 32 * k);
      if constexpr (sizeof(T) == 2) {
        const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].x * inv)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].y * inv)) << 16);
        const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].z * inv)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[k].w * inv)) << 16);
        *reinterpret_cast<uint2*>(u + c) = make_uint2(lo, hi);
      } else {
        *reinterpret_cast<float4*>(u + c) =
            make_float4(v[k].x * inv, v[k].y * inv, v[k].z * inv, v[k].w * inv);
      }
    }
  }
}

int launch_gather_norm_rows(int dtype, int n, int d, const int32_t* tokens, int V, const void* E,
                            float* x, void* u, unsigned* err, cudaStream_t s) {
  if (n <= 0) return GDNBEAM_OK;
  const int esz = dtype == GDNBEAM_BF16 ? 2 : 4;
  if (d % 128 != 0 || d > 128 * kNormMaxVec || ((uintptr_t)E & (4 * esz - 1)) != 0 ||
      ((uintptr_t)x & 15) != 0 || ((uintptr_t)u & (4 * esz - 1)) != 0)
    return GDNBEAM_EINVAL;
  const int blocks = (n + 7) / 8;
  if (dtype == GDNBEAM_BF16)
    gather_norm_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        n, d / 128, tokens, V, (const __nv_bfloat16*)E, x, (__nv_bfloat16*)u, err);
  else
    gather_norm_rows_kernel<float><<<blocks, 256, 0, s>>>(n, d / 128, tokens, V, (const float*)E,
                                                          x, (float*)u, err);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

int launch_rmsnorm_rows(int dtype, int n, int d, const float* x, long long xs, void* u,
                        cudaStream_t s) {
  if (n <= 0) return GDNBEAM_OK;
  int blocks = (n + 7) / 8;
  if (d % 128 == 0 && d <= 128 * kNormMaxVec && xs % 4 == 0 && ((uintptr_t)x & 15) == 0 &&
      ((uintptr_t)u & 15) == 0) {
    if (dtype == GDNBEAM_BF16)
      rmsnorm_rows_vec_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(n, d / 128, x, xs,
                                                                    (__nv_bfloat16*)u);
    else
      rmsnorm_rows_vec_kernel<float><<<blocks, 256, 0, s>>>(n, d / 128, x, xs, (float*)u);
    GDN_LAUNCH_CHECK();
    return GDNBEAM_OK;
  }
  if (dtype == GDNBEAM_BF16)
    rmsnorm_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(n, d, x, xs, (__nv_bfloat16*)u);
  else
    rmsnorm_rows_kernel<float><<<blocks, 256, 0, s>>>(n, d, x, xs, (float*)u);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

// ---------------------------------------------------------------------------
// C = A . B^T on CUDA cores: 64x64 tile, 16-deep k slices, 4x4 per thread
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) simt_gemm_nt_kernel(int M, int N, int K,
    const T* __restrict__ A, int lda, const T* __restrict__ B, int ldb, float* __restrict__ C,
    int ldc) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      int r = i >> 4, kk = i & 15;
      int gk = k0 + kk;
      int gm = m0 + r, gn = n0 + r;
      As[kk][r] = (gm < M && gk < K) ? ldf(A + (size_t)gm * lda + gk) : 0.0f;
      Bs[kk][r] = (gn < N && gk < K) ? ldf(B + (size_t)gn * ldb + gk) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gn = n0 + tx * 4 + j;
      if (gn < N) C[(size_t)gm * ldc + gn] = acc[i][j];
    }
  }
}

int launch_simt_gemm_nt(int dtype, int M, int N, int K, const void* A, int lda, const void* B,
                        int ldb, float* C, int ldc, cudaStream_t s) {
  if (M <= 0 || N <= 0) return GDNBEAM_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  if (grid.y > 65535) return GDNBEAM_EUNSUPPORTED;
  if (dtype == GDNBEAM_BF16)
    simt_gemm_nt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(M, N, K, (const __nv_bfloat16*)A,
        lda, (const __nv_bfloat16*)B, ldb, C, ldc);
  else
    simt_gemm_nt_kernel<float><<<grid, 256, 0, s>>>(M, N, K, (const float*)A, lda,
                                                    (const float*)B, ldb, C, ldc);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

// ---------------------------------------------------------------------------
// Projection epilogue: one warp per (row, head)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void proj_epilogue_kernel(int n, int H, int Hk, int dk, int dv, const float* __restrict__ P,
                                     T* __restrict__ q, T* __restrict__ k, T* __restrict__ v,
                                     float* __restrict__ alpha, float* __restrict__ beta,
                                     gdnbeam_dumps dmp) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= n * H) return;
  int m = gw / H, h = gw % H;  // value head h; key head h as well while h < Hk
  const int Np = 2 * Hk * dk + H * dv + 2 * H;
  const float* row = P + (size_t)m * Np;
  const float* pv = row + 2 * Hk * dk + h * dv;
  if (h < Hk) {
    const float* pq = row + h * dk;
    const float* pk = row + Hk * dk + h * dk;
    float sq = 0.0f, sk = 0.0f;
    for (int c = lane; c < dk; c += 32) { sq += pq[c] * pq[c]; sk += pk[c] * pk[c]; }
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    float iq = 1.0f / sqrtf(sq + 1e-6f), ik = 1.0f / sqrtf(sk + 1e-6f);
    const size_t oq = (size_t)m * Hk * dk + (size_t)h * dk;
    for (int c = lane; c < dk; c += 32) {
      float qq = pq[c] * iq, kk = pk[c] * ik;
      stf(q + oq + c, qq);
      stf(k + oq + c, kk);
      if (dmp.q) dmp.q[oq + c] = qq;
      if (dmp.k) dmp.k[oq + c] = kk;
    }
  }
  const size_t ov = (size_t)m * H * dv + (size_t)h * dv;
  for (int c = lane; c < dv; c += 32) {
    stf(v + ov + c, pv[c]);
    if (dmp.v) dmp.v[ov + c] = pv[c];
  }
  if (lane == 0) {
    float a = decay_gate(row[2 * Hk * dk + H * dv + h]);
    float b = write_gate(row[2 * Hk * dk + H * dv + H + h]);
    alpha[(size_t)m * H + h] = a;
    beta[(size_t)m * H + h] = b;
    if (dmp.alpha) dmp.alpha[(size_t)m * H + h] = a;
    if (dmp.beta) dmp.beta[(size_t)m * H + h] = b;
  }
}

int launch_proj_epilogue(const gdnbeam_config& c, int n, const float* P, void* q, void* k,
                         void* v, float* alpha, float* beta, const gdnbeam_dumps* d,
                         cudaStream_t s) {
  if (n <= 0) return GDNBEAM_OK;
  gdnbeam_dumps dm = d ? *d : gdnbeam_dumps{};
  long long warps = (long long)n * c.H;
  int blocks = (int)((warps + 7) / 8);
  if (c.dtype == GDNBEAM_BF16)
    proj_epilogue_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(n, c.H, key_heads(c), c.d_k, c.d_v, P,
        (__nv_bfloat16*)q, (__nv_bfloat16*)k, (__nv_bfloat16*)v, alpha, beta, dm);
  else
    proj_epilogue_kernel<float><<<blocks, 256, 0, s>>>(n, c.H, key_heads(c), c.d_k, c.d_v, P, (float*)q,
        (float*)k, (float*)v, alpha, beta, dm);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

// ---------------------------------------------------------------------------
// Logits rows: store z in the storage type and lse = max + log sum exp(z - max)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void logits_rows_kernel(int n, int V, const float* __restrict__ Z, T* __restrict__ z,
                                   float* __restrict__ lse, float* __restrict__ zd) {
  int m = blockIdx.x;
  const float* row = Z + (size_t)m * V;
  __shared__ float red[32];
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < V; c += blockDim.x) mx = fmaxf(mx, row[c]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (threadIdx.x == 0) red[0] = w;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float se = 0.0f;
  for (int c = threadIdx.x; c < V; c += blockDim.x) {
    float val = row[c];
    se += expf(val - mx);
    stf(z + (size_t)m * V + c, val);
    if (zd) zd[(size_t)m * V + c] = val;
  }
  for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = se;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    lse[m] = mx + logf(tot);
  }
}

int launch_logits_rows(int dtype, int n, int V, const float* Z, void* z, float* lse,
                       float* z_dump, cudaStream_t s) {
  if (n <= 0) return GDNBEAM_OK;
  if (dtype == GDNBEAM_BF16)
    logits_rows_kernel<__nv_bfloat16><<<n, 256, 0, s>>>(n, V, Z, (__nv_bfloat16*)z, lse, z_dump);
  else
    logits_rows_kernel<float><<<n, 256, 0, s>>>(n, V, Z, (float*)z, lse, z_dump);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
