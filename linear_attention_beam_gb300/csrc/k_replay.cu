// Fused shared-context replay on CUDA cores (shape-general path).
//
// OneLA §2.3 eqs. 6-8 and §2.5: every block takes one (request, head) and a
// tile of beams, reads the shared context state S_ctx once for the whole
// tile, forms u_q = S_ctx q and u_k = S_ctx k for each beam, folds the
// ancestors' records (alpha_j, delta_j, k_j) into both projections, then
// writes delta_t (the new record's vector) and o_t. No per-beam d_v x d_k
// state is formed. The bf16 d = 128 hot path uses the tcgen05 version.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

constexpr int kBeams = 16;    // beams per block
constexpr int kThreads = 128; // one thread per value row of a 128-row block
constexpr int kChunk = 32;    // key columns of S_ctx staged per pass

template <typename T>
__global__ void __launch_bounds__(kThreads) replay_simt_kernel(ReplayArgs a) {
  const int H = a.H, Hk = a.Hk, dk = a.d_k, dv = a.d_v, t = a.t;
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  const int hk = h / (H / Hk);  // the key head this value head reads
  const int b0 = blockIdx.y * kBeams;
  const int nb = min(kBeams, a.W_t - b0);
  const int v0 = blockIdx.z * kThreads;     // first value row of this block
  const int dvb = min(kThreads, dv - v0);    // value rows of this block
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ float sm[];
  float* qs = sm;                          // [kBeams][dk]
  float* ks = qs + kBeams * dk;            // [kBeams][dk]
  float* sc = ks + kBeams * dk;            // [dv][kChunk + 1]
  float* cq = sc + 128 * (kChunk + 1);     // [kBeams][MAX_T]
  float* ck = cq + kBeams * GDNBEAM_MAX_T; // [kBeams][MAX_T]
  float* kq = ck + kBeams * GDNBEAM_MAX_T; // [kBeams]
  int* slot = (int*)(kq + kBeams);         // [kBeams][MAX_T]

  const T* q = (const T*)a.q;
  const T* k = (const T*)a.k;
  const T* v = (const T*)a.v;

  // 1. this tile's queries and keys, and the ancestors' slots
  for (int i = tid; i < nb * dk; i += kThreads) {
    int b = i / dk, c = i % dk;
    size_t off = ((size_t)(r * a.W_t + b0 + b) * Hk + hk) * dk + c;
    qs[i] = ldf(q + off);
    ks[i] = ldf(k + off);
  }
  for (int i = tid; i < nb * t; i += kThreads) {
    int b = i / t, j = i % t;
    int s = a.anc[(size_t)(r * a.W_t + b0 + b) * a.anc_stride + j];
    if (s < 0 || s >= a.depth[j].W_j) {
      raise_error(a.err, GDNBEAM_DERR_SLOT);
      s = -1;
    }
    slot[b * GDNBEAM_MAX_T + j] = s;
  }
  __syncthreads();

  // 2. replay scalars k_j . q_t, k_j . k_t (eqs. 6-7) and k_t . q_t (eq. 8)
  for (int p = warp; p < nb * (t + 1); p += kThreads / 32) {
    int b = p / (t + 1), j = p % (t + 1);
    float sq = 0.0f, sk = 0.0f;
    if (j < t) {
      int s = slot[b * GDNBEAM_MAX_T + j];
      if (s >= 0) {
        const T* kr = (const T*)a.depth[j].k + ((size_t)(r * a.depth[j].W_j + s) * Hk + hk) * dk;
        for (int c = lane; c < dk; c += 32) {
          float kv = ldf(kr + c);
          sq += kv * qs[b * dk + c];
          sk += kv * ks[b * dk + c];
        }
      }
    } else {
      for (int c = lane; c < dk; c += 32) sq += ks[b * dk + c] * qs[b * dk + c];
    }
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (lane == 0) {
      if (j < t) {
        cq[b * GDNBEAM_MAX_T + j] = sq;
        ck[b * GDNBEAM_MAX_T + j] = sk;
      } else {
        kq[b] = sq;
      }
    }
  }

  // 3. u_q = S_ctx q, u_k = S_ctx k for every beam of the tile
  float uq[kBeams], uk[kBeams];
#pragma unroll
  for (int b = 0; b < kBeams; ++b) { uq[b] = 0.0f; uk[b] = 0.0f; }
  const float* S = a.sctx + (size_t)r * a.sctx_rstride + ((size_t)h * dv + v0) * dk;
  for (int c0 = 0; c0 < dk; c0 += kChunk) {
    __syncthreads();
    for (int i = tid; i < dvb * kChunk; i += kThreads) {
      int row = i / kChunk, c = i % kChunk;
      sc[row * (kChunk + 1) + c] = (c0 + c < dk) ? S[(size_t)row * dk + c0 + c] : 0.0f;
    }
    __syncthreads();
    if (tid < dvb) {
      const int cn = min(kChunk, dk - c0);
      for (int c = 0; c < cn; ++c) {
        float sv = sc[tid * (kChunk + 1) + c];
#pragma unroll
        for (int b = 0; b < kBeams; ++b) {
          if (b < nb) {
            uq[b] = fmaf(sv, qs[b * dk + c0 + c], uq[b]);
            uk[b] = fmaf(sv, ks[b * dk + c0 + c], uk[b]);
          }
        }
      }
    }
  }
  __syncthreads();

  // 4. fold the ancestors' records, then eq. 8
  if (tid < dvb) {
    const int i = v0 + tid;
#pragma unroll
    for (int b = 0; b < kBeams; ++b) {
      if (b >= nb) break;
      float u_q = uq[b], u_k = uk[b];
      for (int j = 0; j < t; ++j) {
        int s = slot[b * GDNBEAM_MAX_T + j];
        if (s < 0) continue;
        size_t rec = (size_t)(r * a.depth[j].W_j + s) * H + h;
        float aj = a.depth[j].alpha[rec];
        float dj = ldf((const T*)a.depth[j].delta + rec * dv + i);
        u_q = aj * u_q + dj * cq[b * GDNBEAM_MAX_T + j];
        u_k = aj * u_k + dj * ck[b * GDNBEAM_MAX_T + j];
      }
      size_t row = (size_t)r * a.W_t + b0 + b;
      float al = a.alpha[row * H + h], be = a.beta[row * H + h];
      size_t off = (row * H + h) * dv + i;
      float delta = be * (ldf(v + off) - al * u_k);
      float o = al * u_q + delta * kq[b];
      stf((T*)a.delta_out + off, delta);
      if (a.o_out) stf((T*)a.o_out + off, o);
      if (a.delta_dump) a.delta_dump[off] = delta;
      if (a.o_dump) a.o_dump[off] = o;
      if (a.x_inout) a.x_inout[off] += o;
    }
  }
}

}  // namespace

int launch_replay(int dtype, const ReplayArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.t >= GDNBEAM_MAX_T) return GDNBEAM_EUNSUPPORTED;
  dim3 grid(a.R * a.H, (a.W_t + kBeams - 1) / kBeams, (a.d_v + kThreads - 1) / kThreads);
  if (grid.y > 65535) return GDNBEAM_EUNSUPPORTED;
  size_t smem = sizeof(float) * (2 * kBeams * a.d_k + 128 * (kChunk + 1) +
                                 2 * kBeams * GDNBEAM_MAX_T + kBeams) +
                sizeof(int) * kBeams * GDNBEAM_MAX_T;
  if (dtype == GDNBEAM_BF16) {
    GDN_CUDA(cudaFuncSetAttribute(replay_simt_kernel<__nv_bfloat16>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    replay_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
  } else {
    GDN_CUDA(cudaFuncSetAttribute(replay_simt_kernel<float>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    replay_simt_kernel<float><<<grid, kThreads, smem, s>>>(a);
  }
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
