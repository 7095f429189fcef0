// Exact global top-W beam selection and the ancestry-index update.
//
// Selection (OneLA §1.1: all live beams expand over the codebook and one
// global top-k keeps the survivors) runs in the two exact stages of RecoGEM
// §4.3: a per-row precut keeps each beam row's local top-K (K = min(W_next,
// V)), then a request-level selection picks the W_next winners among the
// precut survivors. A candidate dropped by the precut is beaten by K
// candidates of its own row, so it cannot be among the final K.
//
// Every candidate carries one 64-bit key: the orderable image of its fp32
// score in the high word and (2^32 - 1 - flat index) in the low word, so the
// largest keys are the highest scores with ties going to the lower flat
// index b*V + v. Keys are unique within a request; both stages find the
// K-th largest key by MSB-first 8-bit radix passes.
//
// Ancestry (OneLA §2.4 eq. 9): each child copies its parent's slot list and
// appends the parent's row as the slot of the previous depth.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

constexpr int kRowThreads = 512;
constexpr int kReqThreads = 1024;
constexpr int kMaxSort = 4096;

__device__ __forceinline__ uint64_t make_key(float s, uint32_t flat) {
  return ((uint64_t)orderable(s) << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}

// Block-wide radix search for the K-th largest of n keys read through get().
// Returns (prefix, mask): the K largest keys are exactly those with
// (key & mask) >= prefix. Needs hist[256] and two shared words.
template <typename Get>
__device__ void radix_kth(int n, unsigned K, Get get, unsigned* hist, unsigned* sh,
                          uint64_t& prefix_out, uint64_t& mask_out) {
  uint64_t prefix = 0, mask = 0;
  unsigned remaining = K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      uint64_t key = get(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= remaining) break;
        above += hist[d];
      }
      sh[0] = (unsigned)d;
      sh[1] = remaining - above;
      sh[2] = (hist[d] == remaining - above) ? 1u : 0u;  // whole bucket is taken
    }
    __syncthreads();
    prefix |= (uint64_t)sh[0] << shift;
    mask |= (uint64_t)0xFF << shift;
    remaining = sh[1];
    const bool done = sh[2] != 0;
    __syncthreads();
    if (done) break;
  }
  prefix_out = prefix;
  mask_out = mask;
}

// Stage 1: per beam row, the local top-K keys (unordered) -> cand[row][K].
template <typename T>
__global__ void __launch_bounds__(kRowThreads) select_rowcut_kernel(
    int W_t, int V, int K, const T* __restrict__ logits, const float* __restrict__ lse,
    const float* __restrict__ cum, const float* __restrict__ bias, uint64_t* __restrict__ cand,
    unsigned* err) {
  extern __shared__ uint64_t keys[];  // [V]
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[4];
  const int row = blockIdx.x;
  const int b = row % W_t;
  const float l = lse[row];
  float cp = cum ? cum[row] : 0.0f;
  if (bias) cp = __fadd_rn(cp, bias[row]);
  const T* zr = logits + (size_t)row * V;
  bool bad = false;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    float s = __fadd_rn(cp, __fsub_rn(ldf(zr + v), l));
    if (!isfinite(s)) bad = true;
    keys[v] = make_key(s, (uint32_t)b * (uint32_t)V + (uint32_t)v);
  }
  if (bad) raise_error(err, GDNBEAM_DERR_NONFINITE);
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  uint64_t* out = cand + (size_t)row * K;
  if (K >= V) {
    for (int v = threadIdx.x; v < V; v += blockDim.x) out[v] = keys[v];
    return;
  }
  uint64_t prefix, mask;
  radix_kth(V, (unsigned)K, [&](int i) { return keys[i]; }, hist, sh, prefix, mask);
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    uint64_t key = keys[v];
    if ((key & mask) >= prefix) {
      unsigned idx = atomicAdd(&sh[3], 1u);
      if (idx < (unsigned)K) out[idx] = key;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh[3] != (unsigned)K) raise_error(err, GDNBEAM_DERR_SELECT);
}

// Stage 2: per request, the W_next largest of its W_t*K precut keys, sorted.
__global__ void __launch_bounds__(kReqThreads) select_request_kernel(
    int W_t, int K, int W_next, int V, const uint64_t* __restrict__ cand,
    int32_t* __restrict__ parents, int32_t* __restrict__ tokens, float* __restrict__ cum_next,
    unsigned* err) {
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[4];
  __shared__ uint64_t win[kMaxSort];
  const int r = blockIdx.x;
  const int n = W_t * K;
  const uint64_t* c = cand + (size_t)r * n;
  uint64_t prefix = 0, mask = 0;
  if (W_next < n) {
    radix_kth(n, (unsigned)W_next, [&](int i) { return c[i]; }, hist, sh, prefix, mask);
  }
  int P = 1;
  while (P < W_next) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) win[i] = 0;
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    uint64_t key = c[i];
    if ((key & mask) >= prefix) {
      unsigned idx = atomicAdd(&sh[3], 1u);
      if (idx < (unsigned)W_next) win[idx] = key;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh[3] != (unsigned)W_next) raise_error(err, GDNBEAM_DERR_SELECT);
  // bitonic sort, descending
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        int j = i ^ stride;
        if (j > i) {
          bool desc = (i & size) == 0;
          uint64_t a = win[i], bb = win[j];
          if (desc ? (a < bb) : (a > bb)) { win[i] = bb; win[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < W_next; i += blockDim.x) {
    uint64_t key = win[i];
    uint32_t flat = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu);
    size_t o = (size_t)r * W_next + i;
    parents[o] = (int32_t)(flat / (uint32_t)V);
    tokens[o] = (int32_t)(flat % (uint32_t)V);
    cum_next[o] = from_orderable((uint32_t)(key >> 32));
  }
}

__global__ void ancestry_kernel(int R, int t, int T, int V, int W_prev, int W_t,
                                const int32_t* __restrict__ parents,
                                const int32_t* __restrict__ tokens,
                                const int32_t* __restrict__ anc_prev,
                                const int32_t* __restrict__ sid_prev, int32_t* __restrict__ anc_out,
                                int32_t* __restrict__ sid_out, unsigned* err) {
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= R * W_t) return;
  int r = idx / W_t;
  int tok = tokens[idx];
  if (tok < 0 || tok >= V) {
    raise_error(err, GDNBEAM_DERR_TOKEN);
    tok = 0;
  }
  int32_t* so = sid_out + (size_t)idx * T;
  if (t == 0) {
    so[0] = tok;
    return;
  }
  int p = parents[idx];
  if (p < 0 || p >= W_prev) {
    raise_error(err, GDNBEAM_DERR_PARENT);
    p = 0;
  }
  size_t prow = (size_t)r * W_prev + p;
  if (anc_out) {
    int32_t* ao = anc_out + (size_t)idx * T;
    for (int j = 0; j < t - 1; ++j) ao[j] = anc_prev[prow * T + j];
    ao[t - 1] = p;
  }
  for (int s = 0; s < t; ++s) so[s] = sid_prev[prow * T + s];
  so[t] = tok;
}

}  // namespace

size_t select_scratch_bytes(int R, int W_t, int W_next, int V) {
  int K = W_next < V ? W_next : V;
  return (size_t)R * W_t * K * sizeof(uint64_t);
}

int launch_select(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                  const float* lse, const float* cum, const float* bias, int32_t* parents,
                  int32_t* tokens, float* cum_next, void* scratch, unsigned* err, cudaStream_t s) {
  if (W_next > kMaxSort || V > 16384) return GDNBEAM_EUNSUPPORTED;
  const int K = W_next < V ? W_next : V;
  uint64_t* cand = (uint64_t*)scratch;
  size_t smem = (size_t)V * sizeof(uint64_t);
  if (dtype == GDNBEAM_BF16) {
    auto kern = select_rowcut_kernel<__nv_bfloat16>;
    GDN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<R * W_t, kRowThreads, smem, s>>>(W_t, V, K, (const __nv_bfloat16*)logits, lse, cum,
                                            bias, cand, err);
  } else {
    auto kern = select_rowcut_kernel<float>;
    GDN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<R * W_t, kRowThreads, smem, s>>>(W_t, V, K, (const float*)logits, lse, cum, bias,
                                            cand, err);
  }
  GDN_LAUNCH_CHECK();
  select_request_kernel<<<R, kReqThreads, 0, s>>>(W_t, K, W_next, V, cand, parents, tokens,
                                                  cum_next, err);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

int launch_ancestry(int R, int t, int T, int V, int W_prev, int W_t, const int32_t* parents,
                    const int32_t* tokens, const int32_t* anc_prev, const int32_t* sid_prev,
                    int32_t* anc_out, int32_t* sid_out, unsigned* err, cudaStream_t s) {
  int n = R * W_t;
  if (n <= 0) return GDNBEAM_OK;
  ancestry_kernel<<<(n + 255) / 256, 256, 0, s>>>(R, t, T, V, W_prev, W_t, parents, tokens,
                                                  anc_prev, sid_prev, anc_out, sid_out, err);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
