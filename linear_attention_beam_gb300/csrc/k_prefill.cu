// Prefill recurrence: compresses each request's prompt into S_ctx.
//
// OneLA §1.1/§2.1: the shared prompt is folded into one recurrent state per
// (request, layer, head), shared by every beam. The recurrence is eq. 3 of
// §1.2 run from S = 0. One block per (request, head); the rows of S (d_k
// fp32 values each) stay in registers, two rows per thread split over a few
// threads per row pair, and the next tokens' k, q, v and gates are
// prefetched while the current ones are applied.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

// Packed fp32 pairs: one instruction does two FMAs (sm_100 family).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(uint64_t x) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Each thread holds rows i and i + 64 of S over NC = DK / TPR consecutive
// columns as packed fp32 pairs, so every key or query value read from shared
// memory feeds four FMAs; TPR threads share a row pair and a dot product ends
// in a butterfly over them. Tokens are staged CH at a time in shared memory
// (as fp32), the next chunk's loads in flight while the current one is
// applied, so the per-token loop reads only shared memory and needs no block
// barrier. Each thread's column segment is padded by 16 bytes so the TPR
// threads of a row pair read different banks.
template <typename T, int DK, int TPR, int CH>
__global__ void __launch_bounds__(64 * TPR, TPR <= 4 ? 2 : 1) prefill_scan_kernel(
    int L, int H, int Hk, int dv, const T* __restrict__ q, const T* __restrict__ k,
    const T* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    float* __restrict__ sctx, long long rstride, T* __restrict__ o_last, float* __restrict__ x) {
  constexpr int NC = DK / TPR;            // columns per thread
  constexpr int NP = NC / 2;              // packed pairs per row
  constexpr int EPV = 16 / (int)sizeof(T);  // elements per 16-byte load
  constexpr int NT = 64 * TPR;
  constexpr int KV = DK / EPV;            // 16-byte pieces per k or q row
  constexpr int PF = (CH * (2 * KV + 128 / EPV) + NT - 1) / NT;  // loads per thread per chunk
  constexpr int PAD = TPR > 1 ? 4 : 0;
  constexpr int RS = TPR * (NC + PAD);     // floats per staged k or q row
  extern __shared__ __align__(16) float sm[];
  float* ks = sm;                          // [2][CH][RS]
  float* qs = ks + 2 * CH * RS;            // [2][CH][RS]
  float* vs = qs + 2 * CH * RS;            // [2][CH][128]
  float2* gs = reinterpret_cast<float2*>(vs + 2 * CH * 128);  // [2][CH]
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  const int hk = h / (H / Hk);  // the key head this value head reads
  const int v0 = blockIdx.y * 128;  // this block's 128 value rows
  const int dvb = min(128, dv - v0);
  const int tid = threadIdx.x;
  const int i = tid / TPR, part = tid % TPR, c0 = part * NC;  // rows i and i + 64
  const int VV = dvb / EPV;                // 16-byte pieces of this block's v slice
  const int per_chunk = CH * (2 * KV + VV);
  uint64_t S[2][NP];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int c = 0; c < NP; ++c) S[rr][c] = 0ull;  // +0.0f, +0.0f
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
        int heads, head;
        if (u < CH * KV) { t = u / KV; piece = u % KV; base = k; width = DK; heads = Hk; head = hk; }
        else if (u < 2 * CH * KV) { t = (u - CH * KV) / KV; piece = (u - CH * KV) % KV; base = q; width = DK; heads = Hk; head = hk; }
        else { t = (u - 2 * CH * KV) / VV; piece = (u - 2 * CH * KV) % VV + v0 / EPV; base = v; width = dv; heads = H; head = h; }
        const int pos = chunk * CH + t;
        if (pos < L)
          buf[e] = __ldg(reinterpret_cast<const uint4*>(base + ((row0 + pos) * heads + head) * width) + piece);
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
        for (int xx = 0; xx < EPV; ++xx) dst[xx] = St<T>::to_f(el[xx]);
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
  const bool act0 = i < dvb, act1 = i + 64 < dvb;
  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int sb = chunk & 1;
    uint4 nxt[PF];
    float2 gn;
    if (chunk + 1 < n_chunks) load(chunk + 1, nxt, gn);
    const int steps = min(CH, L - chunk * CH);
    for (int t = 0; t < steps; ++t) {
      const uint64_t* kr = reinterpret_cast<const uint64_t*>(ks + (size_t)(sb * CH + t) * RS + part * (NC + PAD));
      const uint64_t* qr = reinterpret_cast<const uint64_t*>(qs + (size_t)(sb * CH + t) * RS + part * (NC + PAD));
      const float2 g = gs[sb * CH + t];
      uint64_t pa0 = 0ull, pa1 = 0ull, pb0 = 0ull, pb1 = 0ull;
#pragma unroll
      for (int c = 0; c < NP; c += 2) {
        const uint64_t k0 = kr[c];
        pa0 = fma2(S[0][c], k0, pa0);
        pb0 = fma2(S[1][c], k0, pb0);
        if (c + 1 < NP) {
          const uint64_t k1 = kr[c + 1];
          pa1 = fma2(S[0][c + 1], k1, pa1);
          pb1 = fma2(S[1][c + 1], k1, pb1);
        }
      }
      const float2 fa0 = up2(pa0), fa1 = up2(pa1), fb0 = up2(pb0), fb1 = up2(pb1);
      float p0 = (fa0.x + fa0.y) + (fa1.x + fa1.y);
      float p1 = (fb0.x + fb0.y) + (fb1.x + fb1.y);
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) {
        p0 += __shfl_xor_sync(0xffffffffu, p0, o);
        p1 += __shfl_xor_sync(0xffffffffu, p1, o);
      }
      const float* vrow = vs + (size_t)(sb * CH + t) * 128;
      const float d0 = g.y * (vrow[act0 ? i : 0] - g.x * p0);
      const float d1 = g.y * (vrow[act1 ? i + 64 : 0] - g.x * p1);
      const uint64_t aa = pk2(g.x, g.x), dd0 = pk2(d0, d0), dd1 = pk2(d1, d1);
      uint64_t oa0 = 0ull, oa1 = 0ull, ob0 = 0ull, ob1 = 0ull;
#pragma unroll
      for (int c = 0; c < NP; ++c) {
        const uint64_t kc = kr[c], qc = qr[c];
        S[0][c] = fma2(aa, S[0][c], mul2(dd0, kc));
        S[1][c] = fma2(aa, S[1][c], mul2(dd1, kc));
        if (c & 1) {
          oa1 = fma2(S[0][c], qc, oa1);
          ob1 = fma2(S[1][c], qc, ob1);
        } else {
          oa0 = fma2(S[0][c], qc, oa0);
          ob0 = fma2(S[1][c], qc, ob0);
        }
      }
      const float2 ga0 = up2(oa0), ga1 = up2(oa1), gb0 = up2(ob0), gb1 = up2(ob1);
      float o0 = (ga0.x + ga0.y) + (ga1.x + ga1.y);
      float o1 = (gb0.x + gb0.y) + (gb1.x + gb1.y);
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) {
        o0 += __shfl_xor_sync(0xffffffffu, o0, off);
        o1 += __shfl_xor_sync(0xffffffffu, o1, off);
      }
      if (part == 0) {
        const int pos = chunk * CH + t;
        const size_t row = row0 + pos;
        if (act0) {
          if (x) x[(row * H + h) * dv + v0 + i] += o0;
          if (o_last && pos == L - 1) stf(o_last + ((size_t)r * H + h) * dv + v0 + i, o0);
        }
        if (act1) {
          if (x) x[(row * H + h) * dv + v0 + i + 64] += o1;
          if (o_last && pos == L - 1) stf(o_last + ((size_t)r * H + h) * dv + v0 + i + 64, o1);
        }
      }
    }
    // buffer sb ^ 1 was last read in the previous chunk, before its barrier
    if (chunk + 1 < n_chunks) stash(sb ^ 1, nxt, gn);
    __syncthreads();
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int ri = i + 64 * rr;
    if (ri < dvb) {
      float* out = sctx + (size_t)r * rstride + ((size_t)h * dv + v0 + ri) * DK + c0;
#pragma unroll
      for (int c = 0; c < NP; ++c) {
        const float2 f = up2(S[rr][c]);
        out[2 * c] = f.x;
        out[2 * c + 1] = f.y;
      }
    }
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
  prefill_scan_kernel<T, DK, TPR, CH><<<dim3(c.R * c.H, (c.d_v + 127) / 128), 64 * TPR, smem, s>>>(
      L, c.H, key_heads(c), c.d_v, (const T*)q, (const T*)k, (const T*)v, alpha, beta, sctx, rs,
      (T*)o_last, x);
  return GDNBEAM_OK;
}

template <typename T>
int dispatch_dk(const gdnbeam_config& c, int L, const void* q, const void* k, const void* v,
                const float* alpha, const float* beta, float* sctx, long long rs, void* o_last,
                float* x, cudaStream_t s) {
  const int epv = 16 / (int)sizeof(T);
  if (c.d_v % epv != 0 || ((uintptr_t)q & 15) || ((uintptr_t)k & 15) || ((uintptr_t)v & 15) ||
      (key_heads(c) * c.d_k) % epv != 0)
    return GDNBEAM_EUNSUPPORTED;
  int st;
  switch (c.d_k) {
    case 16: st = launch_scan<T, 16, 1>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 32: st = launch_scan<T, 32, 1>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 64: st = launch_scan<T, 64, 2>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 128: st = launch_scan<T, 128, 4>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    case 256: st = launch_scan<T, 256, 8>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s); break;
    default: return GDNBEAM_EUNSUPPORTED;
  }
  if (st) return st;
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

int launch_prefill_scan(const gdnbeam_config& c, int L, const void* q, const void* k,
                        const void* v, const float* alpha, const float* beta, float* sctx,
                        long long rs, void* o_last, float* x, cudaStream_t s, void* scratch,
                        size_t scratch_bytes) {
  if (L <= 0) return GDNBEAM_EINVAL;
  if (c.d_v > 128 && c.d_v % 128 != 0) return GDNBEAM_EUNSUPPORTED;
  const size_t out_bytes = x ? prefill_out_scratch_bytes(c, L) : 0;
  if (tc_prefill_supported(c) && (!x || (scratch && scratch_bytes >= out_bytes))) {
    const long long qw = (long long)key_heads(c) * c.d_k;
    // (bf16 queries: two bytes each)
    const char* q_last = (const char*)q + (size_t)(L - 1) * qw * 2;
    if (!x)
      return launch_prefill_tc(c, L, q_last, (long long)L * qw, k, v, alpha, beta, sctx, rs, o_last, s);
    // stacked layers: the chain leaves every chunk's start state and every
    // token's record in scratch, then every position's o joins the stream
    float* dl = (float*)scratch;
    float* s0 = dl + (size_t)c.R * L * c.H * c.d_v;
    int st = launch_prefill_tc(c, L, q_last, (long long)L * qw, k, v, alpha, beta, sctx, rs, o_last,
                               s, s0, dl);
    if (st) return st;
    return launch_prefill_out_tc(c, L, q, k, alpha, s0, dl, x, s);
  }
  if (c.dtype == GDNBEAM_BF16)
    return dispatch_dk<__nv_bfloat16>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s);
  return dispatch_dk<float>(c, L, q, k, v, alpha, beta, sctx, rs, o_last, x, s);
}

}  // namespace gdnbeam
