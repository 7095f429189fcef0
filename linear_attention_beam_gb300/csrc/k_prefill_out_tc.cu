// Every prompt position's output of the chunked prefill, for stacked layers
// (bf16 storage, d_k = d_v = 128): the residual stream of a stacked model
// needs o_i = S_i q_i at every token i (OneLA §1.2 eq. 3), not only at the
// last one.
//
// The chain kernel (k_prefill_tc.cu) leaves, per (request, head), the state
// at the start of every 64-token chunk (S0) and every token's record delta
// (OneLA §2.2 eq. 4). Within a chunk, with g_i the product of the chunk's
// decays up to and including token i,
//   S_i = g_i S0 + sum_{j<=i} (g_i / g_j) delta_j k_j^T,
// so
//   o_i = g_i (S0 q_i) + sum_{j<=i} (g_i / g_j) (q_i . k_j) delta_j,
// or, with the 128 value rows as the MMA's M and the chunk's tokens as N,
//   O^T = (S0 Q^T) diag(g) + delta^T M^T,   M_ij = (g_i / g_j) q_i.k_j (j <= i).
// The chunks are independent given S0, so one block takes one chunk of one
// (request, head) and the whole prompt runs in parallel. Three tcgen05
// contractions per block:
//   MMA1  G[i][j]    = sum_k Q[i][k] K[j][k]          (A, B: TMA tiles in smem)
//   MMA2  X[v][i]    = sum_k S0[v][k] Q[i][k]         (A: S0 hi/lo in TMEM)
//   MMA3  X[v][i]   += sum_j delta^T[v][j] M[i][j]    (A: delta^T hi/lo in TMEM,
//                                                      B: M hi/lo in smem)
// with X scaled by g_i between MMA2 and MMA3; fp32 operands are split into
// bf16 hi + lo halves (~16 mantissa bits), q and k are exact bf16. The
// output is added to the fp32 residual stream x.
//
// Roles (192 threads; 256 TMEM columns and ~107 KB of shared memory, so two
// blocks share an SM):
//   warp 0      TMA loads of the chunk's query and key rows, and of the
//               residual stream's rows of this head
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2-5   thread = TMEM lane: the chunk's decays, G -> M (lanes < 64,
//               lane = token), S0 and delta^T into TMEM, the g scaling and
//               the residual update (lane = value row)
// Every wait is bounded in time; on a time-out the block raises
// GDNBEAM_DERR_TIMEOUT, drains its copies and MMAs and frees TMEM.
#include <cuda.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int CH = 64;                 // tokens per chunk
constexpr int DH = 128;                // d_k = d_v
constexpr int QBLK = 128 * 128;        // A tile block [128 rows][64 bf16]: 16 KiB (rows >= 64 unused)
constexpr int KBLK = CH * 128;         // B tile block [64 rows][64 bf16]: 8 KiB
constexpr int OFF_Q = 0;               // two column blocks of Q
constexpr int OFF_K = 2 * QBLK;        // two column blocks of K
constexpr int OFF_MHI = OFF_K + 2 * KBLK;
constexpr int OFF_MLO = OFF_MHI + KBLK;
constexpr int OFF_XS = OFF_MLO + KBLK;     // the residual stream's [64 tokens][128 v] fp32
constexpr int OFF_END = OFF_XS + CH * DH * 4;
constexpr int kDynSmem = 1024 + OFF_END;
constexpr uint32_t kLoadBytes = 4 * KBLK;  // 64 rows x 128 of Q and of K
constexpr uint32_t kStreamBytes = CH * DH * 4;

// TMEM columns
constexpr uint32_t cGD = 0;     // G (lanes < 64, 64 fp32 columns), then delta^T hi (32) | lo (32)
constexpr uint32_t cX = 64;     // S0 Q^T, then O^T: fp32 [128 v][64 i]
constexpr uint32_t cSHI = 128;  // S0 hi as A operand (128 k as 64 bf16 pairs)
constexpr uint32_t cSLO = 192;  // S0 lo
constexpr uint32_t kTmemCols = 256;
constexpr int kThreads = 192;

struct PrefillOutParams {
  int R, H, Hk, L, n_chunks;
  const float* alpha;   // [R*L][H]
  const float* s0;      // [R*H][n_chunks][128 v][128 k] chunk-start states (chunk 0 unused);
                        // n_chunks is the chain kernel's (even) chunk count
  const float* delta;   // [R*L][H*128]
  float* x;             // [R*L][H*128] residual stream
  unsigned* err;
};

__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)(((col >> 3) ^ (row & 7)) & 7) << 4) +
         (uint32_t)(col & 7) * 2u;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t bf2_bits(float lo, float hi) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&x);
}
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = bf2_bits(a, b);
  lo = bf2_bits(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_out_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_x, PrefillOutParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[8];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_lg[CH];
  __shared__ float s_half;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int r = blockIdx.y / p.H, h = blockIdx.y % p.H;
  const int hk = h / (p.H / p.Hk);
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };
  const uint32_t in_full = bar(0), g_full = bar(1), ops_ready = bar(2), p_full = bar(3),
                 x_ready = bar(4), o_full = bar(5), drain_bar = bar(6), xs_full = bar(7);
  volatile int* abort = &s_abort;
  const bool has_s0 = c > 0;  // the first chunk starts from S = 0

  if (threadIdx.x == 0) {
    tc::mbar_init(in_full, 1);
    tc::mbar_init(g_full, 1);
    tc::mbar_init(ops_ready, 4);
    tc::mbar_init(p_full, 1);
    tc::mbar_init(x_ready, 4);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(drain_bar, 1);
    tc::mbar_init(xs_full, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ loads
    if (lane == 0) {
      tc::mbar_arrive_expect_tx(in_full, kLoadBytes);
      for (int kb = 0; kb < 2; ++kb) {
        tc::tma_load_3d(base + OFF_Q + kb * QBLK, &tm_q, hk * DH + kb * 64, c * CH, r, in_full);
        tc::tma_load_3d(base + OFF_K + kb * KBLK, &tm_k, hk * DH + kb * 64, c * CH, r, in_full);
      }
      tc::mbar_arrive_expect_tx(xs_full, kStreamBytes);
      tc::tma_load_3d(base + OFF_XS, &tm_x, h * DH, c * CH, r, xs_full);
      tc::mbar_wait_drain(in_full, 0);  // the copies land before the block exits
      tc::mbar_wait_drain(xs_full, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t id64 = tc::idesc_bf16_f32(128, 64);
      bool ok = tc::mbar_wait_sleep(in_full, 0, abort, p.err);
      if (ok) {
        tc::fence_after_sync();
        // MMA1: G = Q K^T (A: 128 query rows, of which the first 64 are the
        // chunk's; B: the chunk's 64 key rows)
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = tc::sw128_desc(base + OFF_Q + kb * QBLK) + 2u * kk;
            const uint64_t b = tc::sw128_desc(base + OFF_K + kb * KBLK) + 2u * kk;
            tc::mma_bf16(tmem + cGD, a, b, id64, (kb | kk) != 0);
          }
        tc::mma_commit(g_full);
        ok = tc::mbar_wait_sleep(ops_ready, 0, abort, p.err);
      }
      if (ok && has_s0) {
        tc::fence_after_sync();
        // MMA2: X = S0 Q^T (B: the chunk's 64 query rows)
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t b = tc::sw128_desc(base + OFF_Q + kb * QBLK) + 2u * kk;
            const uint32_t col = (uint32_t)(kb * 32 + kk * 8);
            tc::mma_bf16_ts(tmem + cX, tmem + cSHI + col, b, id64, (kb | kk) != 0);
            tc::mma_bf16_ts(tmem + cX, tmem + cSLO + col, b, id64, 1u);
          }
        tc::mma_commit(p_full);
        ok = tc::mbar_wait_sleep(x_ready, 0, abort, p.err);
      }
      if (ok) {
        tc::fence_after_sync();
        // MMA3: X += delta^T M^T (three hi/lo products)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bh = tc::sw128_desc(base + OFF_MHI) + 2u * kk;
          const uint64_t bl = tc::sw128_desc(base + OFF_MLO) + 2u * kk;
          const uint32_t col = (uint32_t)(kk * 8);
          tc::mma_bf16_ts(tmem + cX, tmem + cGD + col, bh, id64, (has_s0 || kk > 0) ? 1u : 0u);
          tc::mma_bf16_ts(tmem + cX, tmem + cGD + 32 + col, bh, id64, 1u);
          tc::mma_bf16_ts(tmem + cX, tmem + cGD + col, bl, id64, 1u);
        }
        tc::mma_commit(o_full);
      }
      tc::mma_commit(drain_bar);
      tc::mbar_wait_drain(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------------ rows
    const int lgp = warp & 3;
    const int row = 32 * lgp + lane;  // TMEM lane: a token (< 64) for M, a value row for O
    const uint32_t lb = tmem + ((uint32_t)(32 * lgp) << 16);
    const size_t tok0 = (size_t)r * p.L + (size_t)c * CH;  // the chunk's first prompt row
    const int n_tok = min(CH, p.L - c * CH);
    const size_t xw = (size_t)p.H * DH;
    auto wait = [&](uint32_t b) -> bool {
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_sleep(b, 0, abort, p.err) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    // the chunk's inclusive log2-decay prefix (tokens past the prompt decay
    // by 1); lanes 0-63 are warps 4 and 5
    if (row < CH) {
      const float a = row < n_tok ? __ldg(p.alpha + (tok0 + row) * p.H + h) : 1.f;
      float x = fmaxf(lg2(a), -100.f);  // alpha below 2^-100 acts as 0
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (row == 31) s_half = x;
      tc::named_sync(1, 64);
      if (row >= 32) x += s_half;
      s_lg[row] = x;
    }
    // S0 row (value row `row`) -> hi/lo A operand
    if (has_s0) {
      const float* s0 = p.s0 + (((size_t)(r * p.H + h) * p.n_chunks + c) * DH + row) * DH;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float4 f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __ldg(reinterpret_cast<const float4*>(s0 + 32 * q) + e);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          split2(f[e].x, f[e].y, hi[2 * e], lo[2 * e]);
          split2(f[e].z, f[e].w, hi[2 * e + 1], lo[2 * e + 1]);
        }
        tc::tmem_st16(lb + cSHI + 16 * q, hi);
        tc::tmem_st16(lb + cSLO + 16 * q, lo);
      }
    }
    // delta^T row (value row `row`) of the chunk's tokens, loaded now
    float dv[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i)
      dv[i] = i < n_tok ? __ldg(p.delta + (tok0 + i) * xw + (size_t)h * DH + row) : 0.f;
    // every row warp takes the same outcome (the barrier also publishes s_lg)
    bool ok = tc::named_sync_and(2, 128, wait(g_full));
    if (ok) {
      tc::fence_after_sync();
      if (row < CH) {
        // M row i = row: (g_i / g_j) q_i.k_j for j <= i, as hi/lo bf16, 32
        // columns of G at a time
        const float lgi = s_lg[row];
        uint8_t* mh = gb + OFF_MHI;
        uint8_t* ml = gb + OFF_MLO;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t g[32];
          tc::tmem_ld32_nowait(lb + cGD + 32 * hf, g);
          tc::tmem_wait_ld();
#pragma unroll
          for (int jc = 0; jc < 4; ++jc) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int jl = 8 * jc + 2 * e, j0 = 32 * hf + jl;
              const float m0 = j0 <= row ? ex2(lgi - s_lg[j0]) * __uint_as_float(g[jl]) : 0.f;
              const float m1 = j0 + 1 <= row ? ex2(lgi - s_lg[j0 + 1]) * __uint_as_float(g[jl + 1]) : 0.f;
              split2(m0, m1, hw[e], lw[e]);
            }
            const int col = 32 * hf + 8 * jc;
            *reinterpret_cast<uint4*>(mh + sw128(row, col)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ml + sw128(row, col)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      // delta^T hi/lo over this lane's G columns (each lane reads and then
      // overwrites only its own)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) split2(dv[32 * hf + 2 * e], dv[32 * hf + 2 * e + 1], hi[e], lo[e]);
        tc::tmem_st16(lb + cGD + 16 * hf, hi);
        tc::tmem_st16(lb + cGD + 32 + 16 * hf, lo);
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(ops_ready);
    }
    // X <- X diag(g)
    if (ok && has_s0 && (ok = wait(p_full))) {
      tc::fence_after_sync();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t xv[32];
        tc::tmem_ld32_nowait(lb + cX + 32 * hf, xv);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) xv[e] = __float_as_uint(ex2(s_lg[32 * hf + e]) * __uint_as_float(xv[e]));
        tc::tmem_st32(lb + cX + 32 * hf, xv);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(x_ready);
    }
    // x += o for the chunk's tokens (the stream's rows were staged in shared
    // memory by TMA)
    if (ok && wait(o_full) && wait(xs_full)) {
      tc::fence_after_sync();
      const float* xs = reinterpret_cast<const float*>(gb + OFF_XS) + row;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float o[32];
        tc::tmem_ld32(lb + cX + 32 * hf, o);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i = 32 * hf + e;
          if (i < n_tok) p.x[(tok0 + i) * xw + (size_t)h * DH + row] = xs[i * DH] + o[e];
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// The chain kernel walks 128-token stages, so its chunk count (the stride of
// the start-state buffer) is rounded up to an even number.
inline int state_chunks(int L) { return 2 * ((L + 2 * CH - 1) / (2 * CH)); }

}  // namespace

size_t prefill_out_scratch_bytes(const gdnbeam_config& c, int L) {
  const size_t n_chunks = (size_t)state_chunks(L);
  return (size_t)c.R * c.H * n_chunks * DH * DH * sizeof(float) +
         (size_t)c.R * L * c.H * DH * sizeof(float);
}

int launch_prefill_out_tc(const gdnbeam_config& c, int L, const void* q, const void* k,
                          const float* alpha, const float* s0, const float* delta, float* x,
                          cudaStream_t s) {
  if (L <= 0) return GDNBEAM_EINVAL;
  const int Hk = key_heads(c);
  CUtensorMap mq, mk, mx;
  if (!prefill_rows_map(&mq, q, c.R, L, Hk * DH, CH) || !prefill_rows_map(&mk, k, c.R, L, Hk * DH, CH) ||
      !prefill_stream_map(&mx, x, c.R, L, c.H * DH))
    return GDNBEAM_ECUDA;
  PrefillOutParams p{};
  p.R = c.R; p.H = c.H; p.Hk = Hk; p.L = L;
  p.n_chunks = state_chunks(L);
  p.alpha = alpha; p.s0 = s0; p.delta = delta; p.x = x;
  p.err = error_word();
  GDN_CUDA(cudaFuncSetAttribute(prefill_out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kDynSmem));
  prefill_out_tc_kernel<<<dim3((L + CH - 1) / CH, c.R * c.H), kThreads, kDynSmem, s>>>(mq, mk, mx, p);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
