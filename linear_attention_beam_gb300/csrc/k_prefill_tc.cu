// Chunked prefill on tcgen05 tensor cores (bf16 storage, d_k = d_v = 128):
// the shared context state S_ctx of OneLA §2.1, i.e. eq. 3 (OneLA §1.2) run
// over the prompt from S = 0, evaluated 64 tokens at a time.
//
// Within a chunk with incoming state S0, write g_i for the product of the
// decays alpha of the chunk's tokens up to and including i. Unrolling eq. 3
// (its rank-one form is eq. 4) gives the chunk's records delta_i (the
// delta of eq. 4) and its final state as
//   S_i   = g_i S0 + sum_{j<=i} (g_i / g_j) delta_j k_j^T,
//   delta = T Y,          Y_i = v_i - g_i S0 k_i,
//   T     = (I + diag(beta) L)^-1 diag(beta),
//   L_ij  = (g_i / g_j) k_i.k_j  for j < i (strictly lower),
//   S_C   = g_C S0 + sum_j (g_C / g_j) delta_j k_j^T.
// T depends only on the chunk's keys and gates, so it is built ahead of the
// sequential chain; the chain per chunk is three tensor-core contractions
// with the 128 value rows as the MMA's M:
//   MMA1  Z^T[v][i]      = sum_k S0[v][k] K[i][k]       (A: S0 in TMEM)
//   MMA2  delta^T[v][i]  = sum_m Y^T[v][m] T[i][m]      (A: Y^T in TMEM)
//   MMA3  S[v][k]       += sum_i (r_i delta_i)[v] K[i][k], r_i = g_C / g_i
// with S kept in fp32 in TMEM and the fp32 operands (S0, Y, T, r delta)
// split into bf16 hi + lo halves (~16 mantissa bits); q, k, v are bf16 on
// input and exact as operands. The output is S_ctx and o at the prompt's
// last token (o = S_L q_L).
//
// Roles (448 threads, one block per (request, head), one block per SM):
//   warp 0      TMA loader: 128-token stages of K and V rows (two chunks)
//   warp 1      TMEM owner and MMA issuer (one thread); it also forms
//               K K^T for both chunks of a stage (the Gram matrix of L)
//   warps 2-5   the chain: thread = value row (TMEM lane); per chunk it
//               turns S into the hi/lo A operand (and scales S by g_C),
//               forms Y from Z and v, and r delta from delta
//   warps 6-13  T builders: decays, L from the Gram matrix, the unit lower
//               triangular inverse by 16 x 16 blocks, T in hi/lo and K^T
// Hand-overs are mbarriers; every wait is bounded in time.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int CH = 64;                    // tokens per chunk
constexpr int PAIR = 2 * CH;              // tokens per input stage
constexpr int DH = 128;                   // d_k = d_v
constexpr int KBLK = PAIR * 128;          // [128 rows][64 bf16] block: 16 KiB
constexpr int IN_BYTES = 4 * KBLK;        // K (two column blocks) + V (two): 64 KiB
constexpr int KT_BYTES = DH * CH * 2;     // K^T of a chunk: 16 KiB
constexpr int T_BYTES = CH * CH * 2;      // T hi or lo of a chunk: 8 KiB
constexpr int XS = CH + 4;                // padded fp32 row of the triangular scratch
constexpr int PS = 20;                    // padded row of a 16 x 16 block product

constexpr int OFF_IN = 0;
constexpr int OFF_KT = 2 * IN_BYTES;
constexpr int OFF_THI = OFF_KT + KT_BYTES;
constexpr int OFF_TLO = OFF_THI + T_BYTES;
constexpr int OFF_AS = OFF_TLO + T_BYTES;
constexpr int OFF_XS = OFF_AS + 2 * CH * XS * 4;  // A of both chunks of a stage
constexpr int OFF_PS = OFF_XS + CH * XS * 4;
constexpr int OFF_VEC = OFF_PS + 3 * 16 * PS * 4;      // log2-decay, g, r, beta: [4][64] each
constexpr int OFF_END = OFF_VEC + 4 * 4 * CH * 4 + 64;
constexpr int kDynSmem = 1024 + OFF_END;

// TMEM columns
constexpr uint32_t cSACC = 0;    // S, fp32 [128 v][128 k]
constexpr uint32_t cSAHI = 128;  // S0 hi as A operand (128 k as 64 bf16 pairs)
constexpr uint32_t cSALO = 192;  // S0 lo
constexpr uint32_t cZD = 256;    // Z^T, then delta^T, fp32 [128 v][64 i]
constexpr uint32_t cYAHI = 320;  // Y^T, then r delta^T, hi as A operand (64 i as 32 pairs)
constexpr uint32_t cYALO = 352;  // ... lo
constexpr uint32_t cG = 384;     // K K^T of a stage, fp32 [128][128]
constexpr uint32_t kTmemCols = 512;

constexpr int kChain0 = 2, kChainWarps = 4;
constexpr int kT0 = kChain0 + kChainWarps, kTWarps = 8;
constexpr int kTThreads = 32 * kTWarps;
constexpr int kThreads = 32 * (kT0 + kTWarps);

struct PrefillTcParams {
  int R, H, Hk, L, n_pairs;
  const float *alpha, *beta;  // [R*L][H]
  const uint16_t* q_last;     // per request its last token's query row (Hk*128 bf16)
  long long q_last_ld;        // elements between the requests' rows
  float* sctx;                // S_ctx of head h of request r at sctx + r*rstride + h*128*128
  long long rstride;
  __nv_bfloat16* o_last;      // [R][H*128] or null
  // stacked layers: every chunk's start state and every token's record, for
  // the all-position outputs (k_prefill_out_tc.cu)
  float* s0_out;              // [R*H][n_chunks][128 v][128 k] (chunk 0 not written)
  float* delta_out;           // [R*L][H*128]
  unsigned* err;
};

__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)(((col >> 3) ^ (row & 7)) & 7) << 4) +
         (uint32_t)(col & 7) * 2u;
}
__device__ __forceinline__ float bfv(uint32_t x16) { return __uint_as_float(x16 << 16); }
// the hardware base-2 exponential and logarithm (one MUFU operation each;
// results below the normal range flush to zero)
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
// hi and lo bf16 halves of a pair of fp32 values, packed (lower index low)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = bf2_bits(a, b);
  lo = bf2_bits(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}

template <bool kAllOut>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, PrefillTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[20];  // 9 is unused
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_tok;
  __shared__ float s_scan[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int hk = h / (p.H / p.Hk);
  const int n_chunks = 2 * p.n_pairs;
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  float* As = reinterpret_cast<float*>(gb + OFF_AS);
  float* Xs = reinterpret_cast<float*>(gb + OFF_XS);
  float* Ps = reinterpret_cast<float*>(gb + OFF_PS);
  // per chunk c, in buffer c & 3 (a stage's two chunks are written together)
  float* v_lg = reinterpret_cast<float*>(gb + OFF_VEC);  // [4][64] inclusive log2-decay
  float* v_g = v_lg + 4 * CH;                            // [4][64] g_i
  float* v_r = v_g + 4 * CH;                             // [4][64] g_C / g_i
  float* v_b = v_r + 4 * CH;                             // [4][64] beta_i
  float* v_gc = v_b + 4 * CH;                            // [4] g_C
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };
  auto in_full = [&](int s) { return bar(s); };
  auto in_empty = [&](int s) { return bar(2 + s); };
  const uint32_t g_full = bar(4), g_empty = bar(5), t_full = bar(6), t_empty = bar(7);
  auto lg_full = [&](int b) { return bar(16 + b); };  // decays of a chunk, buffer b = c & 3
  const uint32_t sa_ready = bar(10), z_full = bar(11), ya_ready = bar(12), d_full = bar(13),
                 da_ready = bar(14), s_full = bar(15), drain_bar = bar(8);
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(in_full(s), 1);
      tc::mbar_init(in_empty(s), 1 + kChainWarps + kTWarps);
    }
    for (int b = 0; b < 4; ++b) tc::mbar_init(lg_full(b), 2);
    tc::mbar_init(g_full, 1);
    tc::mbar_init(g_empty, kTWarps);
    tc::mbar_init(t_full, kTWarps);
    tc::mbar_init(t_empty, 1);
    tc::mbar_init(sa_ready, kChainWarps);
    tc::mbar_init(z_full, 1);
    tc::mbar_init(ya_ready, kChainWarps);
    tc::mbar_init(d_full, 1);
    tc::mbar_init(da_ready, kChainWarps);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(drain_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tm_k);
    tc::tma_prefetch(&tm_v);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    if (lane == 0) {
      int issued = 0;
      for (int pr = 0; pr < p.n_pairs; ++pr) {
        const int s = pr & 1;
        if (!tc::mbar_wait_sleep(in_empty(s), ((uint32_t)(pr >> 1) & 1u) ^ 1u, abort, p.err)) break;
        const uint32_t st = base + OFF_IN + (uint32_t)(s * IN_BYTES);
        tc::mbar_arrive_expect_tx(in_full(s), (uint32_t)IN_BYTES);
        for (int kb = 0; kb < 2; ++kb) {
          tc::tma_load_3d(st + kb * KBLK, &tm_k, hk * DH + kb * 64, pr * PAIR, r, in_full(s));
          tc::tma_load_3d(st + (2 + kb) * KBLK, &tm_v, h * DH + kb * 64, pr * PAIR, r, in_full(s));
        }
        issued = pr + 1;
      }
      // the last (up to two) loads issued land before the block exits
      for (int pr = issued - 2 > 0 ? issued - 2 : 0; pr < issued; ++pr)
        tc::mbar_wait_drain(in_full(pr & 1), (uint32_t)(pr >> 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t id64 = tc::idesc_bf16_f32(128, 64);
      constexpr uint32_t id128 = tc::idesc_bf16_f32(128, 128);
      int g_next = 0;  // next stage whose Gram matrix is to be formed
      // Forms K K^T of stages up to `limit`; blocking waits for the inputs,
      // or only if they are already there. False on a failed wait.
      auto issue_g = [&](int limit, bool block) -> bool {
        while (g_next < p.n_pairs && g_next <= limit) {
          const int s = g_next & 1;
          const uint32_t pin = (uint32_t)(g_next >> 1) & 1u;
          const uint32_t pge = (uint32_t)(g_next - 1) & 1u;
          if (block) {
            if (!tc::mbar_wait_sleep(in_full(s), pin, abort, p.err)) return false;
            if (g_next > 0 && !tc::mbar_wait_sleep(g_empty, pge, abort, p.err)) return false;
          } else {
            if (!tc::mbar_try_wait(in_full(s), pin)) return true;
            if (g_next > 0 && !tc::mbar_try_wait(g_empty, pge)) return true;
          }
          tc::fence_after_sync();
          const uint32_t st = base + OFF_IN + (uint32_t)(s * IN_BYTES);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t d = tc::sw128_desc(st + kb * KBLK) + 2u * kk;
              tc::mma_bf16(tmem + cG, d, d, id128, (kb | kk) != 0);
            }
          tc::mma_commit(g_full);
          ++g_next;
        }
        return true;
      };
      for (int c = 0; c < n_chunks; ++c) {
        const int pr = c >> 1, h2 = c & 1, s = pr & 1;
        const uint32_t pc = (uint32_t)c & 1u;
        if (h2 == 0 && !issue_g(pr, true)) break;
        if (!tc::mbar_wait_sleep(sa_ready, pc, abort, p.err)) break;
        tc::fence_after_sync();
        const uint32_t st = base + OFF_IN + (uint32_t)(s * IN_BYTES);
        // MMA1: Z^T = S0 K^T (B: this chunk's 64 key rows)
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = tc::sw128_desc(st + kb * KBLK + h2 * (CH * 128)) + 2u * kk;
            const uint32_t col = (uint32_t)(kb * 32 + kk * 8);
            tc::mma_bf16_ts(tmem + cZD, tmem + cSAHI + col, bd, id64, (kb | kk) != 0);
            tc::mma_bf16_ts(tmem + cZD, tmem + cSALO + col, bd, id64, 1u);
          }
        tc::mma_commit(z_full);
        if (h2 == 1) tc::mma_commit(in_empty(s));  // the stage's keys are read
        if (!issue_g(pr + 1, false)) break;
        if (!tc::mbar_wait_sleep(ya_ready, pc, abort, p.err)) break;
        if (!tc::mbar_wait_sleep(t_full, pc, abort, p.err)) break;
        tc::fence_after_sync();
        // MMA2: delta^T = Y^T T^T (three hi/lo products)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bh = tc::sw128_desc(base + OFF_THI) + 2u * kk;
          const uint64_t bl = tc::sw128_desc(base + OFF_TLO) + 2u * kk;
          const uint32_t col = (uint32_t)(kk * 8);
          tc::mma_bf16_ts(tmem + cZD, tmem + cYAHI + col, bh, id64, kk != 0);
          tc::mma_bf16_ts(tmem + cZD, tmem + cYALO + col, bh, id64, 1u);
          tc::mma_bf16_ts(tmem + cZD, tmem + cYAHI + col, bl, id64, 1u);
        }
        tc::mma_commit(d_full);
        if (!issue_g(pr + 1, false)) break;
        if (!tc::mbar_wait_sleep(da_ready, pc, abort, p.err)) break;
        tc::fence_after_sync();
        // MMA3: S += (r delta)^T K (B: K^T of the chunk); S was scaled by g_C
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = tc::sw128_desc(base + OFF_KT) + 2u * kk;
          const uint32_t col = (uint32_t)(kk * 8);
          tc::mma_bf16_ts(tmem + cSACC, tmem + cYAHI + col, bd, id128, (c > 0 || kk > 0));
          tc::mma_bf16_ts(tmem + cSACC, tmem + cYALO + col, bd, id128, 1u);
        }
        tc::mma_commit(s_full);
        tc::mma_commit(t_empty);
        if (!issue_g(pr + 1, false)) break;
      }
      tc::mma_commit(drain_bar);
      tc::mbar_wait_drain(drain_bar, 0);
    }
  } else if (warp < kT0) {
    // ------------------------------------------------------------------ chain
    const int lgp = warp & 3;
    const int v = 32 * lgp + lane;  // value row = TMEM lane
    const uint32_t lb = tmem + ((uint32_t)(32 * lgp) << 16);
    auto wait = [&](uint32_t b, uint32_t ph) -> bool {
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_sleep(b, ph, abort, p.err) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int pr = c >> 1, h2 = c & 1, s = pr & 1, b = c & 3;
      const uint32_t pc = (uint32_t)c & 1u;
      if (!(ok = wait(lg_full(b), (uint32_t)(c >> 2) & 1u))) break;
      // S0 of this chunk -> hi/lo A operand; S <- g_C S0
      if (c == 0) {
        uint32_t z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tc::tmem_st16(lb + cSAHI + 16 * q, z);
          tc::tmem_st16(lb + cSALO + 16 * q, z);
        }
      } else {
        if (!(ok = wait(s_full, (uint32_t)(c - 1) & 1u))) break;
        tc::fence_after_sync();
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
          uint32_t x[2][32];
          tc::tmem_ld32_nowait(lb + cSACC + 32 * q, x[0]);
          tc::tmem_ld32_nowait(lb + cSACC + 32 * q + 32, x[1]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              split2(__uint_as_float(x[u][2 * e]), __uint_as_float(x[u][2 * e + 1]), hi[e], lo[e]);
            tc::tmem_st16(lb + cSAHI + 16 * (q + u), hi);
            tc::tmem_st16(lb + cSALO + 16 * (q + u), lo);
            if (kAllOut) {  // the chunk's start state, row v
              float4* dst = reinterpret_cast<float4*>(
                  p.s0_out + (((size_t)blockIdx.x * n_chunks + c) * DH + v) * DH + 32 * (q + u));
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(x[u][4 * e]), __uint_as_float(x[u][4 * e + 1]),
                                     __uint_as_float(x[u][4 * e + 2]), __uint_as_float(x[u][4 * e + 3]));
            }
          }
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sa_ready);
      // S <- g_C S0 while MMA1 runs (MMA3 accumulates onto it; its issue
      // waits for this warp's da_ready, after these stores complete)
      if (c > 0) {
        const float gc = v_gc[b];
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t x[32];
          tc::tmem_ld32_nowait(lb + cSACC + 32 * q, x);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __float_as_uint(gc * __uint_as_float(x[e]));
          tc::tmem_st32(lb + cSACC + 32 * q, x);
        }
      }

      // Y^T[v][i] = v_i[v] - g_i Z^T[v][i]
      if (h2 == 0 && !(ok = wait(in_full(s), (uint32_t)(pr >> 1) & 1u))) break;
      if (!(ok = wait(z_full, pc))) break;
      tc::fence_after_sync();
      {
        const uint8_t* vs = gb + OFF_IN + s * IN_BYTES + (2 + (v >> 6)) * KBLK;
        const float* gv = v_g + b * CH;
        uint32_t z[2][32];
        tc::tmem_ld32_nowait(lb + cZD, z[0]);
        tc::tmem_ld32_nowait(lb + cZD + 32, z[1]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i0 = 32 * hf + 2 * e;
            const float v0 = bfv(*reinterpret_cast<const uint16_t*>(vs + sw128(h2 * CH + i0, v & 63)));
            const float v1 = bfv(*reinterpret_cast<const uint16_t*>(vs + sw128(h2 * CH + i0 + 1, v & 63)));
            split2(v0 - gv[i0] * __uint_as_float(z[hf][2 * e]),
                   v1 - gv[i0 + 1] * __uint_as_float(z[hf][2 * e + 1]), hi[e], lo[e]);
          }
          tc::tmem_st16(lb + cYAHI + 16 * hf, hi);
          tc::tmem_st16(lb + cYALO + 16 * hf, lo);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(ya_ready);
        if (h2 == 1) tc::mbar_arrive(in_empty(s));  // the stage's values are read
      }

      // (r delta)^T[v][i] = r_i delta^T[v][i]
      if (!(ok = wait(d_full, pc))) break;
      tc::fence_after_sync();
      {
        const float* rv = v_r + b * CH;
        uint32_t d[2][32];
        tc::tmem_ld32_nowait(lb + cZD, d[0]);
        tc::tmem_ld32_nowait(lb + cZD + 32, d[1]);
        tc::tmem_wait_ld();
        if (kAllOut) {  // the chunk's records, value row v
          const int n_tok = min(CH, p.L - c * CH);
          float* dst = p.delta_out + ((size_t)r * p.L + (size_t)c * CH) * p.H * DH + (size_t)h * DH + v;
#pragma unroll
          for (int i = 0; i < CH; ++i)
            if (i < n_tok) dst[(size_t)i * p.H * DH] = __uint_as_float(d[i >> 5][i & 31]);
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            split2(rv[32 * hf + 2 * e] * __uint_as_float(d[hf][2 * e]),
                   rv[32 * hf + 2 * e + 1] * __uint_as_float(d[hf][2 * e + 1]), hi[e], lo[e]);
          tc::tmem_st16(lb + cYAHI + 16 * hf, hi);
          tc::tmem_st16(lb + cYALO + 16 * hf, lo);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(da_ready);
    }
    // S_ctx row v and o at the last prompt token
    if (ok && wait(s_full, (uint32_t)(n_chunks - 1) & 1u)) {
      tc::fence_after_sync();
      float* out = p.sctx + (size_t)r * p.rstride + (size_t)h * DH * DH + (size_t)v * DH;
      const uint16_t* ql = p.q_last + (size_t)r * p.q_last_ld + (size_t)hk * DH;
      float o = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float x[32];
        tc::tmem_ld32(lb + cSACC + 32 * q, x);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          reinterpret_cast<float4*>(out + 32 * q)[e] =
              make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
#pragma unroll
        for (int e = 0; e < 32; ++e) o = fmaf(x[e], bfv(__ldg(ql + 32 * q + e)), o);
      }
      if (p.o_last) p.o_last[(size_t)r * p.H * DH + (size_t)h * DH + v] = __float2bfloat16_rn(o);
    }
  } else {
    // ------------------------------------------------------------------ T builders
    const int tt = threadIdx.x - 32 * kT0;  // 0 .. 255
    // one thread waits, all T builders take its outcome (they share named
    // barriers, so they must leave together)
    auto t_wait = [&](uint32_t b, uint32_t ph) -> bool {
      if (tt == 0) s_tok = tc::mbar_wait_sleep(b, ph, abort, p.err) ? 1 : 0;
      tc::named_sync(1, kTThreads);
      const bool ok = s_tok != 0;
      tc::named_sync(1, kTThreads);
      return ok;
    };
    // gates of the 128 tokens of stage pr, loaded a stage ahead (tokens
    // past the prompt: alpha = 1, beta = 0)
    auto load_gates = [&](int pr, float& a, float& be) {
      const int tok = pr * PAIR + tt;
      a = 1.f;
      be = 0.f;
      if (tt < PAIR && pr < p.n_pairs && tok < p.L) {
        const size_t idx = ((size_t)r * p.L + tok) * p.H + h;
        a = __ldg(p.alpha + idx);
        be = __ldg(p.beta + idx);
      }
    };
    float a_nx, b_nx;
    load_gates(0, a_nx, b_nx);
    for (int c = 0; c < n_chunks; ++c) {
      const int pr = c >> 1, h2 = c & 1, s = pr & 1;
      float* As_c = As + h2 * CH * XS;
      if (h2 == 0) {
        // decays of both chunks of the stage (thread = token; chunk tt >> 6):
        // inclusive log2-decay prefix, g, g_C / g, beta
        const float a_cur = a_nx, be = b_nx;
        load_gates(pr + 1, a_nx, b_nx);
        if (tt < PAIR) {
          const int hc = tt >> 6, ii = tt & 63, bb = (c + hc) & 3;
          float x = fmaxf(lg2(a_cur), -100.f);  // alpha below 2^-100 acts as 0
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          if (lane == 31) s_scan[tt >> 5] = x;
          tc::named_sync(2, PAIR);
          if (ii >= 32) x += s_scan[2 * hc];
          const float lgc = s_scan[2 * hc] + s_scan[2 * hc + 1];
          v_lg[bb * CH + ii] = x;
          v_g[bb * CH + ii] = ex2(x);
          v_r[bb * CH + ii] = ex2(lgc - x);
          v_b[bb * CH + ii] = be;
          if (ii == 0) v_gc[bb] = ex2(lgc);
          tc::named_sync(2, PAIR);  // s_scan is read before the next stage rewrites it
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(lg_full(bb));
        }
        if (!t_wait(in_full(s), (uint32_t)(pr >> 1) & 1u)) break;
        if (!t_wait(g_full, (uint32_t)pr & 1u)) break;
        // L (scaled by beta) of both chunks from the diagonal blocks of the
        // stage's K K^T: A[i][j] = beta_i (g_i / g_j) k_i.k_j for j < i.
        // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (chunk (w % 4) / 2),
        // columns of half (w - kT0) / 4 of the diagonal block.
        {
          const int lgp = warp & 3, hc = lgp >> 1, bb = (c + hc) & 3;
          const int half = (warp - kT0) >> 2;
          const int i = 32 * (lgp & 1) + lane;
          float gr[32];
          tc::tmem_ld32(tmem + ((uint32_t)(32 * lgp) << 16) + cG + 64 * hc + 32 * half, gr);
          const float lgi = v_lg[bb * CH + i], bi = v_b[bb * CH + i];
          float* Ah = As + hc * CH * XS;
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            float w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = 32 * half + 4 * e4 + u;
              w[u] = j < i ? bi * ex2(lgi - v_lg[bb * CH + j]) * gr[4 * e4 + u] : 0.f;
            }
            *reinterpret_cast<float4*>(Ah + i * XS + 32 * half + 4 * e4) =
                make_float4(w[0], w[1], w[2], w[3]);
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(g_empty);  // the stage's K K^T is read
        }
        tc::named_sync(1, kTThreads);
      }
      // X = (I + A)^-1, unit lower triangular, by 16 x 16 blocks: the four
      // diagonal blocks by forward substitution (a thread per column) ...
      if (tt < CH) {
        const int bk = tt >> 4, cc = tt & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < i; ++j) acc = fmaf(As_c[(16 * bk + i) * XS + 16 * bk + j], x[j], acc);
          x[i] = i == cc ? 1.f : (i < cc ? 0.f : -acc);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Xs[(16 * bk + i) * XS + 16 * bk + cc] = x[i];
      }
      tc::named_sync(1, kTThreads);
      // ... then the blocks below the diagonal, one sub-diagonal at a time:
      // X[bi][bj] = -X[bi][bi] sum_{bj <= k < bi} A[bi][k] X[k][bj]
      // (each thread a strip of four columns)
      auto fma4 = [](float s, const float4 x, float4& acc) {
        acc.x = fmaf(s, x.x, acc.x); acc.y = fmaf(s, x.y, acc.y);
        acc.z = fmaf(s, x.z, acc.z); acc.w = fmaf(s, x.w, acc.w);
      };
      for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;
        const int o = tt;
        const int qb = o >> 6, a = (o >> 2) & 15, b4 = (o & 3) * 4;
        const int bj = qb, bi = qb + d;
        if (o < nblk * 64) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int kb = bj; kb < bi; ++kb) {
            const float* arow = As_c + (16 * bi + a) * XS + 16 * kb;
            const float* xcol = Xs + (16 * kb) * XS + 16 * bj + b4;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 av = *reinterpret_cast<const float4*>(arow + 4 * e4);
              fma4(av.x, *reinterpret_cast<const float4*>(xcol + (4 * e4 + 0) * XS), acc);
              fma4(av.y, *reinterpret_cast<const float4*>(xcol + (4 * e4 + 1) * XS), acc);
              fma4(av.z, *reinterpret_cast<const float4*>(xcol + (4 * e4 + 2) * XS), acc);
              fma4(av.w, *reinterpret_cast<const float4*>(xcol + (4 * e4 + 3) * XS), acc);
            }
          }
          *reinterpret_cast<float4*>(Ps + (qb * 16 + a) * PS + b4) = acc;
        }
        tc::named_sync(1, kTThreads);
        if (o < nblk * 64) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          const float* xrow = Xs + (16 * bi + a) * XS + 16 * bi;
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 xv = *reinterpret_cast<const float4*>(xrow + 4 * e4);
            fma4(xv.x, *reinterpret_cast<const float4*>(Ps + (qb * 16 + 4 * e4 + 0) * PS + b4), acc);
            fma4(xv.y, *reinterpret_cast<const float4*>(Ps + (qb * 16 + 4 * e4 + 1) * PS + b4), acc);
            fma4(xv.z, *reinterpret_cast<const float4*>(Ps + (qb * 16 + 4 * e4 + 2) * PS + b4), acc);
            fma4(xv.w, *reinterpret_cast<const float4*>(Ps + (qb * 16 + 4 * e4 + 3) * PS + b4), acc);
          }
          *reinterpret_cast<float4*>(Xs + (16 * bi + a) * XS + 16 * bj + b4) =
              make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        tc::named_sync(1, kTThreads);
      }
      // the previous chunk's MMAs are done with T and K^T
      if (c > 0 && !t_wait(t_empty, (uint32_t)(c - 1) & 1u)) break;
      // K^T of the chunk: [128 k][64 i], from the stage's key rows
      {
        const uint8_t* ks = gb + OFF_IN + s * IN_BYTES;
        uint8_t* kt = gb + OFF_KT;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int item = tt + kTThreads * it;
          const int k = item & 127, ic = item >> 7;
          const uint8_t* src = ks + (k >> 6) * KBLK;
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i0 = h2 * CH + ic * 8 + 2 * e;
            const uint32_t lo16 = *reinterpret_cast<const uint16_t*>(src + sw128(i0, k & 63));
            const uint32_t hi16 = *reinterpret_cast<const uint16_t*>(src + sw128(i0 + 1, k & 63));
            w4[e] = lo16 | (hi16 << 16);
          }
          *reinterpret_cast<uint4*>(kt + sw128(k, ic * 8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      // T = X diag(beta) as hi/lo: [64 i][64 m]
      {
        uint8_t* th = gb + OFF_THI;
        uint8_t* tl = gb + OFF_TLO;
        const float* bv = v_b + (c & 3) * CH;
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const int item = tt + kTThreads * it;
          const int i = item & 63, mc = item >> 6;
          uint32_t hw[4], lw[4];
          const float4 x0 = *reinterpret_cast<const float4*>(Xs + i * XS + mc * 8);
          const float4 x1 = *reinterpret_cast<const float4*>(Xs + i * XS + mc * 8 + 4);
          const float xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m0 = mc * 8 + 2 * e;
            const float t0 = m0 <= i ? xr[2 * e] * bv[m0] : 0.f;
            const float t1 = m0 + 1 <= i ? xr[2 * e + 1] * bv[m0 + 1] : 0.f;
            split2(t0, t1, hw[e], lw[e]);
          }
          *reinterpret_cast<uint4*>(th + sw128(i, mc * 8)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(tl + sw128(i, mc * 8)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(t_full);
        if (h2 == 1) tc::mbar_arrive(in_empty(s));  // the stage's keys are copied
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = (EncodeTiledFn)ptr;
  }
  return fn;
}

}  // namespace

// [R][L][width] bf16 rows as a 3-D map with a [64 columns][box_rows rows]
// box, 128-byte swizzled; rows past L read as zeros.
bool prefill_rows_map(CUtensorMap* map, const void* ptr, int R, int L, int width, int box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn || ((uintptr_t)ptr & 15) != 0 || (width * 2) % 16 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)L, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)L * width * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 residual stream [R][L][width] as a 3-D map with [128 columns][64
// rows] boxes, unswizzled; rows past L read as zeros.
bool prefill_stream_map(CUtensorMap* map, const float* x, int R, int L, int width) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn || ((uintptr_t)x & 15) != 0 || (width * 4) % 16 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)L, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)width * 4, (cuuint64_t)L * width * 4};
  cuuint32_t box[3] = {128, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_prefill_supported(const gdnbeam_config& c) {
  return c.dtype == GDNBEAM_BF16 && c.d_k == DH && c.d_v == DH;
}

int launch_prefill_tc(const gdnbeam_config& c, int L, const void* q_last, long long q_last_ld,
                      const void* k, const void* v, const float* alpha, const float* beta,
                      float* sctx, long long rstride, void* o_last, cudaStream_t s,
                      float* s0_out, float* delta_out) {
  if (L <= 0) return GDNBEAM_EINVAL;
  const int Hk = key_heads(c);
  if ((long long)c.R * L > 0x7FFFFFFFLL) return GDNBEAM_EUNSUPPORTED;
  if ((s0_out == nullptr) != (delta_out == nullptr)) return GDNBEAM_EINVAL;
  CUtensorMap mk, mv;
  if (!prefill_rows_map(&mk, k, c.R, L, Hk * DH, PAIR) || !prefill_rows_map(&mv, v, c.R, L, c.H * DH, PAIR))
    return GDNBEAM_ECUDA;
  PrefillTcParams p{};
  p.R = c.R; p.H = c.H; p.Hk = Hk; p.L = L;
  p.n_pairs = (L + PAIR - 1) / PAIR;
  p.alpha = alpha; p.beta = beta;
  p.q_last = reinterpret_cast<const uint16_t*>(q_last);
  p.q_last_ld = q_last_ld;
  p.sctx = sctx; p.rstride = rstride;
  p.o_last = reinterpret_cast<__nv_bfloat16*>(o_last);
  p.s0_out = s0_out; p.delta_out = delta_out;
  p.err = error_word();
  if (s0_out) {
    GDN_CUDA(cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kDynSmem));
    prefill_tc_kernel<true><<<c.R * c.H, kThreads, kDynSmem, s>>>(mk, mv, p);
  } else {
    GDN_CUDA(cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kDynSmem));
    prefill_tc_kernel<false><<<c.R * c.H, kThreads, kDynSmem, s>>>(mk, mv, p);
  }
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
