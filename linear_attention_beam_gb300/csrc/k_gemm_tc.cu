// tcgen05 tensor-core GEMMs for the two dense contractions of a decode call:
//   * projections  P = U . W_proj^T  (q, k, v, decay and write gates), with
//     the per-head L2 normalisation of q and k and the gate functions fused
//     into the epilogue (OneLA §1.2 eq. 3 inputs);
//   * codebook logits Z = F . W_o^T, with the bf16 store of z and per-tile
//     (max, sum exp) partials of the row log-normaliser fused in.
//
// Persistent CTA pairs: clusters of two CTAs on two SMs, one CTA per SM,
// run one MMA of M = 256 rows x N = 256 columns per tile
// (tcgen05.mma.cta_group::2). Each CTA stages its own 128 rows of A and its
// own half (128 rows) of the B tile, so a pipeline stage is 32 KB per SM
// instead of 48 KB for a one-CTA 128 x 256 tile, B leaves L2 once per 256
// rows, and the ring holds five or six stages. Roles, 192 (projections) or
// 320 (logits) threads per CTA:
//   warp 0      one thread per CTA issues the TMA loads of that CTA's A and
//               B boxes (128 x 64 bf16, 128-byte swizzle); both CTAs' copies
//               complete on the leader CTA's stage barrier;
//   warp 1      allocates the pair's tensor memory (2 x 256 fp32 columns in
//               each CTA); in the leader CTA one thread issues the pair MMAs
//               (K = 16 each) and commits every stage back to both
//               producers and every finished tile to both CTAs' epilogues;
//   warps 2-5   read this CTA's 128 accumulator rows out of TMEM (lane = tile
//   (2-9)       row) and run the fused epilogue while the next tile
//               accumulates into the other TMEM buffer, then release the
//               buffer on the leader's barrier. Each epilogue warp writes its
//               bf16 outputs 32 rows at a time into its own 128- or 64-byte-
//               swizzled staging boxes (two, used in turn) and stores each
//               box by TMA, so global writes go out as whole rows and a box
//               is refilled while the previous one is still being stored.
// Every mbarrier wait is bounded in time; on a time-out the kernel raises
// GDNBEAM_DERR_TIMEOUT, all roles leave their loops, in-flight copies and
// MMAs are drained (again with a bound) and TMEM is freed.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int BM = 128;  // accumulator rows per CTA; the pair's MMA has M = 2 * BM
constexpr int BN = 256;  // columns per tile, the pair MMA's N
constexpr int BK = 64;
constexpr int CLUSTER = 2;                  // the CTA pair
constexpr int A_BYTES = BM * BK * 2;        // this CTA's A rows
constexpr int B_BYTES = (BN / 2) * BK * 2;  // this CTA's half of the B tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t kTmemCols = 2 * BN;

enum { EPI_LOGITS = 0, EPI_PROJ = 1 };

// Epilogue warps: one per TMEM lane group for the projections, whose
// epilogue hides under the tile's MMAs; two for the logits, each taking half
// the columns, since 256 exponentials per row outlast the MMAs of a short-K
// tile (d_model = 1024).
template <int EPI> struct Epi {
  static constexpr int kWarps = EPI == EPI_LOGITS ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kWarps;
  static constexpr int kStages = EPI == EPI_LOGITS ? 5 : 6;  // operand ring depth
  // one staging box: 32 rows x 32 bf16 (64-byte rows) for the logits, whose
  // eight warps must fit beside the operand ring; 32 rows x 64 bf16
  // (128-byte rows) for the projections. Two boxes per warp, used in turn.
  static constexpr int kBoxCols = EPI == EPI_LOGITS ? 32 : 64;
  static constexpr int kStgBytes = 32 * kBoxCols * 2;
  static constexpr int kStgBufs = 2;
  // the logits pairs' half-row partials, per accumulator buffer
  static constexpr int kHalfBytes = EPI == EPI_LOGITS ? 2 * 4 * 32 * 8 : 0;
  static constexpr int kNumBars = 2 * kStages + 4 + 1;
  // operand ring, staging boxes, partials, barriers, TMEM slot and abort flag
  static constexpr size_t kSmemBytes = (size_t)kStages * STAGE_BYTES +
                                       (size_t)kWarps * kStgBufs * kStgBytes + kHalfBytes + 1024 +
                                       kNumBars * 8 + 16;
};
static_assert(Epi<EPI_LOGITS>::kSmemBytes <= 232448, "shared memory of the logits GEMM");
static_assert(Epi<EPI_PROJ>::kSmemBytes <= 232448, "shared memory of the projection GEMM");

// MMA width for a column tile with n_here valid columns: the full BN, or the
// valid columns rounded up to 32 so each CTA's half of B stays a multiple of
// 16 rows. The epilogues never read past N.
__host__ __device__ __forceinline__ int mma_cols(int n_here) {
  return n_here >= BN ? BN : ((n_here + 31) & ~31);
}

struct EpiArgs {
  int M, N, K;
  unsigned* err;
  // logits
  __nv_bfloat16* z;
  float* z_dump;
  float2* part;  // [M][n_tiles] (max, sum exp(z - max))
  // projections
  int H, Hk;    // value heads, key heads
  int col_off;  // absolute projection column of GEMM column 0 (a multiple of 128)
  __nv_bfloat16 *q, *k, *v;
  float *alpha, *beta;
  float *dq, *dk, *dv, *da, *db;
};

__device__ __forceinline__ void store_f32x32(float* dst, const float (&v)[32]) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int w = 0; w < 8; ++w) d4[w] = make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
}

__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)(((col >> 3) ^ (row & 7)) & 7) << 4) +
         (uint32_t)(col & 7) * 2u;
}

// 64-byte swizzle of a [rows][32 bf16] box: the 16-byte piece c of row r sits
// at piece c ^ ((r >> 1) & 3) of the row (address bits 4-5 XOR bits 7-8).
__device__ __forceinline__ uint32_t sw64_off(int row, int piece) {
  return (uint32_t)row * 64u + ((uint32_t)((piece ^ (row >> 1)) & 3) << 4);
}

// 32 fp32 values of this lane's row as bf16 into columns col0 .. col0+31 of
// a 64-column staging box (row = lane; 128-byte swizzle).
__device__ __forceinline__ void stage_bf16x32(uint8_t* stg, int lane, int col0, const float (&v)[32]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[w * 8 + 2 * j], v[w * 8 + 2 * j + 1]);
      p[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(stg + sw128_off(lane, col0 + 8 * w)) = make_uint4(p[0], p[1], p[2], p[3]);
  }
}

// One epilogue warp's staging boxes in shared memory, filled and stored by
// TMA in turn. acquire() waits until the box about to be filled has been
// read by its previous store (the most recent store may still be reading
// the other box); store() sends the filled box and moves to the next one.
template <int EPI>
struct Stager {
  uint8_t* gen;  // generic address of box 0
  uint32_t sa;   // shared-window address of box 0
  int cur;
  __device__ __forceinline__ uint8_t* acquire(int lane) {
    if (lane == 0) tc::bulk_wait_read<Epi<EPI>::kStgBufs - 1>();
    __syncwarp();
    return gen + cur * Epi<EPI>::kStgBytes;
  }
  // Rows past the map's rows and columns past its columns are not written.
  __device__ __forceinline__ void store(const CUtensorMap* map, int x, int y, int lane) {
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tc::tma_store_2d(map, x, y, sa + (uint32_t)(cur * Epi<EPI>::kStgBytes));
      tc::bulk_commit();
    }
    cur = cur + 1 == Epi<EPI>::kStgBufs ? 0 : cur + 1;
  }
};

// exp(x) for the row normaliser is evaluated as 2^(x log2 e) with the
// hardware base-2 exponential (ex2.approx, relative error about 2^-22).
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed fp32 pairs (low word = first element).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 32 fp32 values (as bits) of this lane's row as bf16 into a 32-column
// staging box (row = lane; 64-byte swizzle).
__device__ __forceinline__ void stage_bf16x32_sw64(uint8_t* stg, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[w * 8 + 2 * j]),
                                               __uint_as_float(r[w * 8 + 2 * j + 1]));
      p[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(stg + sw64_off(lane, w)) = make_uint4(p[0], p[1], p[2], p[3]);
  }
}

// Logits epilogue for one tile row and one half (128 columns) of the tile,
// from accumulator values already in registers (r[c]: the half's columns
// 32c .. 32c+31): bf16 z (staged, stored by TMA in boxes of 32 columns),
// optional fp32 dump, and the half row's (max, sum exp), returned; an empty
// half gives (-inf, 0). y0: first row of the warp's 32; nh: the half's
// first column.
__device__ __forceinline__ float2 epi_logits(const EpiArgs& ea, const CUtensorMap* tmz,
                                             const uint32_t (&r)[4][32], Stager<EPI_LOGITS>& stg,
                                             int lane, int m, int y0, int nh) {
  const int cnt = ea.N - nh;  // valid columns of the half (all 128 except in a last tile)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c * 32 < cnt) {  // warp-uniform
      uint8_t* box = stg.acquire(lane);
      stage_bf16x32_sw64(box, lane, r[c]);
      stg.store(tmz, nh + c * 32, y0, lane);
    }
  }
  if (m >= ea.M || cnt <= 0) return make_float2(-INFINITY, 0.0f);
  if (ea.z_dump) {
    float* d = ea.z_dump + (size_t)m * ea.N + nh;
    for (int c = 0; c < 4; ++c)
      for (int j = 0; j < 32; ++j)
        if (c * 32 + j < cnt) d[c * 32 + j] = __uint_as_float(r[c][j]);
  }
  float mx = -INFINITY;
  if (cnt >= 128) {
    // max by three-input compares; then sum 2^(log2e (v - max)) with packed
    // fp32 pairs: one FMA and one add per two columns, one ex2 per column
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        mx = fmax3(mx, __uint_as_float(r[c][j]), __uint_as_float(r[c][j + 1]));
    const float nb = -mx * kLog2e;
    const uint64_t l2 = pack2(kLog2e, kLog2e), nb2 = pack2(nb, nb);
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const uint64_t t = fma2(((uint64_t)r[c][j + 1] << 32) | r[c][j], l2, nb2);
        acc[c] = add2(acc[c], pack2(ex2(__uint_as_float((uint32_t)t)),
                                    ex2(__uint_as_float((uint32_t)(t >> 32)))));
      }
    const uint64_t a = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
    return make_float2(mx, __uint_as_float((uint32_t)a) + __uint_as_float((uint32_t)(a >> 32)));
  }
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c * 32 + j < cnt) mx = fmaxf(mx, __uint_as_float(r[c][j]));
    const float nb = -mx * kLog2e;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c * 32 + j < cnt) s[c] += ex2(fmaf(__uint_as_float(r[c][j]), kLog2e, nb));
  }
  return make_float2(mx, (s[0] + s[1]) + (s[2] + s[3]));
}

// Projection epilogue for one tile row and one of the tile's two heads
// (head width 128): q and k L2-normalised per head, v as is (bf16, staged
// and stored by TMA in boxes of 64 columns), the gates in fp32. y0: first
// row of the warp's 32; tmq, tmk, tmv: the outputs' maps. (Holding the
// head's 128 accumulator values in registers to read TMEM once measured
// slower than reading q and k twice.)
__device__ __forceinline__ void epi_proj(const EpiArgs& ea, const CUtensorMap* tmq,
                                         const CUtensorMap* tmk, const CUtensorMap* tmv,
                                         uint32_t taddr, Stager<EPI_PROJ>& stg, int lane,
                                         int m, int y0, int n0, int g) {
  const int H = ea.H, Hk = ea.Hk, D = 128;
  const bool row_ok = m < ea.M;
  const int q_end = Hk * D, k_end = 2 * Hk * D, v_end = k_end + H * D;
  if (n0 + g * D >= ea.N) return;
  const int col0 = n0 + g * D + ea.col_off;  // column of the full projection
  const uint32_t ta = taddr + g * D;
  if (col0 < k_end) {
    const bool is_q = col0 < q_end;
    const int head = (is_q ? col0 : col0 - q_end) / D;
    float ss = 0.0f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tc::tmem_ld32(ta + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
    }
    const float inv = 1.0f / sqrtf(ss + 1e-6f);
    float* dmp = is_q ? ea.dq : ea.dk;
    const size_t off = (size_t)m * Hk * D + (size_t)head * D;
#pragma unroll 1
    for (int bx = 0; bx < 2; ++bx) {
      uint8_t* box = stg.acquire(lane);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * bx + cc;
        float v[32];
        tc::tmem_ld32(ta + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= inv;
        stage_bf16x32(box, lane, 32 * cc, v);
        if (row_ok && dmp) store_f32x32(dmp + off + c * 32, v);
      }
      stg.store(is_q ? tmq : tmk, head * D + bx * 64, y0, lane);
    }
  } else if (col0 < v_end) {
    const int head = (col0 - k_end) / D;
    const size_t off = (size_t)m * H * D + (size_t)head * D;
#pragma unroll 1
    for (int bx = 0; bx < 2; ++bx) {
      uint8_t* box = stg.acquire(lane);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * bx + cc;
        float v[32];
        tc::tmem_ld32(ta + c * 32, v);
        stage_bf16x32(box, lane, 32 * cc, v);
        if (row_ok && ea.dv) store_f32x32(ea.dv + off + c * 32, v);
      }
      stg.store(tmv, head * D + bx * 64, y0, lane);
    }
  } else {
    // gate columns: H decay-gate logits, then H write-gate logits
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tc::tmem_ld32(ta + c * 32, v);
      if (!row_ok) continue;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int idx = c * 32 + j;
        if (idx < H) {
          const float a = decay_gate(v[j]);
          ea.alpha[(size_t)m * H + idx] = a;
          if (ea.da) ea.da[(size_t)m * H + idx] = a;
        } else if (idx < 2 * H) {
          const float b = write_gate(v[j]);
          ea.beta[(size_t)m * H + idx - H] = b;
          if (ea.db) ea.db[(size_t)m * H + idx - H] = b;
        }
      }
    }
  }
}

template <int EPI>
__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(Epi<EPI>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                   const __grid_constant__ CUtensorMap tmC2, EpiArgs ea) {
  // output maps: logits z (C0); projections q (C0), k (C1), v (C2)
  using E = Epi<EPI>;
  constexpr int S = E::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  // both CTAs of the pair lay out their shared memory identically: the
  // pair MMA reads the peer's operands at the leader's offsets
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t stg0 = base + S * STAGE_BYTES;  // epilogue warps' staging boxes
  const uint32_t half0 = stg0 + E::kWarps * E::kStgBufs * E::kStgBytes;
  const uint32_t bar0 = half0 + E::kHalfBytes;
  auto full = [&](int s_) { return bar0 + 8u * s_; };
  auto empty = [&](int s_) { return bar0 + 8u * (S + s_); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + E::kNumBars * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto sA = [&](int s_) { return base + (uint32_t)s_ * STAGE_BYTES; };
  auto sB = [&](int s_) { return base + (uint32_t)s_ * STAGE_BYTES + A_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a tile is 2 * BM rows (this CTA's BM of them start at row
  // (2 * tile_row + rank) * BM; rows past M read zeros and are not stored)
  // by BN columns
  const int m_tiles = (ea.M + 2 * BM - 1) / (2 * BM), n_tiles = (ea.N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int k_blocks = (ea.K + BK - 1) / BK;
  const uint32_t rank = tc::cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x / CLUSTER, n_clusters = gridDim.x / CLUSTER;
  constexpr uint16_t kBoth = (uint16_t)((1u << CLUSTER) - 1u);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(full(i), 1);   // leader: its producer's arrival + both CTAs' bytes
      tc::mbar_init(empty(i), 1);  // the leader's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull(a), 1);
      tc::mbar_init(tempty(a), CLUSTER * E::kWarps);  // leader: both CTAs' epilogue warps
    }
    tc::mbar_init(drain_bar, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tmA);
    tc::tma_prefetch(&tmB);
  }
  if (warp == 1) tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  // the peer's barriers are initialised before any copy, commit or arrival
  // reaches them
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int n_issued = 0;  // stage loads issued so far
      bool ok = true;
      for (int tile = cid; tile < num_tiles && ok; tile += n_clusters) {
        const int m0 = (2 * (tile / n_tiles) + (int)rank) * BM;
        const int n0 = (tile % n_tiles) * BN;
        // this CTA's half of the tile's B rows
        const int nb = n0 + (int)rank * (mma_cols(ea.N - n0) / 2);
        for (int kb = 0; kb < k_blocks; ++kb) {
          // the leader's MMAs have finished reading this stage in both CTAs
          if (!tc::mbar_wait(empty(st), ph ^ 1u, abort, ea.err)) { ok = false; break; }
          const uint32_t bar = tc::mapa_shared(full(st), 0);
          if (leader) tc::mbar_arrive_expect_tx(full(st), CLUSTER * STAGE_BYTES);
          tc::tma_load_2d_pair(sA(st), &tmA, kb * BK, m0, bar);
          tc::tma_load_2d_pair(sB(st), &tmB, kb * BK, nb, bar);
          ++n_issued;
          if (++st == S) { st = 0; ph ^= 1u; }
        }
      }
      // every copy of the pair has landed before the CTAs can exit: both
      // CTAs' copies complete on the leader's stage barriers, which its
      // producer drains (the two producers issue the same stages)
      // (the q-th load went to stage q % S in phase (q / S) & 1)
      if (leader)
        for (int q = max(0, n_issued - S); q < n_issued; ++q)
          tc::mbar_wait_drain(full(q % S), (uint32_t)(q / S) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      int i = 0;
      for (int tile = cid; tile < num_tiles && ok; tile += n_clusters, ++i) {
        // a last column tile narrower than BN runs MMAs only as wide as its
        // columns (rounded up to 32); the epilogues never read past N
        const int nm = mma_cols(ea.N - (tile % n_tiles) * BN);
        const uint32_t idesc = tc::idesc_bf16_f32(2 * BM, nm);
        const int acc = i & 1;
        const uint32_t aph = (uint32_t)(i >> 1) & 1u;
        // both CTAs' epilogues have drained this accumulator buffer
        if (!tc::mbar_wait(tempty(acc), aph ^ 1u, abort, ea.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!tc::mbar_wait(full(st), ph, abort, ea.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t ad = tc::sw128_desc(sA(st)), bd = tc::sw128_desc(sB(st));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0);
          tc::mma_commit_pair_mc(empty(st), kBoth);
          if (++st == S) { st = 0; ph ^= 1u; }
        }
        if (ok) tc::mma_commit_pair_mc(tfull(acc), kBoth);
      }
      // every MMA this thread issued has finished before TMEM is released
      tc::mma_commit_pair(drain_bar);
      tc::mbar_wait_drain(drain_bar, 0);
    }
  } else {
    // one or two warps per TMEM lane group (lanes 32*lane_grp .. +31); with
    // two, each takes half the tile's columns and the pair meets at named
    // barrier 1 + lane_grp
    constexpr bool kPairs = E::kWarps == 8;
    const int lane_grp = warp & 3;
    const int half = (warp - 2) >> 2;
    const int pair_bar = 1 + lane_grp;
    const int row = lane_grp * 32 + lane;
    const uint32_t stg_s = stg0 + (uint32_t)((warp - 2) * E::kStgBufs * E::kStgBytes);
    Stager<EPI> stg{gbase + (stg_s - base), stg_s, 0};
    // the second half's row partials, per accumulator buffer
    float2* s_half = reinterpret_cast<float2*>(gbase + (half0 - base));
    int i = 0;
    for (int tile = cid; tile < num_tiles; tile += n_clusters, ++i) {
      const int acc = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      const bool got = tc::mbar_wait(tfull(acc), aph, abort, ea.err);
      // both warps of a pair go on only if both saw the tile, so neither
      // waits at the pair barrier for a partner that left
      if (kPairs) {
        if (!tc::named_sync_and(pair_bar, 64, got)) break;
      } else {
        __syncwarp();  // the TMEM loads below are warp-collective
        if (!got) break;
      }
      tc::fence_after_sync();
      const int m_tile = 2 * (tile / n_tiles) + (int)rank, n_tile = tile % n_tiles;
      const uint32_t taddr = tmem_base + ((uint32_t)(lane_grp * 32) << 16) + (uint32_t)(acc * BN);
      const int m = m_tile * BM + row;
      const int y0 = m_tile * BM + lane_grp * 32;
      if constexpr (EPI == EPI_LOGITS) {
        // this warp's half row into registers, then the accumulator buffer
        // goes back to the MMA before the math and the stores
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32_nowait(taddr + (uint32_t)(half * 128 + c * 32), r[c]);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(tc::mapa_shared(tempty(acc), 0));
        const float2 pr = epi_logits(ea, &tmC0, r, stg, lane, m, y0, n_tile * BN + half * 128);
        float2* sh = s_half + (acc * 4 + lane_grp) * 32;
        if (half) sh[lane] = pr;
        tc::named_sync(pair_bar, 64);
        if (!half && m < ea.M) {
          // merge the halves' (max, sum exp); an empty half has max -inf
          const float2 q = sh[lane];
          const float nm = fmaxf(pr.x, q.x);
          const float sum = (pr.x == -INFINITY ? 0.0f : pr.y * expf(pr.x - nm)) +
                            (q.x == -INFINITY ? 0.0f : q.y * expf(q.x - nm));
          ea.part[(size_t)m * n_tiles + n_tile] = make_float2(nm, sum);
        }
      } else {
        for (int g = 0; g < BN / 128; ++g)
          epi_proj(ea, &tmC0, &tmC1, &tmC2, taddr, stg, lane, m, y0, n_tile * BN, g);
        // this warp's TMEM reads are done: release the buffer on the leader
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(tc::mapa_shared(tempty(acc), 0));
      }
    }
    // the warp's box stores have finished before the CTA leaves
    if (lane == 0) tc::bulk_wait_all();
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  // neither CTA leaves while the leader may still write the peer's TMEM,
  // signal its barriers or read its shared memory
  tc::cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// lse = M + log sum_i s_i exp(m_i - M) over a row's tile partials.
__global__ void lse_reduce_kernel(int n, int n_tiles, const float2* __restrict__ part,
                                  float* __restrict__ lse) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const float2* p = part + (size_t)row * n_tiles;
  float mx = -INFINITY;
  for (int i = lane; i < n_tiles; i += 32) mx = fmaxf(mx, p[i].x);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float s = 0.0f;
  for (int i = lane; i < n_tiles; i += 32) s += p[i].y * expf(p[i].x - mx);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) lse[row] = mx + logf(s);
}

// ---- host side ---------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = (EncodeTiledFn)p;
  }
  return fn;
}

// Row-major bf16 matrix [rows][cols] (rows ld elements apart; ld = 0 means
// cols) as a 2-D tensor map with a box of 64 columns x box_rows rows and
// 128-byte swizzling.
bool make_map(CUtensorMap* map, const void* ptr, int rows, int cols, int box_rows,
              long long ld = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (ld == 0) ld = cols;
  if (((uintptr_t)ptr & 15) != 0 || (ld * 2) % 16 != 0 || ld < cols) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map of a GEMM epilogue: row-major bf16 [rows][cols] with a box of
// box_cols (64: 128-byte swizzle; 32: 64-byte swizzle) x 32 rows, one
// epilogue warp's staging box.
bool make_store_map(CUtensorMap* map, const void* ptr, int rows, int cols, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !ptr || ((uintptr_t)ptr & 15) != 0 || (cols * 2) % 16 != 0) return false;
  if (box_cols != 32 && box_cols != 64) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev];
}

// Clusters of this kernel that fit on the device at once (one CTA per SM;
// a GPC with an odd number of free SMs leaves one of them out).
template <int EPI>
int max_clusters() {
  static int cached[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev][EPI]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CLUSTER * (num_sms() / CLUSTER), 1, 1);
    cfg.blockDim = dim3(Epi<EPI>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Epi<EPI>::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = CLUSTER;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<EPI>, &cfg) != cudaSuccess || n <= 0)
      n = num_sms() / CLUSTER;
    cached[dev][EPI] = n;
  }
  return cached[dev][EPI];
}

// out[i]: the epilogue's output maps (see tc_gemm_kernel); unused ones are
// left zeroed and never referenced.
template <int EPI>
int launch_gemm(const void* A, const void* B, const EpiArgs& ea, const CUtensorMap (&out)[3],
                cudaStream_t s, long long lda = 0) {
  if (ea.M <= 0) return GDNBEAM_OK;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, ea.M, ea.K, BM, lda) || !make_map(&tb, B, ea.N, ea.K, BN / 2))
    return GDNBEAM_ECUDA;
  static bool attr_set[2] = {false, false};
  if (!attr_set[EPI]) {
    GDN_CUDA(cudaFuncSetAttribute(tc_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)Epi<EPI>::kSmemBytes));
    attr_set[EPI] = true;
  }
  const int pair_tiles = (ea.M + 2 * BM - 1) / (2 * BM) * ((ea.N + BN - 1) / BN);
  int clusters = max_clusters<EPI>();
  if (clusters <= 0) return GDNBEAM_ECUDA;
  if (clusters > pair_tiles) clusters = pair_tiles;
  tc_gemm_kernel<EPI><<<CLUSTER * clusters, Epi<EPI>::kThreads, Epi<EPI>::kSmemBytes, s>>>(
      ta, tb, out[0], out[1], out[2], ea);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

bool tc_gemm_supported(const gdnbeam_config& c) {
  const int F = c.residual ? c.d_model : c.H * c.d_v;
  return c.dtype == GDNBEAM_BF16 && c.d_k == 128 && c.d_v == 128 && c.d_model % BK == 0 &&
         F % BK == 0 && c.V % 8 == 0 && 2 * c.H <= 128;
}

int launch_tc_project(const gdnbeam_config& c, int n, const void* u, const void* W_proj, void* q,
                      void* k, void* v, float* alpha, float* beta, const gdnbeam_dumps* d,
                      cudaStream_t s, int cols, long long ldu) {
  const int n_full = 2 * key_heads(c) * c.d_k + c.H * c.d_v + 2 * c.H;
  const int q_cols = key_heads(c) * c.d_k;
  EpiArgs ea{};
  ea.M = n;
  ea.K = c.d_model;
  ea.err = error_word();
  // the projection columns computed: all, all but the queries, or only them
  if (cols == PROJ_ALL) {
    ea.N = n_full;
  } else if (cols == PROJ_NO_Q) {
    ea.col_off = q_cols;
    ea.N = n_full - q_cols;
    W_proj = (const char*)W_proj + (size_t)q_cols * c.d_model * 2;
  } else if (cols == PROJ_Q_ONLY) {
    ea.N = q_cols;
  } else {
    return GDNBEAM_EINVAL;
  }
  ea.H = c.H;
  ea.Hk = key_heads(c);
  ea.q = (__nv_bfloat16*)q;
  ea.k = (__nv_bfloat16*)k;
  ea.v = (__nv_bfloat16*)v;
  ea.alpha = alpha;
  ea.beta = beta;
  if (d) {
    ea.dq = d->q; ea.dk = d->k; ea.dv = d->v; ea.da = d->alpha; ea.db = d->beta;
  }
  CUtensorMap out[3];
  memset(out, 0, sizeof(out));
  const int kw = key_heads(c) * c.d_k;
  // the maps of the outputs this call writes
  const bool want_q = cols != PROJ_NO_Q, want_kv = cols != PROJ_Q_ONLY;
  constexpr int bc = Epi<EPI_PROJ>::kBoxCols;
  if ((want_q && !make_store_map(&out[0], q, n, kw, bc)) ||
      (want_kv && (!make_store_map(&out[1], k, n, kw, bc) ||
                   !make_store_map(&out[2], v, n, c.H * c.d_v, bc))))
    return GDNBEAM_ECUDA;
  return launch_gemm<EPI_PROJ>(u, W_proj, ea, out, s, ldu);
}

size_t tc_logits_scratch_bytes(const gdnbeam_config& c, int n) {
  return (size_t)n * ((c.V + BN - 1) / BN) * sizeof(float2);
}

int launch_tc_logits(const gdnbeam_config& c, int n, const void* feat, const void* W_o, void* z,
                     float* lse, void* scratch, const gdnbeam_dumps* d, cudaStream_t s) {
  EpiArgs ea{};
  ea.M = n;
  ea.N = c.V;
  ea.err = error_word();
  ea.K = c.residual ? c.d_model : c.H * c.d_v;
  ea.z = (__nv_bfloat16*)z;
  ea.z_dump = d ? d->logits : nullptr;
  ea.part = (float2*)scratch;
  CUtensorMap out[3];
  memset(out, 0, sizeof(out));
  if (!make_store_map(&out[0], z, n, c.V, Epi<EPI_LOGITS>::kBoxCols)) return GDNBEAM_ECUDA;
  int st = launch_gemm<EPI_LOGITS>(feat, W_o, ea, out, s);
  if (st) return st;
  const int n_tiles = (c.V + BN - 1) / BN;
  lse_reduce_kernel<<<(n + 7) / 8, 256, 0, s>>>(n, n_tiles, (const float2*)scratch, lse);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}


}  // namespace gdnbeam
