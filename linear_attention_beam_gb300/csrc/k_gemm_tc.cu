// tcgen05 tensor-core GEMMs for the two dense contractions of a decode call:
//   * projections  P = U . W_proj^T  (q, k, v, decay and write gates), with
//     the per-head L2 normalisation of q and k and the gate functions fused
//     into the epilogue (OneLA §1.2 eq. 3 inputs);
//   * codebook logits Z = F . W_o^T, with the bf16 store of z and per-tile
//     (max, sum exp) partials of the row log-normaliser fused in.
//
// Persistent CTAs in clusters of two, one CTA per SM, 192 (projections) or
// 320 (logits) threads in three roles. The two CTAs of a cluster take vertically adjacent tiles (m, n) and
// (m + 1, n) in lockstep and share the B tile: each loads its own A tile and
// one 128-row half of B, multicast into both CTAs, so B leaves L2 once per
// pair of tiles.
//   warp 0      one thread issues TMA tile loads (A 128x64, B 2 x 128x64 bf16,
//               128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      owns the TMEM allocation (2 x 256 fp32 columns) and one thread
//               issues tcgen05.mma (M=128, N=256, K=16) into the accumulator
//               of the current tile, committing each stage back to the
//               producers of both CTAs and each finished tile to the epilogue;
//   warps 2-5   read the accumulator rows out of TMEM (lane = tile row) and
//   (2-9)       run the fused epilogue while the next tile accumulates into
//               the other TMEM buffer. Each epilogue warp writes its bf16
//               outputs 32 rows x 64 columns at a time into its own
//               128-byte-swizzled staging buffer and stores the box by TMA,
//               so global writes go out as whole rows, not one 16-byte piece
//               of 32 different rows per instruction.
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

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int CLUSTER = 2;  // CTAs sharing a B tile
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kNumBars = 2 * STAGES + 4 + 1;

enum { EPI_LOGITS = 0, EPI_PROJ = 1 };

// Epilogue warps: one per TMEM lane group for the projections, whose
// epilogue hides under the tile's MMAs; two for the logits, each taking half
// the columns, since 256 exponentials per row outlast the MMAs of a short-K
// tile (d_model = 1024).
template <int EPI> struct Epi {
  static constexpr int kWarps = EPI == EPI_LOGITS ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kWarps;
  // one epilogue warp's staging box: 32 rows x 32 bf16 (64-byte rows) for the
  // logits, whose eight warps must fit beside the operand ring; 32 rows x 64
  // bf16 (128-byte rows) for the projections
  static constexpr int kBoxCols = EPI == EPI_LOGITS ? 32 : 64;
  static constexpr int kStgBytes = 32 * kBoxCols * 2;
  // operand ring, the epilogue warps' staging boxes, barriers
  static constexpr size_t kSmemBytes =
      (size_t)STAGES * STAGE_BYTES + (size_t)kWarps * kStgBytes + 1024 + kNumBars * 8 + 16;
};
// dynamic plus static shared memory (the logits pair partials, 2 KiB) per block
static_assert(Epi<EPI_LOGITS>::kSmemBytes + 2048 <= 232448, "shared memory of the logits GEMM");
static_assert(Epi<EPI_PROJ>::kSmemBytes + 2048 <= 232448, "shared memory of the projection GEMM");

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

// 32 fp32 values of this lane's row as bf16 into a 32-column staging box
// (row = lane; 64-byte swizzle).
__device__ __forceinline__ void stage_bf16x32_sw64(uint8_t* stg, int lane, const float (&v)[32]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[w * 8 + 2 * j], v[w * 8 + 2 * j + 1]);
      p[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(stg + sw64_off(lane, w)) = make_uint4(p[0], p[1], p[2], p[3]);
  }
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

// Waits until this warp's previous box store has read its staging buffer.
__device__ __forceinline__ void staging_free(int lane) {
  if (lane == 0) tc::bulk_wait_read<0>();
  __syncwarp();
}

// Sends the warp's staged box to (x, y) of the map.
__device__ __forceinline__ void staging_store(const CUtensorMap* map, int x, int y, uint32_t stg_s,
                                              int lane) {
  tc::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tc::tma_store_2d(map, x, y, stg_s);
    tc::bulk_commit();
  }
}

// Logits epilogue for one tile row and one half of the tile's columns: bf16
// z (staged, stored by TMA in boxes of 32 columns), optional fp32 dump, and
// the half row's (max, sum exp), returned. y0: first row of the warp's 32.
__device__ __forceinline__ float2 epi_logits(const EpiArgs& ea, const CUtensorMap* tmz, uint32_t taddr,
                                             uint8_t* stg, uint32_t stg_s, int lane, int m, int y0,
                                             int n0, int half) {
  float run_max = -INFINITY, run_sum = 0.0f;
  const bool row_ok = m < ea.M;
#pragma unroll 1
  for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
    const int n = n0 + c * 32;
    if (n >= ea.N) break;  // warp-uniform
    staging_free(lane);
    float v[32];
    tc::tmem_ld32(taddr + c * 32, v);
    stage_bf16x32_sw64(stg, lane, v);
    staging_store(tmz, n, y0, stg_s, lane);  // rows past M, columns past N are not written
    {
      if (!row_ok) continue;
      if (ea.z_dump) {
        const size_t off = (size_t)m * ea.N + n;
        if (n + 32 <= ea.N) {
          store_f32x32(ea.z_dump + off, v);
        } else {
          for (int j = 0; j < 32 && n + j < ea.N; ++j) ea.z_dump[off + j] = v[j];
        }
      }
      const int cnt = min(32, ea.N - n);
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cnt) cm = fmaxf(cm, v[j]);
      const float nm = fmaxf(run_max, cm);
      float sm = run_sum * expf(run_max - nm);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cnt) sm += expf(v[j] - nm);
      run_sum = sm;
      run_max = nm;
    }
  }
  return make_float2(run_max, run_sum);
}

// Projection epilogue for one tile row and one of the tile's two heads
// (head width 128): q and k L2-normalised per head, v as is (bf16, staged
// and stored by TMA in boxes of 64 columns), the gates in fp32. y0: first
// row of the warp's 32; tmq, tmk, tmv: the outputs' maps.
__device__ __forceinline__ void epi_proj(const EpiArgs& ea, const CUtensorMap* tmq,
                                         const CUtensorMap* tmk, const CUtensorMap* tmv,
                                         uint32_t taddr, uint8_t* stg, uint32_t stg_s, int lane,
                                         int m, int y0, int n0, int g) {
  const int H = ea.H, Hk = ea.Hk, D = 128;
  const bool row_ok = m < ea.M;
  const int q_end = Hk * D, k_end = 2 * Hk * D, v_end = k_end + H * D;
  {
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
        staging_free(lane);
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * bx + cc;
          float v[32];
          tc::tmem_ld32(ta + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= inv;
          stage_bf16x32(stg, lane, 32 * cc, v);
          if (row_ok && dmp) store_f32x32(dmp + off + c * 32, v);
        }
        staging_store(is_q ? tmq : tmk, head * D + bx * 64, y0, stg_s, lane);
      }
    } else if (col0 < v_end) {
      const int head = (col0 - k_end) / D;
      const size_t off = (size_t)m * H * D + (size_t)head * D;
#pragma unroll 1
      for (int bx = 0; bx < 2; ++bx) {
        staging_free(lane);
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * bx + cc;
          float v[32];
          tc::tmem_ld32(ta + c * 32, v);
          stage_bf16x32(stg, lane, 32 * cc, v);
          if (row_ok && ea.dv) store_f32x32(ea.dv + off + c * 32, v);
        }
        staging_store(tmv, head * D + bx * 64, y0, stg_s, lane);
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
}

template <int EPI>
__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(Epi<EPI>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                   const __grid_constant__ CUtensorMap tmC2, EpiArgs ea) {
  // output maps: logits z (C0); projections q (C0), k (C1), v (C2)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t stg0 = base + STAGES * STAGE_BYTES;  // epilogue warps' staging boxes
  const uint32_t bar0 = stg0 + Epi<EPI>::kWarps * Epi<EPI>::kStgBytes;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + kNumBars * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto sA = [&](int s) { return base + (uint32_t)s * STAGE_BYTES; };
  auto sB = [&](int s) { return base + (uint32_t)s * STAGE_BYTES + A_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (ea.M + BM - 1) / BM, n_tiles = (ea.N + BN - 1) / BN;
  // pair tiles: rows 2 mp and 2 mp + 1 (the second may lie past M: its A
  // box reads zeros and its rows are not stored) against one B tile
  const int num_tiles = ((m_tiles + 1) / 2) * n_tiles;
  const int k_blocks = (ea.K + BK - 1) / BK;
  const int rank = (int)tc::cluster_ctarank();
  const int cid = blockIdx.x / CLUSTER, n_clusters = gridDim.x / CLUSTER;
  const uint16_t both = (uint16_t)((1u << CLUSTER) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), CLUSTER);  // the MMA commits of both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull(a), 1);
      tc::mbar_init(tempty(a), Epi<EPI>::kWarps);
    }
    tc::mbar_init(drain_bar, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tmA);
    tc::tma_prefetch(&tmB);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  // the peer's barriers are initialised before any copy or commit reaches them
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false;
      bool ok = true;
      for (int tile = cid; tile < num_tiles && ok; tile += n_clusters) {
        const int m0 = (2 * (tile / n_tiles) + rank) * BM, n0 = (tile % n_tiles) * BN;
        for (int kb = 0; kb < k_blocks; ++kb) {
          // the stage is free in both CTAs (the peer's half of B lands here too)
          if (!tc::mbar_wait(empty(s), ph ^ 1u, abort, ea.err)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(full(s), STAGE_BYTES);
          tc::tma_load_2d(sA(s), &tmA, kb * BK, m0, full(s));
          tc::tma_load_2d_mc(sB(s) + rank * (BN / 2) * 128, &tmB, kb * BK, n0 + rank * (BN / 2),
                             full(s), both);
          issued[s] = true;
          issued_phase[s] = ph;
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      // every copy this thread started has landed before the CTA can exit
      for (int i = 0; i < STAGES; ++i)
        if (issued[i]) tc::mbar_wait_drain(full(i), issued_phase[i]);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_full = tc::idesc_bf16_f32(BM, BN);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int i = 0;
      for (int tile = cid; tile < num_tiles && ok; tile += n_clusters, ++i) {
        // a last column tile narrower than BN runs MMAs only as wide as its
        // columns (rounded up to 16); the epilogues never read past N
        const int n_here = ea.N - (tile % n_tiles) * BN;
        const uint32_t idesc =
            n_here >= BN ? idesc_full : tc::idesc_bf16_f32(BM, (n_here + 15) & ~15);
        const int acc = i & 1;
        const uint32_t aph = (uint32_t)(i >> 1) & 1u;
        if (!tc::mbar_wait(tempty(acc), aph ^ 1u, abort, ea.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!tc::mbar_wait(full(s), ph, abort, ea.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t ad = tc::sw128_desc(sA(s)), bd = tc::sw128_desc(sB(s));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0);
          tc::mma_commit_mc(empty(s), both);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (ok) tc::mma_commit(tfull(acc));
      }
      // every MMA this thread issued has finished before TMEM is released
      tc::mma_commit(drain_bar);
      tc::mbar_wait_drain(drain_bar, 0);
    }
  } else {
    // one or two warps per TMEM lane group (lanes 32*lane_grp .. +31); with
    // two, each takes half the tile's columns and the pair meets at named
    // barrier 1 + lane_grp
    constexpr bool kPairs = Epi<EPI>::kWarps == 8;
    const int lane_grp = warp & 3;
    const int half = (warp - 2) >> 2;
    const int pair_bar = 1 + lane_grp;
    const int row = lane_grp * 32 + lane;
    const uint32_t stg_s = stg0 + (uint32_t)(warp - 2) * Epi<EPI>::kStgBytes;
    uint8_t* stg = gbase + (stg_s - base);
    __shared__ float2 s_half[2][4][32];  // the second half's row partials, per accumulator
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
      const int m_tile = 2 * (tile / n_tiles) + rank, n_tile = tile % n_tiles;
      const uint32_t taddr = tmem_base + ((uint32_t)(lane_grp * 32) << 16) + (uint32_t)(acc * BN);
      const int m = m_tile * BM + row;
      const int y0 = m_tile * BM + lane_grp * 32;
      if (EPI == EPI_LOGITS) {
        const float2 pr = epi_logits(ea, &tmC0, taddr, stg, stg_s, lane, m, y0, n_tile * BN, half);
        if (half) s_half[acc][lane_grp][lane] = pr;
        tc::named_sync(pair_bar, 64);
        if (!half && m < ea.M) {
          // merge the halves' (max, sum exp); an empty half has max -inf
          const float2 q = s_half[acc][lane_grp][lane];
          const float nm = fmaxf(pr.x, q.x);
          const float sum = (pr.x == -INFINITY ? 0.0f : pr.y * expf(pr.x - nm)) +
                            (q.x == -INFINITY ? 0.0f : q.y * expf(q.x - nm));
          ea.part[(size_t)m * n_tiles + n_tile] = make_float2(nm, sum);
        }
      } else {
        for (int g = 0; g < BN / 128; ++g)
          epi_proj(ea, &tmC0, &tmC1, &tmC2, taddr, stg, stg_s, lane, m, y0, n_tile * BN, g);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tempty(acc));
    }
    // the warp's box stores have finished before the CTA leaves
    if (lane == 0) tc::bulk_wait_all();
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  // neither CTA leaves while the other may still multicast into it or
  // arrive on its barriers
  tc::cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, kTmemCols);
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
  const int pair_tiles = ((ea.M + BM - 1) / BM + 1) / 2 * ((ea.N + BN - 1) / BN);
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
