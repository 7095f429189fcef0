// Fused shared-context replay on tcgen05 tensor cores (bf16; d_k 128 or 256,
// d_v a multiple of 128 up to 512). The kernel template lives here; each key
// width is instantiated in its own translation unit.
//
// OneLA §2.5: one block per (request, head) holds that head's S_ctx for the
// whole call and reuses it for every beam tile; per tile it forms the two
// projections of §2.3 eqs. 6-7 from S_ctx, folds the ancestors' records
// (alpha_j, delta_j, k_j) into them, evaluates eq. 8 and writes only delta_t
// (the new record) and o_t. No per-beam d_v x d_k state exists anywhere.
//
// Mapping to sm_103a:
//   * One block per (request, head, 128 value rows), or per range of its beam
//     tiles when those triples alone are too few to fill the SMs. Its S_ctx
//     rows (fp32 in memory) are split into bf16 hi + lo halves and kept in
//     tensor memory as the A operand (M = 128 value rows) of two MMAs per K
//     step, so the contraction keeps ~16 mantissa bits of S_ctx and shared
//     memory is left to the beam pipeline.
//   * Beams go in tiles of 32. A producer warp stages per tile, by TMA, the
//     32 queries and keys (the B operand, N = 64: q rows then k rows, 128-byte
//     swizzled) and the 32 value rows; that warp and two more gather each
//     beam's ancestor records delta_j, four rows per request. (The SM issues
//     small TMA requests at a limited rate, so the ancestor keys k_j, which
//     only the scalar warps read, are loaded by those warps directly.) Stages
//     sit on an mbarrier ring several tiles deep.
//   * Gates, ancestor slots and ancestor decays of all the block's beams are
//     read once into a shared table at block start by every thread (while
//     the epilogue warps' S_ctx loads are in flight), so no global load sits
//     on the per-tile path.
//   * One thread issues tcgen05.mma into a double-buffered TMEM accumulator:
//     column b holds u_q of beam b, column 32 + b its u_k, lane = value row.
//   * Four scalar warps compute the replay scalars k_j.q_t, k_j.k_t and
//     k_t.q_t of each tile and turn them into per-beam coefficients of the
//     fold; eight epilogue warps (thread = value row; two warps per TMEM lane
//     group, 16 beams each) fold the records, apply eq. 8 and write delta_t
//     and o_t into double-buffered shared boxes that TMA stores to memory.
//     Roles hand tiles over through mbarriers only, so warps drift freely.
// Every wait is bounded in time (GDNBEAM_DERR_TIMEOUT on expiry).
#pragma once
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int VR = 128;           // value rows per block (the MMA's M)
constexpr int NB = 32;            // beams per tile
constexpr int kEpiWarps = 8;      // two per TMEM lane group; each folds 16 beams of a tile
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kScalWarps = 4;     // replay-scalar warps, eight beams of a tile each
constexpr int kThreads = 64 + kEpiThreads + 64 + 32 * kScalWarps;  // producer, MMA, epilogue,
                                                                   // two record loaders, scalars
constexpr int kMaxDepth = 6;      // replay depths this kernel stages
constexpr int V_BYTES = NB * VR * 2;        // v rows (this block's 128 values): 8 KiB
constexpr int REC_D = NB * VR * 2;          // delta_j rows of one depth (128 values): 8 KiB
constexpr int OUT_BYTES = 2 * NB * VR * 2;  // delta_t and o_t rows of one tile: 16 KiB
constexpr int OUT_WARP = 2 * 16 * 32 * 2;   // one warp's [16 beams][32 rows] of delta_t and o_t
constexpr int kMaxStages = 6;
// per key width: q and k rows of a tile, and one depth's records (delta_j
// for this block's values, then k_j)
template <int DK> struct Width {
  static constexpr int B_BYTES = 2 * NB * DK * 2;
  static constexpr int REC_BYTES = REC_D;  // the scalar warps read k_j from global memory
  // TMEM columns: two accumulators of 2 * NB, then S_ctx hi and lo (DK / 2 each)
  static constexpr uint32_t kColAHi = 4 * NB, kColALo = 4 * NB + DK / 2;
  static constexpr uint32_t kTmemCols = DK == 128 ? 256 : 512;
};

// Ancestor records of each depth as 2-D maps [R * W_j * heads rows][width]
// with a one-row, 64-column box, read four rows at a time.
struct RecMaps {
  CUtensorMap d[kMaxDepth];
};

struct TcReplayParams {
  int R, H, Hk, dv, t, W_t, n_tiles, stages, stage_bytes;
  int tiles_per_block;  // beam tiles of one block; blockIdx.z picks the range
  int first_tiles;      // > 0: two blocks per triple, tiles [0, first_tiles) and the rest
  const float* sctx;
  long long sctx_rstride;
  const float *alpha, *beta;
  const float* rec_a[kMaxDepth];
  const uint16_t* rec_k[kMaxDepth];  // ancestor keys [R * W_j][Hk * DK] bf16
  int W_j[kMaxDepth];
  const int32_t* anc;
  int anc_stride;
  int store_o;  // 0: o_t goes only to x_inout and the dumps
  float* x_inout;
  float *delta_dump, *o_dump;
  unsigned* err;
};

// Byte offset of element (row, col) of a [rows][64] bf16 block in the
// 128-byte swizzled layout TMA writes (16-byte chunks XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)(((col >> 3) ^ (row & 7)) & 7) << 4) +
         (uint32_t)(col & 7) * 2u;
}

__device__ __forceinline__ float bf(uint32_t x16) { return __uint_as_float(x16 << 16); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Dynamic shared memory (1024-byte aligned base):
//   stages x [B: q rows | k rows per 64-column block (swizzled)]
//            [V: value rows, two [32][64] boxes]
//            [REC per depth: delta_j rows | k_j rows, each as two [32][64] halves]
//   table: (alpha_t, beta_t) per beam, then per beam and depth the ancestor
//          slot and its decay (negative for a slot outside its depth).
// EXTRA: the fp32 dumps or the residual stream are written as well.
template <int TD, bool EXTRA, int DK>  // replay depth t of this call, key width
__global__ void __launch_bounds__(kThreads, 1)
    replay_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_d,
                     const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ RecMaps rm,
                     TcReplayParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 11];
  // replay scalars of two tiles: per beam (beta_t, K0, Q0, k_t.q_t) and per
  // ancestor record (K_j, Q_j), the fold written out:
  //   delta_t = beta_t v + K0 u_k + sum_j K_j delta_j,
  //   o_t = Q0 u_q + sum_j Q_j delta_j + (k_t.q_t) delta_t
  __shared__ float4 s_beam[2][NB];
  __shared__ float2 s_rec[2][NB][TD > 0 ? TD : 1];
  // delta_t and o_t of two tiles, per epilogue warp a [16 beams][32 rows] box of each
  __shared__ __align__(1024) uint8_t s_out[2][OUT_BYTES];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  constexpr int t = TD;
  constexpr int B_BYTES = Width<DK>::B_BYTES, REC_BYTES = Width<DK>::REC_BYTES;
  constexpr uint32_t kColAHi = Width<DK>::kColAHi, kColALo = Width<DK>::kColALo;
  constexpr uint32_t kTmemCols = Width<DK>::kTmemCols;
  const int vb = blockIdx.y;   // which 128 value rows of the head
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  // this block's beam tiles: tile0 .. tile0 + nt - 1, beams bb .. bb + nbeams - 1
  int tile0, nt;
  if (p.first_tiles > 0) {
    tile0 = blockIdx.z == 0 ? 0 : p.first_tiles;
    nt = blockIdx.z == 0 ? p.first_tiles : p.n_tiles - p.first_tiles;
  } else {
    tile0 = blockIdx.z * p.tiles_per_block;
    nt = min(p.tiles_per_block, p.n_tiles - tile0);
  }
  const int bb = tile0 * NB;
  const int nbeams = min(nt * NB, p.W_t - bb);
  // the table holds this block's beams, indexed from bb
  float2* tab_ab = reinterpret_cast<float2*>(gbase + p.stages * p.stage_bytes);
  int* tab_slot = reinterpret_cast<int*>(tab_ab + p.tiles_per_block * NB);
  float* tab_aj = reinterpret_cast<float*>(tab_slot + p.tiles_per_block * NB * t);
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(kMaxStages + s); };
  auto tfull = [&](int a) { return bar(2 * kMaxStages + a); };
  auto tempty = [&](int a) { return bar(2 * kMaxStages + 2 + a); };
  auto sfull = [&](int a) { return bar(2 * kMaxStages + 4 + a); };   // scalars of a tile written
  auto sempty = [&](int a) { return bar(2 * kMaxStages + 6 + a); };  // scalars of a tile used
  const uint32_t a_ready = bar(2 * kMaxStages + 8);
  const uint32_t drain_bar = bar(2 * kMaxStages + 10);
  volatile int* abort = &s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int hk = h / (p.H / p.Hk);  // the key head this value head reads
  constexpr int v_off = B_BYTES;
  constexpr int rec_off = B_BYTES + V_BYTES;
  constexpr int kEpi0 = 2, kRec0 = 2 + kEpiWarps, kScal0 = kRec0 + 2;  // first warp of each role

  // Epilogue warps: their S_ctx row (vb * 128 + i_row, K half hb) in batches
  // of 32 values; the first batches are requested before anything else (the
  // barrier and TMEM set-up, the table), so those latencies overlap.
  const bool epi_warp = warp >= kEpi0 && warp < kEpi0 + kEpiWarps;
  const int e_hb = (warp - kEpi0) >> 2, e_row = (warp & 3) * 32 + lane;
  const float* S = p.sctx + (size_t)r * p.sctx_rstride + (size_t)h * p.dv * DK +
                   (size_t)(vb * VR + e_row) * DK + e_hb * (DK / 2);
  constexpr int kBatches = DK / 64;
  constexpr int kEarly = kBatches < 2 ? kBatches : 2;
  float4 xe[kEarly][8];
  if (epi_warp) {
#pragma unroll
    for (int bt = 0; bt < kEarly; ++bt)
#pragma unroll
      for (int c = 0; c < 8; ++c) xe[bt][c] = __ldg(reinterpret_cast<const float4*>(S) + bt * 8 + c);
  }
  // so are this thread's first beam's ancestor slots and gates (the table
  // below)
  int sl0[TD > 0 ? TD : 1];
  float2 ab0 = make_float2(0.0f, 0.0f);
  if ((int)threadIdx.x < nbeams) {
    const size_t row = (size_t)r * p.W_t + bb + threadIdx.x;
#pragma unroll
    for (int j = 0; j < t; ++j) sl0[j] = p.anc[row * p.anc_stride + j];
    ab0 = make_float2(p.alpha[row * p.H + h], p.beta[row * p.H + h]);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      tc::mbar_init(full(s), TD > 0 ? 3 : 1);  // the producer and the record loaders
      // released by the MMA commit, every epilogue warp and every scalar warp
      tc::mbar_init(empty(s), 1 + kEpiWarps + kScalWarps);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull(a), 1);
      tc::mbar_init(tempty(a), kEpiWarps);
      tc::mbar_init(sfull(a), kScalWarps);
      tc::mbar_init(sempty(a), kEpiWarps);
    }
    tc::mbar_init(a_ready, kEpiWarps);
    tc::mbar_init(drain_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tm_q); tc::tma_prefetch(&tm_k); tc::tma_prefetch(&tm_v);
    tc::tma_prefetch(&tm_d); tc::tma_prefetch(&tm_o);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = s_tmem;

  // The block's table, built by every thread (one beam each at W = 512):
  // gates, ancestor slots and decays of every beam. The slot loads go out
  // together before the dependent decay loads.
  for (int b = threadIdx.x; b < nbeams; b += kThreads) {
    const size_t row = (size_t)r * p.W_t + bb + b;
    int sl[TD > 0 ? TD : 1];
    if (b == (int)threadIdx.x) {  // requested at the top
#pragma unroll
      for (int j = 0; j < t; ++j) sl[j] = sl0[j];
      tab_ab[b] = ab0;
    } else {
#pragma unroll
      for (int j = 0; j < t; ++j) sl[j] = p.anc[row * p.anc_stride + j];
      tab_ab[b] = make_float2(p.alpha[row * p.H + h], p.beta[row * p.H + h]);
    }
#pragma unroll
    for (int j = 0; j < t; ++j) {
      float a = -1.0f;  // marks a slot outside its depth: the record is skipped
      if (sl[j] < 0 || sl[j] >= p.W_j[j]) {
        raise_error(p.err, GDNBEAM_DERR_SLOT);
        sl[j] = 0;
      } else {
        a = p.rec_a[j][((size_t)r * p.W_j[j] + sl[j]) * p.H + h];
      }
      tab_slot[b * t + j] = sl[j];
      tab_aj[b * t + j] = a;
    }
  }
  __syncthreads();  // the table is complete

  // A tile's record requests (four beams, one 64-column half of one depth's
  // delta_j rows each; the keys k_j are read by the scalar warps) are split
  // round-robin over three warps: the producer (w = 0) and the two record
  // loaders (w = 1, 2).
  constexpr int kRecReq = 16 * t;  // requests per tile
  auto rec_share = [](int w) { return (kRecReq - w + 2) / 3; };
  auto issue_records = [&](int w, int i, uint32_t st, int s) {
    const int l0 = i * NB;  // the tile's first beam in the table
    const int nb = min(NB, nbeams - l0);
    for (int m = lane;; m += 32) {
      const int rq = 3 * m + w;
      if (rq >= kRecReq) break;
      const int j = rq >> 4, cb = (rq >> 3) & 1, gq = rq & 7;
      int y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b = 4 * gq + u;  // beams past the tile's end repeat a valid row
        const int sl = b < nb ? tab_slot[(l0 + b) * t + j] : 0;
        y[u] = (r * p.W_j[j] + sl) * p.H + h;  // delta_j rows are per value head
      }
      const uint32_t dst = st + rec_off + (uint32_t)(j * REC_BYTES + cb * (NB * 128) + gq * (4 * 128));
      tc::tma_gather4(dst, &rm.d[j], vb * VR + cb * 64, y[0], y[1], y[2], y[3], full(s));
    }
    __syncwarp();
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // q, k and v boxes of every tile (lane 0) and its share of the records
    bool issued[kMaxStages] = {};
    uint32_t issued_ph[kMaxStages] = {};
    int ok = 1;
    for (int i = 0; i < nt; ++i) {
      const int s = i % p.stages;
      const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
      if (lane == 0) ok = tc::mbar_wait_sleep(empty(s), ph ^ 1u, abort, p.err) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // the whole warp stops together
      const uint32_t st = base + (uint32_t)(s * p.stage_bytes);
      const int b0 = bb + i * NB;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(full(s), (uint32_t)(B_BYTES + V_BYTES + rec_share(0) * 512));
        for (int kb = 0; kb < DK / 64; ++kb) {
          const uint32_t bk = st + kb * (2 * NB * 128);
          tc::tma_load_3d(bk, &tm_q, hk * DK + kb * 64, b0, r, full(s));
          tc::tma_load_3d(bk + NB * 128, &tm_k, hk * DK + kb * 64, b0, r, full(s));
        }
        for (int kb = 0; kb < 2; ++kb)
          tc::tma_load_3d(st + v_off + kb * (NB * 128), &tm_v, h * p.dv + vb * VR + kb * 64, b0, r,
                          full(s));
        issued[s] = true;
        issued_ph[s] = ph;
      }
      if (t > 0) issue_records(0, i, st, s);
    }
    if (lane == 0)
      for (int s = 0; s < p.stages; ++s)
        if (issued[s]) tc::mbar_wait_drain(full(s), issued_ph[s]);
  } else if (warp >= kRec0 && warp < kScal0) {
    // ---------------------------------------------------------------- records
    // record loader w = 1 or 2: its share of every tile's record requests
    if (t > 0) {
      const int w = 1 + warp - kRec0;
      int ok = 1;
      bool issued[kMaxStages] = {};
      uint32_t issued_ph[kMaxStages] = {};
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i % p.stages;
        const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
        if (lane == 0) ok = tc::mbar_wait_sleep(empty(s), ph ^ 1u, abort, p.err) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // the whole warp stops together
        const uint32_t st = base + (uint32_t)(s * p.stage_bytes);
        if (lane == 0) tc::mbar_expect_tx(full(s), (uint32_t)(rec_share(w) * 512));
        __syncwarp();
        issue_records(w, i, st, s);
        if (lane == 0) {
          tc::mbar_arrive(full(s));
          issued[s] = true;
          issued_ph[s] = ph;
        }
      }
      if (lane == 0)
        for (int s = 0; s < p.stages; ++s)
          if (issued[s]) tc::mbar_wait_drain(full(s), issued_ph[s]);
    }
  } else if (warp >= kScal0) {
    // ---------------------------------------------------------------- scalars
    // replay scalars k_j.q_t, k_j.k_t (eqs. 6-7) and k_t.q_t (eq. 8) of every
    // tile into buffer i & 1, turned into the fold's combined coefficients:
    // four lanes per beam, 32 dimensions each; warp sw takes beams 8 sw ..
    // 8 sw + 7
    const int sw = warp - kScal0;
    const int bl = sw * 8 + (lane >> 2);
    const int c0 = (lane & 3) * (DK / 4);
    // The ancestor keys come from global memory (the lane's DK / 4
    // dimensions of each depth's row, kChunks 16-byte pieces); the first
    // kPre depths are requested before the tile's stage is awaited.
    constexpr int kChunks = DK / 32;
    constexpr int kPre = TD < 12 / kChunks ? TD : 12 / kChunks;
    auto key_row = [&](int l0, int j) {
      const int sl = l0 + bl < nbeams ? tab_slot[(l0 + bl) * t + j] : 0;
      return reinterpret_cast<const uint4*>(
          p.rec_k[j] + ((size_t)(r * p.W_j[j] + sl) * p.Hk + hk) * DK + c0);
    };
    bool ok = true;
    for (int i = 0; ok && i < nt; ++i) {
      const int s = i % p.stages;
      const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
      const int sb = i & 1;
      const uint32_t sph = (uint32_t)(i >> 1) & 1u;
      const int l0 = i * NB;  // the tile's first beam in the table
      const int nb = min(NB, nbeams - l0);
      uint4 kr[kPre > 0 ? kPre : 1][kChunks];
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const uint4* kp = key_row(l0, j);
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) kr[j][ch] = __ldg(kp + ch);
      }
      // the buffer's previous tile has been folded, and this tile has landed
      if (__any_sync(0xffffffffu, !tc::mbar_wait_sleep(sempty(sb), sph ^ 1u, abort, p.err) ||
                                      !tc::mbar_wait_sleep(full(s), ph, abort, p.err))) {
        ok = false;
        break;
      }
      const uint8_t* gst = gbase + s * p.stage_bytes;
      float part[1 + 2 * TD];
#pragma unroll
      for (int x = 0; x < 1 + 2 * TD; ++x) part[x] = 0.f;
#pragma unroll
      for (int ch = 0; ch < DK / 32; ++ch) {  // 8 dimensions per step
        const int c = c0 + ch * 8, kb = c >> 6, cc = c & 63;
        const uint8_t* bk = gst + kb * (2 * NB * 128);
        const uint4 qw = *reinterpret_cast<const uint4*>(bk + sw128_off(bl, cc));
        const uint4 kw = *reinterpret_cast<const uint4*>(bk + sw128_off(NB + bl, cc));
        const uint32_t qa[4] = {qw.x, qw.y, qw.z, qw.w}, ka[4] = {kw.x, kw.y, kw.z, kw.w};
        float q8[8], k8[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          q8[2 * e] = bf(qa[e] & 0xFFFFu); q8[2 * e + 1] = bf(qa[e] >> 16);
          k8[2 * e] = bf(ka[e] & 0xFFFFu); k8[2 * e + 1] = bf(ka[e] >> 16);
        }
#pragma unroll
        for (int x = 0; x < 8; ++x) part[0] = fmaf(k8[x], q8[x], part[0]);
#pragma unroll
        for (int j = 0; j < t; ++j) {
          const uint4 rw = j < kPre ? kr[j < kPre ? j : 0][ch] : __ldg(key_row(l0, j) + ch);
          const uint32_t ra[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float r0 = bf(ra[e] & 0xFFFFu), r1 = bf(ra[e] >> 16);
            part[1 + 2 * j] = fmaf(r0, q8[2 * e], fmaf(r1, q8[2 * e + 1], part[1 + 2 * j]));
            part[2 + 2 * j] = fmaf(r0, k8[2 * e], fmaf(r1, k8[2 * e + 1], part[2 + 2 * j]));
          }
        }
      }
#pragma unroll
      for (int o = 2; o > 0; o >>= 1)
#pragma unroll
        for (int x = 0; x < 1 + 2 * TD; ++x) part[x] += __shfl_xor_sync(0xffffffffu, part[x], o);
      if ((lane & 3) == 0 && bl < nb) {
        // The fold u <- alpha_j u + delta_j c_j over j = 0 .. t-1 (eqs. 6-7)
        // leaves u = (prod_j alpha_j) u_ctx + sum_j (c_j prod_{m > j} alpha_m)
        // delta_j; eq. 8 is linear in both projections.
        const float2 ab = tab_ab[l0 + bl];  // (alpha_t, beta_t)
        float tail = 1.f;                   // prod_{m > j} alpha_m
#pragma unroll
        for (int j = t - 1; j >= 0; --j) {
          const float a = tab_aj[(l0 + bl) * t + j];
          const bool use = a >= 0.f;  // a skipped record leaves both projections unchanged
          const float wq = use ? part[1 + 2 * j] * tail : 0.f;
          const float wk = use ? part[2 + 2 * j] * tail : 0.f;
          s_rec[sb][bl][j] = make_float2(-ab.y * ab.x * wk, ab.x * wq);
          if (use) tail *= a;
        }
        s_beam[sb][bl] = make_float4(ab.y, -ab.y * ab.x * tail, ab.x * tail, part[0]);
      }
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(sfull(sb));
        tc::mbar_arrive(empty(s));  // this warp is done reading the stage
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(VR, 2 * NB);
      bool ok = tc::mbar_wait_sleep(a_ready, 0, abort, p.err);
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i % p.stages;
        const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
        const int acc = i & 1;
        const uint32_t aph = (uint32_t)(i >> 1) & 1u;
        if (!tc::mbar_wait_sleep(full(s), ph, abort, p.err)) break;
        if (!tc::mbar_wait_sleep(tempty(acc), aph ^ 1u, abort, p.err)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(acc * 2 * NB);
        const uint32_t st = base + (uint32_t)(s * p.stage_bytes);
#pragma unroll
        for (int kb = 0; kb < DK / 64; ++kb) {
          const uint64_t bd = tc::sw128_desc(st + kb * (2 * NB * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t col = (uint32_t)(kb * 32 + kk * 8);  // 16 K elements = 8 columns
            tc::mma_bf16_ts(d, tmem_base + kColAHi + col, bd + 2u * kk, idesc, (kb | kk) != 0);
            tc::mma_bf16_ts(d, tmem_base + kColALo + col, bd + 2u * kk, idesc, 1u);
          }
        }
        tc::mma_commit(empty(s));
        tc::mma_commit(tfull(acc));
      }
      tc::mma_commit(drain_bar);
      tc::mbar_wait_drain(drain_bar, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kEpi0;               // 0..7
    const int hb = ew >> 2;                    // which half of a tile (beams) / of K this warp takes
    const int lg = warp & 3;                   // TMEM lane group
    const int i_row = lg * 32 + lane;          // value row = TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(lg * 32) << 16);

    // the S_ctx batches -> bf16 hi / lo words in TMEM
    {
      auto put = [&](const float4 (&x)[8], int bt) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float xs[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float a0 = xs[2 * e], a1 = xs[2 * e + 1];
            const float h0 = __bfloat162float(__float2bfloat16_rn(a0));
            const float h1 = __bfloat162float(__float2bfloat16_rn(a1));
            hi[2 * c + e] = pack_bf16(h0, h1);
            lo[2 * c + e] = pack_bf16(a0 - h0, a1 - h1);
          }
        }
        const uint32_t col = (uint32_t)(hb * (DK / 4) + bt * 16);
        tc::tmem_st16(lane_base + kColAHi + col, hi);
        tc::tmem_st16(lane_base + kColALo + col, lo);
      };
#pragma unroll
      for (int bt = 0; bt < kEarly; ++bt) put(xe[bt], bt);
#pragma unroll
      for (int bt = kEarly; bt < kBatches; ++bt) {
        float4 x[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = __ldg(reinterpret_cast<const float4*>(S) + bt * 8 + c);
        put(x, bt);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(a_ready);
    }

    // A failed wait marks this warp dead: it then skips all work but keeps
    // making its arrivals, so no other role waits on it forever.
    bool dead = false;
    // residual stream element of beam e of this thread's half of tile i
    auto goff = [&](int i, int e) {
      return (((size_t)r * p.W_t + bb + i * NB + hb * 16 + e) * p.H + h) * p.dv + vb * VR + i_row;
    };
    // the residual values of a tile are loaded one tile ahead
    float xr[EXTRA ? 16 : 1];
    auto load_x = [&](int i, float (&dst)[EXTRA ? 16 : 1]) {
      if constexpr (EXTRA) {
        const int nbi = i < nt ? min(NB, p.W_t - (bb + i * NB)) : 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = hb * 16 + e < nbi ? p.x_inout[goff(i, e)] : 0.f;
      }
    };
    if (EXTRA && p.x_inout) load_x(0, xr);
    for (int i = 0; i < nt; ++i) {
      const int s = i % p.stages;
      const int acc = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      const int sb = i & 1;
      const int b0 = bb + i * NB;
      const int nb = min(NB, p.W_t - b0);
      float xn[EXTRA ? 16 : 1];
      if (EXTRA && p.x_inout) load_x(i + 1, xn);
      if (!dead) dead = __any_sync(0xffffffffu, !tc::mbar_wait_sleep(sfull(sb), aph, abort, p.err));
      if (!dead) dead = __any_sync(0xffffffffu, !tc::mbar_wait_sleep(tfull(acc), aph, abort, p.err));
      if (!dead) {
        tc::fence_after_sync();
        const uint8_t* gst = gbase + s * p.stage_bytes;
        const uint32_t ta = lane_base + (uint32_t)(acc * 2 * NB + hb * 16);
        uint32_t uq[16], uk[16];
        tc::tmem_ld16_nowait(ta, uq);
        tc::tmem_ld16_nowait(ta + NB, uk);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tempty(acc));
        const uint8_t* rd = gst + rec_off + (i_row >> 6) * (NB * 128) + (i_row & 63) * 2;
        const uint8_t* vs = gst + v_off + (i_row >> 6) * (NB * 128) + (i_row & 63) * 2;
        uint8_t* os = &s_out[sb][(hb * 4 + lg) * OUT_WARP] + lane * 2;
        // the store of two tiles ago has read this output buffer (the one
        // after it, to the other buffer, may still be in flight)
        if (lane == 0) tc::bulk_wait_read<1>();
        __syncwarp();
        // every beam of the half tile is computed; rows past the last beam
        // are never stored (the tile store clips them)
        // (all 16 beams are folded into registers first and stored after,
        // so no shared-memory store sits between the loads)
        float dl[16], ol[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int b = hb * 16 + e;
          const float4 bm = s_beam[sb][b];
          const float vv = bf(*reinterpret_cast<const uint16_t*>(vs + b * 128));
          float delta = fmaf(bm.y, __uint_as_float(uk[e]), bm.x * vv);
          float o = bm.z * __uint_as_float(uq[e]);
#pragma unroll
          for (int j = 0; j < t; ++j) {
            const float2 rc = s_rec[sb][b][j];
            const float dj = bf(*reinterpret_cast<const uint16_t*>(rd + j * REC_BYTES + b * 128));
            delta = fmaf(rc.x, dj, delta);
            o = fmaf(rc.y, dj, o);
          }
          dl[e] = delta;
          ol[e] = fmaf(bm.w, delta, o);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          *reinterpret_cast<__nv_bfloat16*>(os + e * 64) = __float2bfloat16_rn(dl[e]);
          *reinterpret_cast<__nv_bfloat16*>(os + OUT_WARP / 2 + e * 64) = __float2bfloat16_rn(ol[e]);
        }
        if constexpr (EXTRA) {
          if (p.x_inout) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (hb * 16 + e < nb) p.x_inout[goff(i, e)] = xr[e] + ol[e];
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            if (hb * 16 + e < nb) {
              if (p.delta_dump) p.delta_dump[goff(i, e)] = dl[e];
              if (p.o_dump) p.o_dump[goff(i, e)] = ol[e];
            }
          }
        }
        // this warp's boxes go out by TMA
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (hb * 16 < nb) {
            const uint32_t ob = tc::smem_u32(&s_out[sb][(hb * 4 + lg) * OUT_WARP]);
            tc::tma_store_3d(&tm_d, h * p.dv + vb * VR + lg * 32, b0 + hb * 16, r, ob);
            if (p.store_o)
              tc::tma_store_3d(&tm_o, h * p.dv + vb * VR + lg * 32, b0 + hb * 16, r, ob + OUT_WARP / 2);
          }
          tc::bulk_commit();
        }
      }
      // this warp is done with the tile's stage and scalars
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(sempty(sb));
        tc::mbar_arrive(empty(s));
      }
      if constexpr (EXTRA) {
#pragma unroll
        for (int e = 0; e < 16; ++e) xr[e] = xn[e];
      }
    }
    if (lane == 0) tc::bulk_wait_all();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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

// [R][W_t][width] bf16 as a 3-D map with a box_cols x box_rows x 1 box.
inline bool beam_map(CUtensorMap* map, const void* ptr, int R, int W_t, int width, bool swizzle,
                     int box_cols = 64, int box_rows = NB) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || ((uintptr_t)ptr & 15) != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)W_t, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)W_t * width * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][cols] bf16 (one record per row) as a 2-D map with a one-row, 64-column box.
inline bool rows_map(CUtensorMap* map, const void* ptr, long long rows, int cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || ((uintptr_t)ptr & 15) != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Makespan, in tile times, of `base` blocks of each size sizes[0..n) run in
// launch order (every block of the first size before any of the next, as
// grid z is the slowest index), each on the SM that frees first, one block
// per SM; a block costs its tiles plus a prologue of about three tiles.
inline long long list_schedule(long long base, const int* sizes, int n, int sms) {
  std::vector<long long> h((size_t)sms, 0);  // SM free times, a min-heap
  long long mk = 0;
  for (int z = 0; z < n; ++z)
    for (long long b = 0; b < base; ++b) {
      std::pop_heap(h.begin(), h.end(), std::greater<long long>());
      h.back() += sizes[z] + 3;
      mk = std::max(mk, h.back());
      std::push_heap(h.begin(), h.end(), std::greater<long long>());
    }
  return mk;
}

// When the uniform split leaves a short grid's last wave part full, each
// triple's tiles may go in two unequal blocks instead: all the large ones
// first, then the small ones fill the SMs that free early. Returns the size
// of the first block, or 0 when no such split beats `tpb`-tile blocks.
// (Decided once per grid shape.)
inline int two_piece_split(long long base, int n_tiles, int tpb, int sms) {
  static std::mutex mu;
  static std::map<std::tuple<long long, int, int, int>, int> memo;
  const auto key = std::make_tuple(base, n_tiles, tpb, sms);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = memo.find(key);
  if (it != memo.end()) return it->second;
  int best = 0;
  if (sms > 0 && base < 4LL * sms && n_tiles >= 4) {
    const int ns = (n_tiles + tpb - 1) / tpb;
    std::vector<int> uni((size_t)ns, tpb);
    uni.back() = n_tiles - tpb * (ns - 1);
    long long best_cost = list_schedule(base, uni.data(), ns, sms);
    for (int first = (n_tiles + 1) / 2; first < n_tiles; ++first) {
      const int sizes[2] = {first, n_tiles - first};
      const long long c = list_schedule(base, sizes, 2, sms);
      if (c < best_cost) {
        best_cost = c;
        best = first;
      }
    }
  }
  memo[key] = best;
  return best;
}

// Launches the kernel for key width DK (the caller checked the shape).
template <int DK>
int launch_tc_replay_dk(const ReplayArgs& a, cudaStream_t s) {
  constexpr int B_BYTES = Width<DK>::B_BYTES, REC_BYTES = Width<DK>::REC_BYTES;
  TcReplayParams p{};
  p.R = a.R; p.H = a.H; p.Hk = a.Hk; p.dv = a.d_v; p.t = a.t; p.W_t = a.W_t;
  p.n_tiles = (a.W_t + NB - 1) / NB;
  // Beam tiles per block. When (request, head, value block) triples are too
  // few to fill the SMs, the tiles of one triple are split over several
  // blocks (each reads its own copy of S_ctx). The split minimises
  // waves x (tiles per block + a prologue worth about three tiles: TMEM
  // set-up, S_ctx and the table), one block per SM.
  {
    const long long base = (long long)a.R * a.H * (a.d_v / VR);
    const long long sms = sm_count();
    long long best_cost = -1;
    for (int ns = 1; ns <= p.n_tiles; ++ns) {
      const int tpb = (p.n_tiles + ns - 1) / ns;
      if ((p.n_tiles + tpb - 1) / tpb != ns) continue;  // same as a smaller split
      const long long cost = (base * ns + sms - 1) / sms * (tpb + 3);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        p.tiles_per_block = tpb;
      }
    }
    p.first_tiles = two_piece_split(base, p.n_tiles, p.tiles_per_block, (int)sms);
    if (p.first_tiles > 0) p.tiles_per_block = p.first_tiles;  // the larger block
  }
  const int nsplit =
      p.first_tiles > 0 ? 2 : (p.n_tiles + p.tiles_per_block - 1) / p.tiles_per_block;
  p.stage_bytes = B_BYTES + V_BYTES + a.t * REC_BYTES;
  const size_t table = (size_t)p.tiles_per_block * NB * (8 + 8 * a.t);
  const int static_bytes = 2 * OUT_BYTES + 10 * 1024;  // output tiles, scalar buffers, barriers
  const long long budget = 227LL * 1024 - static_bytes - 1024 - (long long)table;
  p.stages = budget > 0 ? (int)(budget / p.stage_bytes) : 0;
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  // one stage still runs (loads of a tile then wait for the previous tile's
  // consumers); none left (deep replay on a wide beam) takes the CUDA cores
  if (p.stages < 1) return launch_replay(GDNBEAM_BF16, a, s);
  p.sctx = a.sctx; p.sctx_rstride = a.sctx_rstride;
  p.alpha = a.alpha; p.beta = a.beta;
  RecMaps rm;
  memset(&rm, 0, sizeof(rm));
  for (int j = 0; j < a.t; ++j) {
    p.rec_a[j] = a.depth[j].alpha;
    p.rec_k[j] = reinterpret_cast<const uint16_t*>(a.depth[j].k);
    p.W_j[j] = a.depth[j].W_j;
    if (((uintptr_t)a.depth[j].k & 15) || ((uintptr_t)a.depth[j].delta & 15)) return GDNBEAM_EINVAL;
    const long long rows = (long long)a.R * a.depth[j].W_j * a.H;
    if (rows > 0x7FFFFFFFLL) return launch_replay(GDNBEAM_BF16, a, s);
    if (!rows_map(&rm.d[j], a.depth[j].delta, rows, a.d_v)) return GDNBEAM_ECUDA;
  }
  p.anc = a.anc; p.anc_stride = a.anc_stride;
  p.x_inout = a.x_inout; p.delta_dump = a.delta_dump; p.o_dump = a.o_dump; p.err = a.err;
  p.store_o = a.o_out != nullptr;
  if (!a.o_out && !a.x_inout) return GDNBEAM_EINVAL;
  if (((uintptr_t)a.sctx & 15) || (a.sctx_rstride % 4) != 0) return GDNBEAM_EINVAL;
  CUtensorMap mq, mk, mv, md, mo;
  const int kw = a.Hk * DK, vw = a.H * a.d_v;
  if (!beam_map(&mq, a.q, a.R, a.W_t, kw, true) || !beam_map(&mk, a.k, a.R, a.W_t, kw, true) ||
      !beam_map(&mv, a.v, a.R, a.W_t, vw, false) ||
      !beam_map(&md, a.delta_out, a.R, a.W_t, vw, false, 32, 16) ||
      !beam_map(&mo, a.o_out ? a.o_out : a.delta_out, a.R, a.W_t, vw, false, 32, 16))
    return GDNBEAM_ECUDA;
  const size_t dyn = 1024 + (size_t)p.stages * p.stage_bytes + table;
  const bool extra = a.delta_dump || a.o_dump || a.x_inout;
  const dim3 grid(a.R * a.H, a.d_v / VR, nsplit);
  switch (a.t) {
#define GDN_REPLAY_TC(TD_)                                                                      \
  case TD_:                                                                                     \
    if (extra) {                                                                                \
      GDN_CUDA(cudaFuncSetAttribute(replay_tc_kernel<TD_, true, DK>,                            \
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));    \
      replay_tc_kernel<TD_, true, DK><<<grid, kThreads, dyn, s>>>(mq, mk, mv, md, mo, rm, p);   \
    } else {                                                                                    \
      GDN_CUDA(cudaFuncSetAttribute(replay_tc_kernel<TD_, false, DK>,                           \
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));    \
      replay_tc_kernel<TD_, false, DK><<<grid, kThreads, dyn, s>>>(mq, mk, mv, md, mo, rm, p);  \
    }                                                                                           \
    break;
    GDN_REPLAY_TC(0) GDN_REPLAY_TC(1) GDN_REPLAY_TC(2) GDN_REPLAY_TC(3) GDN_REPLAY_TC(4)
    GDN_REPLAY_TC(5) GDN_REPLAY_TC(6)
#undef GDN_REPLAY_TC
    default: return launch_replay(GDNBEAM_BF16, a, s);
  }
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace
}  // namespace gdnbeam
