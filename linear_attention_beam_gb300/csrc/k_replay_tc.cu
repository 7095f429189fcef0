// Fused shared-context replay on tcgen05 tensor cores (bf16, d_k = d_v = 128).
//
// OneLA §2.5: one block per (request, head) loads that head's S_ctx once and
// reuses it for every beam tile; per tile it forms the two projections of
// §2.3 eqs. 6-7 from S_ctx, folds the ancestors' records (alpha_j, delta_j,
// k_j) into them, evaluates eq. 8 and writes only delta_t (the new record)
// and o_t. No per-beam d_v x d_k state exists anywhere.
//
// Mapping to sm_103a:
//   * S_ctx is fp32 in memory; the block splits it into bf16 hi + lo halves
//     in shared memory (128-byte swizzled, K-major), the A operand (M = 128
//     value rows) of two MMAs per K step, so the contraction keeps ~16
//     mantissa bits of S_ctx.
//   * Beams go in tiles of 32. Per tile one producer warp stages by TMA the
//     32 queries and 32 keys as the B operand (N = 64: q rows then k rows),
//     the 32 value rows, and with 256-byte bulk copies each beam's ancestor
//     records delta_j and k_j, found through the ancestry index; stages are
//     double-buffered on mbarriers.
//   * One thread issues tcgen05.mma into a double-buffered TMEM accumulator:
//     column b holds u_q of beam b, column 32 + b its u_k, lane = value row.
//   * Four epilogue warps (thread = value row i) compute the replay scalars
//     k_j.q_t, k_j.k_t and k_t.q_t, fold the records, apply eq. 8, and write
//     delta_t and o_t into shared tiles that TMA stores to memory.
// Every wait is bounded in time (GDNBEAM_DERR_TIMEOUT on expiry).
#include <cuda.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int D = 128;            // head width (d_k = d_v)
constexpr int NB = 32;            // beams per tile
constexpr int kEpiWarps = 8;      // two per SM sub-partition; each folds 16 beams of a tile
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kMaxDepth = 6;      // replay depths this kernel stages
constexpr int A_BYTES = 2 * D * D;          // one bf16 half of S_ctx: 32 KiB
constexpr int B_BYTES = 2 * NB * D * 2;     // q and k rows: 16 KiB
constexpr int REC_BYTES = 2 * NB * D * 2;   // delta_j and k_j rows of one depth: 16 KiB
constexpr int META_BYTES = 1024;            // per-beam gates and ancestors' decays
constexpr int kMaxStages = 4;

struct TcReplayParams {
  int R, H, t, W_t, n_tiles, stages, stage_bytes;
  const float* sctx;
  long long sctx_rstride;
  const float *alpha, *beta;
  const __nv_bfloat16* v;
  const __nv_bfloat16* rec_k[kMaxDepth];
  const __nv_bfloat16* rec_d[kMaxDepth];
  const float* rec_a[kMaxDepth];
  int W_j[kMaxDepth];
  const int32_t* anc;
  int anc_stride;
  __nv_bfloat16 *delta_out, *o_out;
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

// Stage layout: [B: q rows | k rows, per 64-column block][REC per depth:
// delta rows | k rows][META: (alpha_t, beta_t) per beam, alpha_j per beam and
// depth (negative for a slot outside its depth)].
template <int TD>  // replay depth t of this call
__global__ void __launch_bounds__(kThreads, 1)
    replay_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     TcReplayParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 6];
  // replay scalars of two tiles (the fold reads one while the next is computed)
  __shared__ float4 s_beam[2][NB];                              // (alpha_t, beta_t, k_t.q_t, -)
  __shared__ float4 s_rec[2][NB][TD > 0 ? TD : 1];              // (alpha_j, k_j.q_t, k_j.k_t, -)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA_hi = base, sA_lo = base + A_BYTES;
  const uint32_t sStage0 = base + 2 * A_BYTES;
  uint8_t* gStage0 = gbase + 2 * A_BYTES;
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(kMaxStages + s); };
  auto tfull = [&](int a) { return bar(2 * kMaxStages + a); };
  auto tempty = [&](int a) { return bar(2 * kMaxStages + 2 + a); };
  const uint32_t a_ready = bar(2 * kMaxStages + 4);
  const uint32_t drain_bar = bar(2 * kMaxStages + 5);
  volatile int* abort = &s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x / p.H, h = blockIdx.x % p.H;
  constexpr int t = TD;
  const int rec_off = B_BYTES;
  const int meta_off = rec_off + t * REC_BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      tc::mbar_init(full(s), 32);  // every producer lane arrives after its stores and copies
      tc::mbar_init(empty(s), 2);  // released by the MMA commit and by the epilogue
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull(a), 1);
      tc::mbar_init(tempty(a), kEpiWarps);
    }
    tc::mbar_init(a_ready, kEpiWarps);
    tc::mbar_init(drain_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tm_q); tc::tma_prefetch(&tm_k);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), 128);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    bool issued[kMaxStages] = {false, false, false, false};
    uint32_t issued_ph[kMaxStages] = {0, 0, 0, 0};
    for (int i = 0; i < p.n_tiles; ++i) {
      const int s = i % p.stages;
      const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
      const int b0 = i * NB;
      const int nb = min(NB, p.W_t - b0);
      // this tile's gates and ancestor slots, fetched before the stage frees
      int slot[TD > 0 ? TD : 1];
      float a_j[TD > 0 ? TD : 1];
      float al = 0.f, be = 0.f;
      if (lane < nb) {
        const size_t row = (size_t)r * p.W_t + b0 + lane;
        al = p.alpha[row * p.H + h];
        be = p.beta[row * p.H + h];
#pragma unroll
        for (int j = 0; j < t; ++j) {
          int sl = p.anc[row * p.anc_stride + j];
          a_j[j] = -1.0f;  // marks a slot outside its depth: the record is skipped
          if (sl < 0 || sl >= p.W_j[j]) {
            raise_error(p.err, GDNBEAM_DERR_SLOT);
            sl = 0;
          } else {
            a_j[j] = p.rec_a[j][((size_t)r * p.W_j[j] + sl) * p.H + h];
          }
          slot[j] = sl;
        }
      }
      int ok = 0;
      if (lane == 0) ok = tc::mbar_wait_sleep(empty(s), ph ^ 1u, abort, p.err) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // the whole warp stops together
      const uint32_t st = sStage0 + (uint32_t)(s * p.stage_bytes);
      uint8_t* gst = gStage0 + s * p.stage_bytes;
      if (lane == 0) {
        tc::mbar_expect_tx(full(s), (uint32_t)(B_BYTES + t * nb * 2 * D * 2));
        for (int kb = 0; kb < 2; ++kb) {
          const uint32_t bk = st + kb * (2 * NB * 128);
          tc::tma_load_3d(bk, &tm_q, h * D + kb * 64, b0, r, full(s));
          tc::tma_load_3d(bk + NB * 128, &tm_k, h * D + kb * 64, b0, r, full(s));
        }
      }
      __syncwarp();
      if (lane < nb) {
        float2* albe = reinterpret_cast<float2*>(gst + meta_off);
        float* ajs = reinterpret_cast<float*>(gst + meta_off + NB * 8);
        albe[lane] = make_float2(al, be);
#pragma unroll
        for (int j = 0; j < t; ++j) {
          ajs[lane * kMaxDepth + j] = a_j[j];
          const size_t rec = ((size_t)r * p.W_j[j] + slot[j]) * p.H + h;
          const uint32_t dst = st + rec_off + j * REC_BYTES + lane * (D * 2);
          tc::bulk_load(dst, p.rec_d[j] + rec * D, D * 2, full(s));
          tc::bulk_load(dst + NB * D * 2, p.rec_k[j] + rec * D, D * 2, full(s));
        }
      }
      tc::mbar_arrive(full(s));  // releases this lane's stage stores
      if (lane == 0) { issued[s] = true; issued_ph[s] = ph; }
    }
    if (lane == 0)
      for (int s = 0; s < p.stages; ++s)
        if (issued[s]) tc::mbar_wait_drain(full(s), issued_ph[s]);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(D, 2 * NB);
      bool ok = tc::mbar_wait_sleep(a_ready, 0, abort, p.err);
      for (int i = 0; ok && i < p.n_tiles; ++i) {
        const int s = i % p.stages;
        const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
        const int acc = i & 1;
        const uint32_t aph = (uint32_t)(i >> 1) & 1u;
        if (!tc::mbar_wait_sleep(full(s), ph, abort, p.err)) break;
        if (!tc::mbar_wait_sleep(tempty(acc), aph ^ 1u, abort, p.err)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(acc * 2 * NB);
        const uint32_t st = sStage0 + (uint32_t)(s * p.stage_bytes);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ahi = tc::sw128_desc(sA_hi + kb * (D * 128));
          const uint64_t alo = tc::sw128_desc(sA_lo + kb * (D * 128));
          const uint64_t bd = tc::sw128_desc(st + kb * (2 * NB * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc::mma_bf16(d, ahi + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0);
            tc::mma_bf16(d, alo + 2u * kk, bd + 2u * kk, idesc, 1u);
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
    const int ew = warp - 2;                   // 0..7
    const int ep = threadIdx.x - 64;           // 0..255
    const int hb = ew >> 2;                    // which 16 beams of a tile this warp folds
    const int lg = warp & 3;                   // TMEM lane group
    const int i_row = lg * 32 + lane;          // value row = TMEM lane

    // S_ctx of this (request, head) -> bf16 hi / lo A operands, while the
    // producer already streams the first tiles
    {
      const float* S = p.sctx + (size_t)r * p.sctx_rstride + (size_t)h * D * D;
      constexpr int kUnits = D * (D / 8) / kEpiThreads;  // 8 row-chunks per thread
      float4 xv[kUnits][2];
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = ep + k * kEpiThreads, row = u >> 4, chunk = u & 15;
        xv[k][0] = __ldg(reinterpret_cast<const float4*>(S + (size_t)row * D + chunk * 8));
        xv[k][1] = __ldg(reinterpret_cast<const float4*>(S + (size_t)row * D + chunk * 8 + 4));
      }
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = ep + k * kEpiThreads, row = u >> 4, chunk = u & 15;
        const float xs[8] = {xv[k][0].x, xv[k][0].y, xv[k][0].z, xv[k][0].w,
                             xv[k][1].x, xv[k][1].y, xv[k][1].z, xv[k][1].w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat16 h0 = __float2bfloat16_rn(xs[2 * e]), h1 = __float2bfloat16_rn(xs[2 * e + 1]);
          __nv_bfloat16 l0 = __float2bfloat16_rn(xs[2 * e] - __bfloat162float(h0));
          __nv_bfloat16 l1 = __float2bfloat16_rn(xs[2 * e + 1] - __bfloat162float(h1));
          hi[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lo[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        const int kb = chunk >> 3, col = (chunk & 7) * 8;
        const uint32_t off = (uint32_t)kb * (D * 128) + sw128_off(row, col);
        *reinterpret_cast<uint4*>(gbase + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(gbase + A_BYTES + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(a_ready);
    }

    // replay scalars k_j.q_t, k_j.k_t (eqs. 6-7) and k_t.q_t (eq. 8) of tile
    // i into buffer i & 1; warp ew takes beams ew, ew + 8, ew + 16, ew + 24
    auto scalars = [&](int i) -> bool {
      const int s = i % p.stages;
      const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
      const int nb = min(NB, p.W_t - i * NB);
      if (__any_sync(0xffffffffu, !tc::mbar_wait_sleep(full(s), ph, abort, p.err))) return false;
      const uint8_t* gst = gStage0 + s * p.stage_bytes;
      const float2* albe = reinterpret_cast<const float2*>(gst + meta_off);
      const float* ajs = reinterpret_cast<const float*>(gst + meta_off + NB * 8);
      const int c = lane * 4, kb = c >> 6, cc = c & 63;
      const uint8_t* bk = gst + kb * (2 * NB * 128);
      float part[4][1 + 2 * TD];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int b = ew + 8 * e;
        const uint2 qw = *reinterpret_cast<const uint2*>(bk + sw128_off(b, cc));
        const uint2 kw = *reinterpret_cast<const uint2*>(bk + sw128_off(NB + b, cc));
        const float q4[4] = {bf(qw.x & 0xFFFF), bf(qw.x >> 16), bf(qw.y & 0xFFFF), bf(qw.y >> 16)};
        const float k4[4] = {bf(kw.x & 0xFFFF), bf(kw.x >> 16), bf(kw.y & 0xFFFF), bf(kw.y >> 16)};
        float kq = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) kq = fmaf(k4[x], q4[x], kq);
        part[e][0] = kq;
#pragma unroll
        for (int j = 0; j < t; ++j) {
          const uint8_t* kr = gst + rec_off + j * REC_BYTES + NB * D * 2 + b * (D * 2);
          const uint2 rw = *reinterpret_cast<const uint2*>(kr + c * 2);
          const float r4[4] = {bf(rw.x & 0xFFFF), bf(rw.x >> 16), bf(rw.y & 0xFFFF), bf(rw.y >> 16)};
          float cq = 0.f, ck = 0.f;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            cq = fmaf(r4[x], q4[x], cq);
            ck = fmaf(r4[x], k4[x], ck);
          }
          part[e][1 + 2 * j] = cq;
          part[e][2 + 2 * j] = ck;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int x = 0; x < 1 + 2 * TD; ++x)
            part[e][x] += __shfl_xor_sync(0xffffffffu, part[e][x], o);
      if (lane == 0) {
        const int sb = i & 1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int b = ew + 8 * e;
          if (b >= nb) continue;
          const float2 ab = albe[b];
          s_beam[sb][b] = make_float4(ab.x, ab.y, part[e][0], 0.f);
#pragma unroll
          for (int j = 0; j < t; ++j) {
            const float a = ajs[b * kMaxDepth + j];
            // a skipped record leaves both projections unchanged
            s_rec[sb][b][j] = a >= 0.f ? make_float4(a, part[e][1 + 2 * j], part[e][2 + 2 * j], 0.f)
                                       : make_float4(1.f, 0.f, 0.f, 0.f);
          }
        }
      }
      return true;
    };

    // this thread's value entries of its 16 beams of tile i, loaded one tile
    // ahead so the fold never waits on them
    auto load_values = [&](int i, uint16_t (&vr)[16]) {
      const int b0 = i * NB, nb = min(NB, p.W_t - b0);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int b = hb * 16 + e;
        vr[e] = b < nb ? __ldg(reinterpret_cast<const uint16_t*>(
                             p.v + (((size_t)r * p.W_t + b0 + b) * p.H + h) * D + i_row))
                       : (uint16_t)0;
      }
    };
    uint16_t vraw[16];
    if (p.n_tiles > 0) load_values(0, vraw);

    // A failed wait marks the epilogue dead: it then skips all work but keeps
    // taking part in the named barriers, so no epilogue warp waits forever.
    bool dead = p.n_tiles > 0 ? !scalars(0) : false;
    tc::named_sync(1, kEpiThreads);
    for (int i = 0; i < p.n_tiles; ++i) {
      const int s = i % p.stages;
      const int acc = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      const int sb = i & 1;
      const int b0 = i * NB;
      const int nb = min(NB, p.W_t - b0);
      uint16_t vnext[16];
      if (i + 1 < p.n_tiles) load_values(i + 1, vnext);
      if (!dead && i + 1 < p.n_tiles) dead = !scalars(i + 1);
      if (!dead) dead = __any_sync(0xffffffffu, !tc::mbar_wait_sleep(tfull(acc), aph, abort, p.err));
      if (!dead) {
        tc::fence_after_sync();
        const uint8_t* gst = gStage0 + s * p.stage_bytes;
        const uint32_t ta = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(acc * 2 * NB + hb * 16);
        uint32_t uq[16], uk[16];
        tc::tmem_ld16_nowait(ta, uq);
        tc::tmem_ld16_nowait(ta + NB, uk);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tempty(acc));
        const uint8_t* rd = gst + rec_off + i_row * 2;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int b = hb * 16 + e;
          if (b < nb) {
            float u_q = __uint_as_float(uq[e]), u_k = __uint_as_float(uk[e]);
#pragma unroll
            for (int j = 0; j < t; ++j) {
              const float4 rc = s_rec[sb][b][j];
              const float dj = bf(*reinterpret_cast<const uint16_t*>(rd + j * REC_BYTES + b * (D * 2)));
              u_q = fmaf(rc.x, u_q, dj * rc.y);
              u_k = fmaf(rc.x, u_k, dj * rc.z);
            }
            const float4 bm = s_beam[sb][b];
            const float vv = bf(vraw[e]);
            const float delta = bm.y * (vv - bm.x * u_k);
            const float o = fmaf(bm.x, u_q, delta * bm.z);
            const size_t goff = (((size_t)r * p.W_t + b0 + b) * p.H + h) * D + i_row;
            p.delta_out[goff] = __float2bfloat16_rn(delta);
            p.o_out[goff] = __float2bfloat16_rn(o);
            if (p.delta_dump) p.delta_dump[goff] = delta;
            if (p.o_dump) p.o_dump[goff] = o;
            if (p.x_inout) p.x_inout[goff] += o;
          }
        }
      }
      // every epilogue warp is done with stage s and with scalar buffer sb
      tc::named_sync(1, kEpiThreads);
      if (ep == 0 && !dead) tc::mbar_arrive(empty(s));
      if (i + 1 < p.n_tiles) {
#pragma unroll
        for (int e = 0; e < 16; ++e) vraw[e] = vnext[e];
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, 128);
  }
}

// ---- host side -----------------------------------------------------------------

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

// [R][W_t][H*128] bf16 as a 3-D map with a box_cols x box_rows x 1 box.
bool beam_map(CUtensorMap* map, const void* ptr, int R, int W_t, int H, bool swizzle,
              int box_cols = 64, int box_rows = NB) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || ((uintptr_t)ptr & 15) != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)H * D, (cuuint64_t)W_t, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)H * D * 2, (cuuint64_t)W_t * H * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_replay_supported(int dtype, int d_k, int d_v) {
  return dtype == GDNBEAM_BF16 && d_k == D && d_v == D;
}

int launch_tc_replay(const ReplayArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.t > kMaxDepth || a.d_k != D || a.d_v != D) return launch_replay(GDNBEAM_BF16, a, s);
  TcReplayParams p{};
  p.R = a.R; p.H = a.H; p.t = a.t; p.W_t = a.W_t;
  p.n_tiles = (a.W_t + NB - 1) / NB;
  p.stage_bytes = B_BYTES + a.t * REC_BYTES + META_BYTES;
  const int static_bytes = 8 * 1024;  // scalar buffers and barriers
  const int budget = 227 * 1024 - static_bytes - 1024 - 2 * A_BYTES;
  p.stages = budget / p.stage_bytes;
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  if (p.stages < 2) return launch_replay(GDNBEAM_BF16, a, s);
  p.sctx = a.sctx; p.sctx_rstride = a.sctx_rstride;
  p.alpha = a.alpha; p.beta = a.beta;
  p.v = (const __nv_bfloat16*)a.v;
  for (int j = 0; j < a.t; ++j) {
    p.rec_k[j] = (const __nv_bfloat16*)a.depth[j].k;
    p.rec_d[j] = (const __nv_bfloat16*)a.depth[j].delta;
    p.rec_a[j] = a.depth[j].alpha;
    p.W_j[j] = a.depth[j].W_j;
    if (((uintptr_t)p.rec_k[j] & 15) || ((uintptr_t)p.rec_d[j] & 15)) return GDNBEAM_EINVAL;
  }
  p.anc = a.anc; p.anc_stride = a.anc_stride;
  p.delta_out = (__nv_bfloat16*)a.delta_out; p.o_out = (__nv_bfloat16*)a.o_out;
  p.x_inout = a.x_inout; p.delta_dump = a.delta_dump; p.o_dump = a.o_dump; p.err = a.err;
  if (((uintptr_t)a.sctx & 15) || (a.sctx_rstride % 4) != 0) return GDNBEAM_EINVAL;
  CUtensorMap mq, mk;
  if (!beam_map(&mq, a.q, a.R, a.W_t, a.H, true) || !beam_map(&mk, a.k, a.R, a.W_t, a.H, true))
    return GDNBEAM_ECUDA;
  const size_t dyn = 1024 + 2 * A_BYTES + (size_t)p.stages * p.stage_bytes;
  switch (a.t) {
#define GDN_REPLAY_TC(TD_)                                                                   \
  case TD_:                                                                                  \
    GDN_CUDA(cudaFuncSetAttribute(replay_tc_kernel<TD_>,                                     \
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));   \
    replay_tc_kernel<TD_><<<a.R * a.H, kThreads, dyn, s>>>(mq, mk, p);                       \
    break;
    GDN_REPLAY_TC(0) GDN_REPLAY_TC(1) GDN_REPLAY_TC(2) GDN_REPLAY_TC(3) GDN_REPLAY_TC(4)
    GDN_REPLAY_TC(5) GDN_REPLAY_TC(6)
#undef GDN_REPLAY_TC
    default: return launch_replay(GDNBEAM_BF16, a, s);
  }
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace gdnbeam
