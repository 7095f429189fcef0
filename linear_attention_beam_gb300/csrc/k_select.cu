// Exact global top-W beam selection and the ancestry-index update.
//
// Selection (OneLA §1.1: all live beams expand over the codebook and one
// global top-k keeps the survivors) orders candidate (b, v) of a request by
//   s = fl32(cum'_b + fl32(z_bv - lse_b)),  cum'_b = fl32(cum_b + bias_b),
// descending, ties to the lower flat index b*V + v. Every candidate carries
// one 64-bit key: the orderable image of s in the high word and
// (2^32 - 1 - flat) in the low word, so larger keys rank first and keys are
// unique within a request.
//
// Fast path, one block per request (a read of only the listed logit tiles):
//   bound   the scores of one real candidate per (row, 256-code tile) — the
//           tile maximum, which the logits GEMM already produces for the
//           log-normaliser — and the W-th largest of them, tau; the tiles
//           whose maximum reaches tau are listed;
//   filter  every code of the listed tiles with s >= tau is kept on chip;
//   select  exact top-W of the kept codes by radix search on the keys, sorted.
// If at least W candidates are kept, every candidate left out scores below
// the W-th largest kept one, so the result is exact whatever tau was.
// tau is the score of a real candidate, so at least W candidates reach it and
// the W best all lie in listed tiles. When more candidates reach tau than fit
// on chip (scores dominated by a few parents, every code of whose rows clears
// the bound), the bound is narrowed over the listed tiles' codes by an
// 11-bit radix histogram of the 32-bit score keys until the codes reaching
// it fit, and they are collected again: still exact.
// A request that cannot be narrowed (more candidates tie at one score than
// fit) falls back to the two exact stages of RecoGEM §4.3: a per-row precut
// to the local top-K (K = min(W, V)), then a request-level selection among
// the survivors; a candidate the precut drops is beaten by K candidates of
// its own row.
//
// Ancestry (OneLA §2.4 eq. 9): each child copies its parent's slot list and
// appends the parent's row as the slot of the previous depth.
#include <atomic>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace gdnbeam {

namespace {

constexpr int kTile = 256;           // codes per hint tile (the logits GEMM tile width)
constexpr int kFinalThreads = 1024;   // threads of a request's selection block
constexpr int kFinalSmemKeys = 16384; // candidates a selection block keeps on chip
constexpr int kRowThreads = 512;
constexpr int kReqThreads = 1024;
constexpr int kMaxSort = 4096;

__device__ __forceinline__ uint64_t make_key(uint32_t ord, uint32_t flat) {
  return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}

__device__ __forceinline__ float score(float cp, float zv, float l) {
  return __fadd_rn(cp, __fsub_rn(zv, l));
}

// Order-preserving integer keys of stored logits (larger value, larger key;
// NaN patterns sort beyond the infinities).
template <typename T> struct SKey;
template <> struct SKey<__nv_bfloat16> {
  static constexpr uint32_t kNegInf = 0x007Fu, kPosInf = 0xFF80u;
  static __device__ __forceinline__ float value(uint32_t k) {
    const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(b << 16);
  }
};
template <> struct SKey<float> {
  static constexpr uint32_t kNegInf = 0x007FFFFFu, kPosInf = 0xFF800000u;
  static __device__ __forceinline__ float value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
};

// The block of a request's cluster that filters listed tile i (the tile's
// index in the request's hint array): a multiplicative hash of i spread over
// `parts` blocks, so tiles of one code range do not all go to one block.
// A listed (row b, tile) pair is stored as b << tile_bits(n_tiles) | tile,
// so the filter splits it with a shift and a mask.
__device__ __forceinline__ int tile_bits(int n_tiles) {
  return n_tiles > 1 ? 32 - __clz(n_tiles - 1) : 0;
}
__device__ __forceinline__ int tile_owner(uint32_t i, int parts) {
  return (int)(((uint64_t)(i * 0x9E3779B1u) * (uint32_t)parts) >> 32);
}

// Blocks in this block's cluster (1 without a cluster launch).
__device__ __forceinline__ uint32_t cluster_nctas() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// Loads from the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t ld_cluster_u32(const void* p, uint32_t rank) {
  uint32_t v;
  const uint32_t a = tc::mapa_shared(tc::smem_u32(p), rank);
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_cluster_u64(const void* p, uint32_t rank) {
  uint64_t v;
  const uint32_t a = tc::mapa_shared(tc::smem_u32(p), rank);
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ float cum_prime(const float* cum, const float* bias, size_t row) {
  float cp = cum ? cum[row] : 0.0f;
  if (bias) cp = __fadd_rn(cp, bias[row]);
  return cp;
}

// Block-wide MSB-first radix search for the K-th largest of n keys read
// through get(). Returns prefix such that the keys >= prefix are the K
// largest (with ties at the K-th value all included when keys repeat).
// Needs hist[256] and sh[3] in shared memory.
template <typename Key, typename Get>
__device__ Key radix_kth(int n, unsigned K, Get get, unsigned* hist, unsigned* sh) {
  Key prefix = 0, mask = 0;
  unsigned remaining = K;
  for (int shift = 8 * (int)sizeof(Key) - 8; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      Key key = get(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(unsigned)(key >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // The highest bucket d >= 1 whose count from the top reaches
      // `remaining` (bucket 0 when none does): lane l scans buckets
      // 255 - 8l down to 248 - 8l after a warp scan of the lane totals.
      const int l = threadIdx.x;
      unsigned cnt[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        cnt[k] = hist[255 - 8 * l - k];
        tot += cnt[k];
      }
      unsigned incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += y;
      }
      const unsigned excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
      const int target = hit ? __ffs(hit) - 1 : 31;
      if (l == target) {
        unsigned above = excl;
        int d = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int bin = 255 - 8 * l - k;
          if (bin == 0 || above + cnt[k] >= remaining) {
            d = bin;
            break;
          }
          above += cnt[k];
        }
        sh[0] = (unsigned)d;
        sh[1] = remaining - above;
        sh[2] = (hist[d] == remaining - above) ? 1u : 0u;  // the whole bucket is taken
      }
    }
    __syncthreads();
    prefix |= (Key)sh[0] << shift;
    mask |= (Key)0xFF << shift;
    remaining = sh[1];
    const bool done = sh[2] != 0;
    __syncthreads();
    if (done) break;
  }
  return prefix;
}

// Sorts win[0..P) descending (P a power of two) and writes the first W_next.
__device__ void sort_and_emit(uint64_t* win, int P, int W_next, int V, int32_t* parents,
                              int32_t* tokens, float* cum_next) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        int j = i ^ stride;
        if (j > i) {
          bool desc = (i & size) == 0;
          uint64_t a = win[i], b = win[j];
          if (desc ? (a < b) : (a > b)) { win[i] = b; win[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < W_next; i += blockDim.x) {
    uint64_t key = win[i];
    uint32_t flat = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu);
    parents[i] = (int32_t)(flat / (uint32_t)V);
    tokens[i] = (int32_t)(flat % (uint32_t)V);
    cum_next[i] = from_orderable((uint32_t)(key >> 32));
  }
}

// Writes the W_next (<= kOrderMax) unique keys of win[] in descending order.
// Each warp sorts runs of 32 keys in registers (a bitonic network over
// shuffles) and writes them back; then each key's rank is its place in its
// run plus, for every other run, the count of that run's keys above it (a
// binary search in the sorted run). win must have room for the last run's
// padding up to a multiple of 32.
constexpr int kOrderMax = 1024;
__device__ void order_and_emit(uint64_t* win, int W_next, int V, int32_t* parents,
                               int32_t* tokens, float* cum_next) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  const int runs = (W_next + 31) >> 5;
  for (int run = warp; run < runs; run += n_warps) {
    const int i = run * 32 + lane;
    uint64_t v = i < W_next ? win[i] : 0ull;  // padding sorts below every key
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
        // blocks of k lanes alternate direction; the whole run ends descending
        const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
        v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
      }
    }
    win[i] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < W_next; i += blockDim.x) {
    const uint64_t key = win[i];
    const int mine = i >> 5;
    int rank = i & 31;
    for (int b = 0; b < runs; ++b) {
      if (b == mine) continue;
      const uint64_t* rb = win + 32 * b;
      int pos = 0;
#pragma unroll
      for (int st = 16; st > 0; st >>= 1)
        if (rb[pos + st - 1] > key) pos += st;
      if (rb[pos] > key) ++pos;
      rank += pos;
    }
    const uint32_t flat = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu);
    parents[rank] = (int32_t)(flat / (uint32_t)V);
    tokens[rank] = (int32_t)(flat % (uint32_t)V);
    cum_next[rank] = from_orderable((uint32_t)(key >> 32));
  }
}

__device__ __forceinline__ int high_bit(uint32_t x) { return 31 - __clz(x); }
__device__ __forceinline__ int high_bit(uint64_t x) { return 63 - __clzll(x); }

// Block-wide search for the K-th largest of n keys (read through get()),
// all of which lie in [lo, hi]. Each round histograms the keys inside the
// window on the 8 bits below the highest bit where its ends differ, keeps
// the bin that holds the K-th largest and narrows the window to it, until
// that bin is taken whole or holds a single value. Returns prefix such that
// the keys >= prefix are the K largest, ties at the K-th value all
// included. bins: kBins words of shared memory; sh: 4 words. Starting from
// the keys' own range skips the leading bits they all share, where fixed
// digits put nearly every key into one bucket.
constexpr int kBins = 256;
template <typename Key, typename Get>
__device__ Key radix_window(int n, unsigned K, Key lo, Key hi, Get get, unsigned* bins,
                            unsigned* sh) {
  unsigned remaining = K;  // rank of the target among the window's keys
  const int lane = threadIdx.x & 31;
  while (lo < hi) {
    const int p = high_bit(lo ^ hi);
    const int shift = p >= 7 ? p - 7 : 0;
    const Key base = lo >> shift;  // (hi >> shift) - base < kBins
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) bins[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const Key key = get(i);
      if (key >= lo && key <= hi) atomicAdd(&bins[(unsigned)((key >> shift) - base)], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the highest bin d whose count from the top of the window reaches
      // `remaining`; lane l owns bins 255 - 8l - k, k = 0..7
      unsigned cnt[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        cnt[k] = bins[kBins - 1 - 8 * lane - k];
        tot += cnt[k];
      }
      unsigned incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
      if (hit == 0u && lane == 0) sh[2] = 0xFFFFFFFFu;  // fewer keys than K in the window
      if (hit != 0u && lane == __ffs(hit) - 1) {
        unsigned acc = excl;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (acc + cnt[k] >= remaining) {
            sh[0] = (unsigned)(kBins - 1 - 8 * lane - k);
            sh[1] = remaining - acc;  // rank of the target within the bin
            sh[2] = cnt[k];
            break;
          }
          acc += cnt[k];
        }
      }
    }
    __syncthreads();
    const unsigned d = sh[0], rem = sh[1], c = sh[2];
    __syncthreads();  // everyone has read sh before the next round writes it
    if (c == 0xFFFFFFFFu) return lo;
    const Key blo = (base + (Key)d) << shift;
    const Key bhi = ((base + (Key)d + 1) << shift) - 1;  // wraps to the top at the last bin
    const Key nlo = blo > lo ? blo : lo;
    if (c == rem) return nlo;  // the whole bin is taken
    lo = nlo;
    hi = bhi < hi ? bhi : hi;
    remaining = rem;
  }
  return lo;
}

struct SelScratch {
  int* fb_flag;     // [R] request needs the fallback
  int* fb_any;      // [1] some request needs the fallback (reset by the fallback's last kernel)
  uint64_t* pre;    // [R*W_t][K] fallback precut keys
  float2* hint;     // [R*W_t][n_tiles] tile maxima computed here when not supplied
  uint32_t* tlist;  // [R][cap_tiles] (row, tile) pairs whose maximum reaches the bound, b << tile_bits | tile
  float* cut;       // [R*W_t] rows' cutoff logits, when the rows do not fit on chip
  int cap;          // candidates a request may keep on chip before the bound is narrowed
  int cap_tiles;
};

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// Room for the listed tiles of one request: every (row, tile) pair, so the
// list never overflows and always holds every tile that can hold one of the
// W best (4 bytes per pair, 1/128 of the bf16 logits).
int cap_tiles_of(int W_t, int W_next, int V) {
  (void)W_next;
  return W_t * ((V + kTile - 1) / kTile);
}

int cap_of(int W_t, int W_next, int V) {
  long long cap = 16LL * W_next;
  if (cap < V) cap = V;
  if (cap > (long long)W_t * V) cap = (long long)W_t * V;
  return (int)cap;
}

SelScratch carve_sel(void* base, int R, int W_t, int W_next, int V, size_t* total) {
  SelScratch s{};
  const int K = W_next < V ? W_next : V;
  const int n_tiles = (V + kTile - 1) / kTile;
  s.cap = cap_of(W_t, W_next, V);
  s.cap_tiles = cap_tiles_of(W_t, W_next, V);
  char* p = (char*)base;
  size_t off = 0;
  auto take = [&](size_t b) { char* q = p ? p + off : nullptr; off += a256(b); return q; };
  s.fb_flag = (int*)take((size_t)R * 4);
  s.fb_any = (int*)take(16);
  s.pre = (uint64_t*)take((size_t)R * W_t * K * 8);
  s.hint = (float2*)take((size_t)R * W_t * n_tiles * sizeof(float2));
  s.tlist = (uint32_t*)take((size_t)R * s.cap_tiles * 4);
  s.cut = (float*)take((size_t)R * W_t * 4);
  if (total) *total = off;
  return s;
}

// ---- hint pre-pass: the maximum stored logit of every (row, 256-code tile)
template <typename T>
__global__ void tile_max_kernel(int n, int V, int n_tiles, const T* __restrict__ z,
                                float2* __restrict__ hint, unsigned* err) {
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)n * n_tiles) return;
  const int row = (int)(w / n_tiles), tile = (int)(w % n_tiles);
  const T* zr = z + (size_t)row * V + (size_t)tile * kTile;
  const int cnt = min(kTile, V - tile * kTile);
  float mx = -INFINITY;
  bool bad = false;
  for (int c = lane; c < cnt; c += 32) {
    const float zv = ldf(zr + c);
    bad |= !isfinite(zv);
    mx = fmaxf(mx, zv);
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) hint[w] = make_float2(mx, 0.0f);
  if (bad) raise_error(err, GDNBEAM_DERR_NONFINITE);
}

// ---- bound: the W_next-th largest hint score of request r, and the tiles
// that can hold a candidate. A code scores at most its tile's maximum (the
// score is monotone in the stored logit within a row), so only tiles whose
// maximum reaches the bound are listed. Writes the rows' parameters and
// ss.tlist of the request (the list also to slist, up to slist_cap entries)
// and returns the bound, the largest hint key and the list length (the same
// in every thread); hkeys holds smem_keys 32-bit keys.
struct Bound {
  uint32_t t, hmax;
  int n_list;  // tiles reaching the bound
  int n_own;   // of them, this block's share (tile_owner == part)
};

// Per-row parameters of a request: cum' and lse, and the row's cutoff logit
// once the bound is known. They sit in shared memory (cum', lse, cutoff, -)
// when the request's rows fit, else they are read from global memory and the
// cutoffs kept in ss.cut.
constexpr int kSmemRows = 4000;

struct Rows {
  float4* s;  // [W_t] on chip, or null
  const float *lse, *cum, *bias;
  float* cut;
  size_t base;  // the request's first row
  __device__ __forceinline__ float4 get(int b) const {
    if (s) return s[b];
    const size_t row = base + b;
    return make_float4(cum_prime(cum, bias, row), lse[row], cut[row], 0.0f);
  }
  __device__ __forceinline__ void set_cut(int b, float c) const {
    if (s) s[b].z = c; else cut[base + b] = c;
  }
};

template <typename T>
__device__ Bound bound_phase(int r, int W_t, int n_tiles, int W_next,
                            const float2* __restrict__ hint, const Rows& rows,
                            const SelScratch& ss, uint32_t* hkeys, int smem_keys, uint32_t* slist,
                            int slist_cap, unsigned* bins, int part, int parts, unsigned* err) {
  __shared__ unsigned sh[4];
  __shared__ int s_cnt, s_own;
  __shared__ uint32_t s_wlo[32], s_whi[32];
  const int n_h = W_t * n_tiles;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_own = 0;
  }
  // the rows' parameters; a row whose lse or cumulative score is not finite
  // is flagged
  for (int b = threadIdx.x; b < W_t; b += blockDim.x) {
    const size_t row = rows.base + b;
    const float cp = cum_prime(rows.cum, rows.bias, row), l = rows.lse[row];
    if (!isfinite(l) || !isfinite(cp)) raise_error(err, GDNBEAM_DERR_NONFINITE);
    if (rows.s) rows.s[b] = make_float4(cp, l, 0.0f, 0.0f);
  }
  __syncthreads();
  auto key_of = [&](int i) -> uint32_t {
    const int b = i / n_tiles;
    const float4 rp = rows.get(b);
    const float zm = hint[(rows.base + b) * n_tiles + (i % n_tiles)].x;
    const float zs = St<T>::to_f(St<T>::from_f(zm));
    return orderable(score(rp.x, zs, rp.y));
  };
  // the hint keys (kept on chip when they fit) and the block's smallest and
  // largest, which bound the search below
  // Each thread issues eight hint loads before it uses any: the hints are
  // mostly not in L2 (the logits were written after them), and eight misses
  // in flight per thread instead of one cut this pass by more than half.
  const bool on_chip = n_h <= smem_keys;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  const float2* hreq = hint + rows.base * n_tiles;
  for (int i0 = threadIdx.x; i0 < n_h; i0 += 8 * blockDim.x) {
    float zm[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      zm[u] = i < n_h ? hreq[i].x : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n_h) {
        const float4 rp = rows.get(i / n_tiles);
        const float zs = St<T>::to_f(St<T>::from_f(zm[u]));  // stored value of the tile's top element
        const uint32_t key = orderable(score(rp.x, zs, rp.y));
        if (on_chip) hkeys[i] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    s_wlo[threadIdx.x >> 5] = kmin;
    s_whi[threadIdx.x >> 5] = kmax;
  }
  __syncthreads();
  uint32_t klo = 0xFFFFFFFFu, khi = 0u;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    klo = min(klo, s_wlo[w]);
    khi = max(khi, s_whi[w]);
  }
  uint32_t t = 0u;  // too few hints for a bound: keep every tile
  if (W_next <= n_h) {
    if (on_chip)
      t = radix_window<uint32_t>(n_h, (unsigned)W_next, klo, khi, [&](int i) { return hkeys[i]; },
                                 bins, sh);
    else
      t = radix_window<uint32_t>(n_h, (unsigned)W_next, klo, khi, key_of, bins, sh);
  }
  // the tiles whose hint reaches t: all of them to the request's list in
  // global memory (written by block part 0 alone), this block's share to its
  // on-chip list (every tile when parts = 1)
  uint32_t* list = ss.tlist + (size_t)r * ss.cap_tiles;
  // thread i's (row, tile) = (i / n_tiles, i % n_tiles), stepped along
  // with i (one division per thread)
  const int tb = tile_bits(n_tiles);
  const int db = (int)blockDim.x / n_tiles, dt = (int)blockDim.x % n_tiles;
  int cb = (int)threadIdx.x / n_tiles, ct = (int)threadIdx.x % n_tiles;
  auto step_bt = [&]() {
    cb += db;
    ct += dt;
    if (ct >= n_tiles) { ct -= n_tiles; ++cb; }
  };
  if (parts == 1) {
    for (int i = threadIdx.x; i < n_h; i += blockDim.x, step_bt()) {
      if ((on_chip ? hkeys[i] : key_of(i)) >= t) {
        const uint32_t e = ((uint32_t)cb << tb) | (uint32_t)ct;
        const int pos = atomicAdd(&s_cnt, 1);
        if (pos < ss.cap_tiles) list[pos] = e;
        if (pos < slist_cap) slist[pos] = e;  // the on-chip copy, when it fits
      }
    }
  } else {
    int mine = 0;  // listed tiles this thread saw (the other blocks count them too)
    for (int i = threadIdx.x; i < n_h; i += blockDim.x, step_bt()) {
      if ((on_chip ? hkeys[i] : key_of(i)) >= t) {
        const uint32_t e = ((uint32_t)cb << tb) | (uint32_t)ct;
        ++mine;
        if (part == 0) {
          const int pos = atomicAdd(&s_cnt, 1);
          if (pos < ss.cap_tiles) list[pos] = e;
        }
        if (tile_owner(e, parts) == part) {
          const int q = atomicAdd(&s_own, 1);
          if (q < slist_cap) slist[q] = e;
        }
      }
    }
    if (part != 0) {
      for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
      if (lane == 0 && mine) atomicAdd(&s_cnt, mine);
    }
  }
  // each row's cutoff: the smallest stored value whose score reaches t, by
  // bisection over the storage keys (scores are monotone in the stored
  // value within a row); NaN when no code of the row can qualify
  for (int b = threadIdx.x; b < W_t; b += blockDim.x) {
    const float4 rp = rows.get(b);
    const float cp = rp.x, l = rp.y;
    uint32_t lo = SKey<T>::kNegInf, hi = SKey<T>::kPosInf + 1u;  // hi: none reaches t
    while (lo < hi) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      if (orderable(score(cp, SKey<T>::value(mid), l)) >= t) hi = mid; else lo = mid + 1u;
    }
    rows.set_cut(b, SKey<T>::value(lo));
  }
  __syncthreads();  // the list, the cutoffs and the counters are complete
  return Bound{t, khi, s_cnt, s_own};
}

// Eight stored codes as loaded: one 16-byte word of bf16, two of fp32.
template <typename T> struct Codes8;
template <> struct Codes8<__nv_bfloat16> {
  uint4 w;
  __device__ __forceinline__ void load(const __nv_bfloat16* __restrict__ zr, int v0, int V, bool vec) {
    if (vec && v0 + 8 <= V) {
      w = __ldg(reinterpret_cast<const uint4*>(zr + v0));
    } else {
      uint16_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = v0 + e < V ? __bfloat16_as_ushort(zr[v0 + e]) : (uint16_t)0x7FC0u;
      w = make_uint4(h[0] | (uint32_t)h[1] << 16, h[2] | (uint32_t)h[3] << 16,
                     h[4] | (uint32_t)h[5] << 16, h[6] | (uint32_t)h[7] << 16);
    }
  }
  __device__ __forceinline__ float at(int e) const {
    const uint32_t x = e < 2 ? w.x : e < 4 ? w.y : e < 6 ? w.z : w.w;
    return __uint_as_float(((x >> (16 * (e & 1))) & 0xFFFFu) << 16);
  }
};
template <> struct Codes8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* __restrict__ zr, int v0, int V, bool vec) {
    if (vec && v0 + 8 <= V) {
      a = __ldg(reinterpret_cast<const float4*>(zr + v0));
      b = __ldg(reinterpret_cast<const float4*>(zr + v0 + 4));
    } else {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = v0 + e < V ? zr[v0 + e] : __int_as_float(0x7FC00000);
      a = make_float4(f[0], f[1], f[2], f[3]);
      b = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  __device__ __forceinline__ float at(int e) const {
    const float4& q = e < 4 ? a : b;
    const int k = e & 3;
    return k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w;
  }
};

// Visits the listed tiles of a request (list: n_list entries, on chip or in
// global memory) with the whole block, one warp per tile, several tiles per
// warp at a time so their loads overlap. Each lane compares its eight codes
// with the row's cutoff. A tile with few codes reaching it (the usual case)
// has each lane call f(o, flat) for each of its codes, with the code's score
// key and flat index, independently of the other lanes. A tile dense with
// them (scores dominated by the row's parent) has every lane of the warp call
// dense(hits, o, flat0) together, with its hit mask and the hits' keys.
constexpr int kDenseHits = 32;

template <typename T, typename F, typename D>
__device__ __forceinline__ void for_listed_codes(int V, int n_tiles, int n_list, const uint32_t* list,
                                                 const T* __restrict__ z, const Rows& rows, F&& f,
                                                 D&& dense, int part = 0, int parts = 1) {
  constexpr int EPL = kTile / 32;
  constexpr int U = sizeof(T) == 2 ? 6 : 3;  // tiles in flight per warp
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const bool vec = (V % 8) == 0 && ((uintptr_t)z & 15) == 0;
  const int tb = tile_bits(n_tiles);
  const uint32_t tmask = (1u << tb) - 1u;
  for (int j0 = (threadIdx.x >> 5) * U; j0 < n_list; j0 += warps * U) {
    uint32_t ids[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      ids[u] = j0 + u < n_list ? list[j0 + u] : 0xFFFFFFFFu;
      // with parts > 1, only tiles whose id falls in this block's share
      if (parts > 1 && ids[u] != 0xFFFFFFFFu && tile_owner(ids[u], parts) != part)
        ids[u] = 0xFFFFFFFFu;
    }
    Codes8<T> zc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ids[u] == 0xFFFFFFFFu) continue;
      const int b = (int)(ids[u] >> tb), tile = (int)(ids[u] & tmask);
      zc[u].load(z + (rows.base + b) * (size_t)V, tile * kTile + lane * EPL, V, vec);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ids[u] == 0xFFFFFFFFu) continue;
      const int b = (int)(ids[u] >> tb), tile = (int)(ids[u] & tmask);
      const float4 rp = rows.get(b);
      unsigned hits = 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if (zc[u].at(e) >= rp.z) hits |= 1u << e;  // NaN never compares true
      const uint32_t flat0 = (uint32_t)b * (uint32_t)V + (uint32_t)(tile * kTile + lane * EPL);
      // warp-uniform: the same tile in every lane
      if (__reduce_add_sync(0xffffffffu, (unsigned)__popc(hits)) > (unsigned)kDenseHits) {
        uint32_t o[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = (hits >> e) & 1u ? orderable(score(rp.x, zc[u].at(e), rp.y)) : 0u;
        dense(hits, o, flat0);
        continue;
      }
      while (hits) {
        const int e = __ffs(hits) - 1;
        hits &= hits - 1u;
        f(orderable(score(rp.x, zc[u].at(e), rp.y)), flat0 + (uint32_t)e);
      }
    }
  }
}

// Writes the 64-bit selection keys of every listed code whose score key
// reaches lo into keys[0 .. target) and returns how many there are (those
// past target are counted, not written).
template <typename T>
__device__ int append_listed(int V, int n_tiles, int n_list, const uint32_t* list, uint32_t lo,
                             int target, const T* __restrict__ z, const Rows& rows, uint64_t* keys,
                             int part = 0, int parts = 1) {
  __shared__ unsigned s_cnt;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_cnt = 0u;
  __syncthreads();
  auto put = [&](unsigned pos, uint32_t o, uint32_t flat) {
    if (pos < (unsigned)target) keys[pos] = make_key(o, flat);
  };
  for_listed_codes<T>(
      V, n_tiles, n_list, list, z, rows,
      [&](uint32_t o, uint32_t flat) {
        if (o >= lo) put(atomicAdd(&s_cnt, 1u), o, flat);
      },
      [&](unsigned hits, const uint32_t (&o)[kTile / 32], uint32_t flat0) {
        // one atomic per warp: the lanes' places from a scan of their counts
        unsigned keep = 0;
#pragma unroll
        for (int e = 0; e < kTile / 32; ++e)
          if (((hits >> e) & 1u) && o[e] >= lo) keep |= 1u << e;
        const unsigned mine = (unsigned)__popc(keep);
        unsigned incl = mine;
#pragma unroll
        for (int q = 1; q < 32; q <<= 1) {
          const unsigned y = __shfl_up_sync(0xffffffffu, incl, q);
          if (lane >= q) incl += y;
        }
        unsigned pos = 0;
        if (lane == 31 && incl) pos = atomicAdd(&s_cnt, incl);
        pos = __shfl_sync(0xffffffffu, pos, 31) + incl - mine;
#pragma unroll
        for (int e = 0; e < kTile / 32; ++e)
          if ((keep >> e) & 1u) put(pos++, o[e], flat0 + (uint32_t)e);
      },
      part, parts);
  __syncthreads();
  return (int)s_cnt;
}

// ---- narrowing: more codes reach the bound than fit on chip. Raises the
// bound from t until at most `target` listed codes reach it (and still at
// least W_next). Each round histograms the score keys inside the window
// [lo, hi] on the 11 bits below the highest bit where lo and hi differ,
// counts the codes above hi, and keeps the bin holding the W_next-th
// largest. Returns false when more codes tie at one score than fit.
constexpr int kRefineBins = 2048;
static_assert(kRefineBins * 4 <= kFinalSmemKeys * 8, "the bins live in the final block's key area");

template <typename T>
__device__ bool narrow_bound(int V, int n_tiles, int n_list, const uint32_t* list, int W_next,
                             int target, const T* __restrict__ z, const Rows& rows, uint32_t* bins,
                             uint32_t t, uint32_t hmax, uint32_t* lo_out) {
  __shared__ unsigned s_above, s_res[4];
  const int lane = threadIdx.x & 31;
  uint32_t lo = t, hi = hmax;
  for (int round = 0; round < 8 && lo <= hi; ++round) {
    const int p = lo == hi ? 0 : 31 - __clz(lo ^ hi);
    const int shift = p >= 10 ? p - 10 : 0;
    const uint32_t base = lo >> shift;  // (hi >> shift) - base < kRefineBins
    for (int i = threadIdx.x; i < kRefineBins; i += blockDim.x) bins[i] = 0u;
    if (threadIdx.x == 0) s_above = 0u;
    __syncthreads();
    for_listed_codes<T>(
        V, n_tiles, n_list, list, z, rows,
        [&](uint32_t o, uint32_t) {
          if (o > hi) atomicAdd(&s_above, 1u);
          else if (o >= lo) atomicAdd(&bins[(o >> shift) - base], 1u);
        },
        [&](unsigned hits, const uint32_t (&o)[kTile / 32], uint32_t) {
          unsigned over = 0;
#pragma unroll
          for (int e = 0; e < kTile / 32; ++e) {
            if (!((hits >> e) & 1u)) continue;
            if (o[e] > hi) ++over;
            else if (o[e] >= lo) atomicAdd(&bins[(o[e] >> shift) - base], 1u);
          }
          over = __reduce_add_sync(0xffffffffu, over);
          if (lane == 0 && over) atomicAdd(&s_above, over);
        });
    __syncthreads();
    if (threadIdx.x < 32) {
      // highest bin d whose count from the top of the window reaches the
      // remaining rank; lane l owns bins 2047 - 64 l - k, k = 0..63
      const unsigned above = s_above;
      const unsigned remaining = above < (unsigned)W_next ? (unsigned)W_next - above : 0u;
      unsigned tot = 0;
      for (int k = 0; k < 64; ++k) tot += bins[kRefineBins - 1 - 64 * lane - ((k + lane) & 63)];
      unsigned incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, remaining > 0 && excl < remaining && incl >= remaining);
      if (lane == 0) s_res[3] = hit ? 1u : 0u;
      if (hit && lane == __ffs(hit) - 1) {
        unsigned acc = excl;
        for (int k = 0; k < 64; ++k) {
          const int bin = kRefineBins - 1 - 64 * lane - k;
          const unsigned c = bins[bin];
          if (acc + c >= remaining) {
            s_res[0] = (unsigned)bin;
            s_res[1] = acc;  // codes of the window above bin
            s_res[2] = c;
            break;
          }
          acc += c;
        }
      }
    }
    __syncthreads();
    if (!s_res[3]) return false;  // fewer than W_next codes reach lo: bound inconsistent
    const uint32_t d = s_res[0];
    const unsigned total = s_above + s_res[1] + s_res[2];
    const uint32_t blo = max(lo, (uint32_t)((uint64_t)(base + d) << shift));
    const uint32_t bhi = min(hi, (uint32_t)(((uint64_t)(base + d + 1) << shift) - 1));
    __syncthreads();  // everyone has read s_res and the bins
    lo = blo;
    if (total <= (unsigned)target) {
      *lo_out = lo;
      return true;
    }
    if (blo == bhi) return false;  // more codes tie at one score than fit
    hi = bhi;
  }
  return false;
}

// ---- the fast path, one block per request: the bound, the candidates of
// the listed tiles (narrowing the bound if they do not fit on chip), and
// their exact top-W_next, sorted. A request it cannot finish is flagged for
// the exact fallback.
template <typename T>
__global__ void __launch_bounds__(kFinalThreads) select_fused_kernel(
    int W_t, int V, int n_tiles, int W_next, const float2* __restrict__ hint,
    const T* __restrict__ z, const float* __restrict__ lse, const float* __restrict__ cum,
    const float* __restrict__ bias, SelScratch ss, int bound_keys, int rows_on_chip,
    int32_t* __restrict__ parents, int32_t* __restrict__ tokens, float* __restrict__ cum_next,
    unsigned* err) {
  // first the bound's hint keys (32-bit), then the candidates' keys (64-bit);
  // after them the rows' parameters when they fit
  extern __shared__ uint64_t keys[];
  __shared__ unsigned sh[4];
  __shared__ uint64_t win[kMaxSort];
  __shared__ int s_nloc;
  // A request runs on one block, or on a cluster of csize blocks when
  // requests are fewer than the SMs: every block computes the same bound,
  // each filters its share of the listed tiles (tile_owner), and the
  // first block gathers the others' candidates from their shared memory and
  // finishes the selection alone.
  const int csize = (int)cluster_nctas();
  const int rank = (int)tc::cluster_ctarank();
  const int r = blockIdx.x / csize;
  // the tile list is kept on chip in the sort window (idle until the end)
  // when it fits
  uint32_t* slist = reinterpret_cast<uint32_t*>(win);
  constexpr int kSlist = 2 * kMaxSort;
  const Rows rows{rows_on_chip ? reinterpret_cast<float4*>(keys + kFinalSmemKeys) : nullptr, lse, cum,
                  bias, ss.cut, (size_t)r * W_t};
  // the radix bins share the sort window too: the bound's search ends
  // before the tile list is written there, and the top-W search before the
  // window is filled
  unsigned* bins = reinterpret_cast<unsigned*>(win);
  const Bound bd = bound_phase<T>(r, W_t, n_tiles, W_next, hint, rows, ss,
                                  reinterpret_cast<uint32_t*>(keys), bound_keys, slist, kSlist,
                                  bins, rank, csize, err);
  const uint32_t t = bd.t, hmax = bd.hmax;
  const int n_tc = bd.n_list;
  const int n_list = min(n_tc, ss.cap_tiles);
  // the whole list: on chip with one block per request when it fits, else
  // the copy in global memory
  const uint32_t* full = ss.tlist + (size_t)r * ss.cap_tiles;
  const bool on_chip_list = n_list <= kSlist;  // the same in every block of the cluster
  const uint32_t* list = on_chip_list && csize == 1 ? slist : full;
  const int target = min(ss.cap, kFinalSmemKeys);
  int n_c;
  if (csize == 1) {
    n_c = append_listed<T>(V, n_tiles, n_list, list, t, target, z, rows, keys);
  } else {
    // this block's share: its on-chip list, or the global list (written by
    // block 0, complete once the cluster has met) with the other tiles skipped
    if (!on_chip_list) tc::cluster_sync();
    n_c = on_chip_list
              ? append_listed<T>(V, n_tiles, bd.n_own, slist, t, target, z, rows, keys)
              : append_listed<T>(V, n_tiles, n_list, full, t, target, z, rows, keys, rank, csize);
    if (threadIdx.x == 0) s_nloc = n_c;
    tc::cluster_sync();  // every block's candidates are in its shared memory
    if (rank == 0) {
      int total = n_c;
      for (int q = 1; q < csize; ++q) total += (int)ld_cluster_u32(&s_nloc, q);
      if (total <= target) {
        int off = n_c;
        for (int q = 1; q < csize; ++q) {
          const int nq = (int)ld_cluster_u32(&s_nloc, q);
          for (int i = threadIdx.x; i < nq; i += blockDim.x) keys[off + i] = ld_cluster_u64(&keys[i], q);
          off += nq;
        }
      }
      n_c = total;  // above target: narrowed below over the whole list
    }
    tc::cluster_sync();  // block 0 has read the others' candidates
    if (rank != 0) return;
  }
  uint32_t lo_key = t;
  if (n_c > target && n_c >= W_next && n_tc <= ss.cap_tiles) {
    n_c = narrow_bound<T>(V, n_tiles, n_list, list, W_next, target, z, rows,
                          reinterpret_cast<uint32_t*>(keys), t, hmax, &lo_key)
              ? append_listed<T>(V, n_tiles, n_list, list, lo_key, target, z, rows, keys)
              : -1;
  }
  if (n_c < W_next || n_c > target || n_tc > ss.cap_tiles) {
    if (threadIdx.x == 0) {
      ss.fb_flag[r] = 1;
      atomicOr(ss.fb_any, 1);
    }
    return;
  }
  if (threadIdx.x == 0) ss.fb_flag[r] = 0;
  // every kept key has a score key of at least lo_key (the bound, raised if
  // narrowed) and at most the largest hint key
  uint64_t prefix = 0;
  if (W_next < n_c)
    prefix = radix_window<uint64_t>(n_c, (unsigned)W_next, (uint64_t)lo_key << 32,
                                    ((uint64_t)hmax << 32) | 0xFFFFFFFFull,
                                    [&](int i) { return keys[i]; }, bins, sh);
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  // the keys >= prefix are exactly the W_next best (keys are unique); they
  // go to the window a warp at a time
  const int lane = threadIdx.x & 31;
  for (int i0 = threadIdx.x & ~31; i0 < n_c; i0 += blockDim.x) {
    const int i = i0 + lane;
    const uint64_t key = i < n_c ? keys[i] : 0ull;
    const bool keep = i < n_c && key >= prefix;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (m == 0u) continue;
    unsigned pos = 0;
    if (lane == 0) pos = atomicAdd(&sh[3], (unsigned)__popc(m));
    pos = __shfl_sync(0xffffffffu, pos, 0) + (unsigned)__popc(m & ((1u << lane) - 1u));
    if (keep && pos < (unsigned)W_next) win[pos] = key;
  }
  __syncthreads();
  const size_t o = (size_t)r * W_next;
  if (W_next <= kOrderMax) {
    order_and_emit(win, W_next, V, parents + o, tokens + o, cum_next + o);
  } else {
    int P = 1;
    while (P < W_next) P <<= 1;
    for (int i = W_next + threadIdx.x; i < P; i += blockDim.x) win[i] = 0;  // below every key
    __syncthreads();
    sort_and_emit(win, P, W_next, V, parents + o, tokens + o, cum_next + o);
  }
}

// ---- fallback stage 1: per-row local top-K (rows of flagged requests only)
template <typename T>
__global__ void __launch_bounds__(kRowThreads) select_rowcut_kernel(
    int n_rows, int W_t, int V, int K, const T* __restrict__ logits, const float* __restrict__ lse,
    const float* __restrict__ cum, const float* __restrict__ bias, SelScratch ss, unsigned* err) {
  extern __shared__ uint64_t rkeys[];  // [V]
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[4];
  if (*(volatile int*)ss.fb_any == 0) return;
  for (int row = blockIdx.x; row < n_rows; row += gridDim.x) {
    if (!ss.fb_flag[row / W_t]) continue;
    const int b = row % W_t;
    const float l = lse[row];
    const float cp = cum_prime(cum, bias, row);
    const T* zr = logits + (size_t)row * V;
    __syncthreads();
    for (int v = threadIdx.x; v < V; v += blockDim.x)
      rkeys[v] = make_key(orderable(score(cp, ldf(zr + v), l)), (uint32_t)b * (uint32_t)V + (uint32_t)v);
    if (threadIdx.x == 0) sh[3] = 0;
    __syncthreads();
    uint64_t* out = ss.pre + (size_t)row * K;
    if (K >= V) {
      for (int v = threadIdx.x; v < V; v += blockDim.x) out[v] = rkeys[v];
      continue;
    }
    const uint64_t prefix = radix_kth<uint64_t>(V, (unsigned)K, [&](int i) { return rkeys[i]; }, hist, sh);
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      uint64_t key = rkeys[v];
      if (key >= prefix) {
        unsigned idx = atomicAdd(&sh[3], 1u);
        if (idx < (unsigned)K) out[idx] = key;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && sh[3] != (unsigned)K) raise_error(err, GDNBEAM_DERR_SELECT);
  }
}

// ---- fallback stage 2: request-level top-W_next among the precut keys
__global__ void __launch_bounds__(kReqThreads) select_request_kernel(
    int W_t, int K, int W_next, int V, SelScratch ss, int32_t* __restrict__ parents,
    int32_t* __restrict__ tokens, float* __restrict__ cum_next, unsigned* err) {
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[4];
  __shared__ uint64_t win[kMaxSort];
  const int r = blockIdx.x;
  // the row precut has read the flag: clear it for the next selection
  if (r == 0 && threadIdx.x == 0) *ss.fb_any = 0;
  if (!ss.fb_flag[r]) return;
  const int n = W_t * K;
  const uint64_t* c = ss.pre + (size_t)r * n;
  auto get = [&](int i) { return c[i]; };
  uint64_t prefix = 0;
  if (W_next < n) prefix = radix_kth<uint64_t>(n, (unsigned)W_next, get, hist, sh);
  int P = 1;
  while (P < W_next) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) win[i] = 0;
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    uint64_t key = c[i];
    if (key >= prefix) {
      unsigned idx = atomicAdd(&sh[3], 1u);
      if (idx < (unsigned)W_next) win[idx] = key;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh[3] != (unsigned)W_next) raise_error(err, GDNBEAM_DERR_SELECT);
  const size_t o = (size_t)r * W_next;
  sort_and_emit(win, P, W_next, V, parents + o, tokens + o, cum_next + o);
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

template <typename T>
int run_select(int R, int W_t, int W_next, int V, const T* z, const float* lse, const float* cum,
               const float* bias, const float2* hint, int32_t* parents, int32_t* tokens,
               float* cum_next, void* scratch, unsigned* err, cudaStream_t s) {
  const int K = W_next < V ? W_next : V;
  const int n = R * W_t;
  const int n_tiles = (V + kTile - 1) / kTile;
  SelScratch ss = carve_sel(scratch, R, W_t, W_next, V, nullptr);
  if (!hint) {
    const long long warps = (long long)n * n_tiles;
    tile_max_kernel<T><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(n, V, n_tiles, z, ss.hint, err);
    GDN_LAUNCH_CHECK();
    hint = ss.hint;
  }
  // bound, filter and exact top-W of each request in one block
  const int n_h = W_t * n_tiles;
  const int bound_keys = n_h <= 2 * kFinalSmemKeys ? n_h : 0;  // 32-bit keys in the key area
  const int rows_on_chip = W_t <= kSmemRows ? 1 : 0;
  const size_t fused_smem = (size_t)kFinalSmemKeys * 8 + (rows_on_chip ? (size_t)W_t * 16 : 0);
  GDN_CUDA(cudaFuncSetAttribute(select_fused_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)fused_smem));
  // a cluster of blocks per request while requests are fewer than the SMs
  int csize = 1;
  while (csize < 4 && (long long)R * csize * 2 <= sm_count()) csize *= 2;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * csize), 1, 1);
    cfg.blockDim = dim3(kFinalThreads, 1, 1);
    cfg.dynamicSmemBytes = fused_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)csize;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    GDN_CUDA(cudaLaunchKernelEx(&cfg, select_fused_kernel<T>, W_t, V, n_tiles, W_next, hint, z, lse,
                                cum, bias, ss, bound_keys, rows_on_chip, parents, tokens, cum_next,
                                err));
  }
  GDN_LAUNCH_CHECK();
  // exact fallback for requests whose buffer was short or overflowed
  const size_t row_smem = (size_t)V * 8;
  GDN_CUDA(cudaFuncSetAttribute(select_rowcut_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)row_smem));
  const int rc_grid = n < sm_count() ? n : sm_count();  // one wave: cheap when it exits at once
  select_rowcut_kernel<T><<<rc_grid, kRowThreads, row_smem, s>>>(n, W_t, V, K, z, lse, cum, bias,
                                                                 ss, err);
  GDN_LAUNCH_CHECK();
  select_request_kernel<<<R, kReqThreads, 0, s>>>(W_t, K, W_next, V, ss, parents, tokens, cum_next,
                                                  err);
  GDN_LAUNCH_CHECK();
  return GDNBEAM_OK;
}

}  // namespace

int sm_count() {
  static std::atomic<int> sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 132;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

size_t select_scratch_bytes(int R, int W_t, int W_next, int V) {
  size_t total = 0;
  carve_sel(nullptr, R, W_t, W_next, V, &total);
  return total;
}

int launch_select(int R, int W_t, int W_next, int V, int dtype, const void* logits,
                  const float* lse, const float* cum, const float* bias, const float2* hint,
                  int32_t* parents, int32_t* tokens, float* cum_next, void* scratch,
                  unsigned* err, cudaStream_t s) {
  if (W_next > kMaxSort || V > 16384) return GDNBEAM_EUNSUPPORTED;
  if (dtype == GDNBEAM_BF16)
    return run_select<__nv_bfloat16>(R, W_t, W_next, V, (const __nv_bfloat16*)logits, lse, cum,
                                     bias, hint, parents, tokens, cum_next, scratch, err, s);
  return run_select<float>(R, W_t, W_next, V, (const float*)logits, lse, cum, bias, hint, parents,
                           tokens, cum_next, scratch, err, s);
}

int launch_tile_max(int dtype, int n, int V, const void* z, float2* hint, unsigned* err,
                    cudaStream_t s) {
  const int n_tiles = (V + kTile - 1) / kTile;
  const long long warps = (long long)n * n_tiles;
  if (warps == 0) return GDNBEAM_OK;
  if (dtype == GDNBEAM_BF16)
    tile_max_kernel<__nv_bfloat16><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(
        n, V, n_tiles, (const __nv_bfloat16*)z, hint, err);
  else
    tile_max_kernel<float><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(n, V, n_tiles,
                                                                      (const float*)z, hint, err);
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
