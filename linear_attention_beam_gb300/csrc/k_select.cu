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
// Fast path (one read of the logits):
//   bound   per request, the scores of one real candidate per (row, 256-code
//           tile) — the tile maximum, which the logits GEMM already produces
//           for the log-normaliser — and the W-th largest of them, tau;
//   filter  every candidate with s >= tau is appended to the request's buffer;
//   final   exact top-W of the buffer by radix search on the keys, sorted.
// If the buffer holds at least W candidates, every candidate left out scores
// below the W-th largest kept one, so the result is exact whatever tau was.
// tau is the score of a real candidate, so at least W candidates reach it and
// the W best all lie in listed tiles. When more candidates reach tau than the
// buffer holds (scores dominated by a few parents, every code of whose rows
// clears the bound), the final kernel narrows the bound over the listed
// tiles' codes by an 11-bit radix histogram of the 32-bit score keys until
// the codes reaching it fit, then refills the buffer: still exact.
// A request that cannot be narrowed (more candidates tie at one score than
// the buffer holds) falls back to the two exact stages of RecoGEM §4.3: a
// per-row precut to the local top-K (K = min(W, V)), then a request-level
// selection among the survivors; a candidate the precut drops is beaten by K
// candidates of its own row.
//
// Ancestry (OneLA §2.4 eq. 9): each child copies its parent's slot list and
// appends the parent's row as the slot of the previous depth.
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

namespace {

constexpr int kTile = 256;           // codes per hint tile (the logits GEMM tile width)
constexpr int kBoundThreads = 1024;
constexpr int kFilterThreads = 256;
constexpr int kFilterBlocksPerReq = 32;  // 256 warps share a request's listed tiles
constexpr int kFinalThreads = 1024;
constexpr int kFinalSmemKeys = 16384; // candidates a final block keeps on chip
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

struct SelScratch {
  int* count;       // [R] candidates appended by the filter
  uint32_t* thr;    // [R] orderable score bound
  int* fb_flag;     // [R] request needs the fallback
  int* fb_any;      // [1]
  uint64_t* cand;   // [R][cap]
  uint64_t* pre;    // [R*W_t][K] fallback precut keys
  float2* hint;     // [R*W_t][n_tiles] tile maxima computed here when not supplied
  int* tcount;      // [R] (row, tile) pairs whose tile maximum reaches the bound
  uint32_t* tlist;  // [R][cap_tiles] those pairs, as b * n_tiles + tile
  float* cut;       // [R*W_t] per row the smallest stored logit whose score reaches the bound
  uint32_t* hmax;   // [R] the largest tile-maximum score key (the request's best score)
  int cap;
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
  s.count = (int*)take((size_t)R * 4);
  s.thr = (uint32_t*)take((size_t)R * 4);
  s.fb_flag = (int*)take((size_t)R * 4);
  s.fb_any = (int*)take(16);
  s.cand = (uint64_t*)take((size_t)R * s.cap * 8);
  s.pre = (uint64_t*)take((size_t)R * W_t * K * 8);
  s.hint = (float2*)take((size_t)R * W_t * n_tiles * sizeof(float2));
  s.tcount = (int*)take((size_t)R * 4);
  s.tlist = (uint32_t*)take((size_t)R * s.cap_tiles * 4);
  s.cut = (float*)take((size_t)R * W_t * 4);
  s.hmax = (uint32_t*)take((size_t)R * 4);
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

// ---- bound: the W_next-th largest hint score of each request, and the tiles
// that can hold a candidate. A code scores at most its tile's maximum (the
// score is monotone in the stored logit within a row), so only tiles whose
// maximum reaches the bound are listed for the filter.
template <typename T>
__global__ void __launch_bounds__(kBoundThreads) select_bound_kernel(
    int W_t, int V, int n_tiles, int W_next, const float2* __restrict__ hint,
    const float* __restrict__ lse, const float* __restrict__ cum, const float* __restrict__ bias,
    SelScratch ss, int smem_keys, unsigned* err) {
  extern __shared__ uint32_t hkeys[];
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[3];
  __shared__ int s_cnt;
  __shared__ unsigned s_max;
  const int r = blockIdx.x;
  const int n_h = W_t * n_tiles;
  if (threadIdx.x == 0) {
    ss.count[r] = 0;
    s_cnt = 0;
    s_max = 0u;
    if (r == 0) *ss.fb_any = 0;
  }
  // a row whose lse or cumulative score is not finite is flagged
  for (int b = threadIdx.x; b < W_t; b += blockDim.x) {
    const size_t row = (size_t)r * W_t + b;
    if (!isfinite(lse[row]) || !isfinite(cum_prime(cum, bias, row)))
      raise_error(err, GDNBEAM_DERR_NONFINITE);
  }
  auto key_of = [&](int i) -> uint32_t {
    const int b = i / n_tiles;
    const size_t row = (size_t)r * W_t + b;
    const float zm = hint[row * n_tiles + (i % n_tiles)].x;
    const float zs = St<T>::to_f(St<T>::from_f(zm));  // stored value of the tile's top element
    return orderable(score(cum_prime(cum, bias, row), zs, lse[row]));
  };
  const bool on_chip = n_h <= smem_keys;
  uint32_t t = 0u;  // too few hints for a bound: keep every tile
  if (W_next <= n_h) {
    if (on_chip) {
      for (int i = threadIdx.x; i < n_h; i += blockDim.x) hkeys[i] = key_of(i);
      __syncthreads();
      t = radix_kth<uint32_t>(n_h, (unsigned)W_next, [&](int i) { return hkeys[i]; }, hist, sh);
    } else {
      t = radix_kth<uint32_t>(n_h, (unsigned)W_next, key_of, hist, sh);
    }
  }
  if (threadIdx.x == 0) ss.thr[r] = t;
  // each row's cutoff: the smallest stored value whose score reaches t, by
  // bisection over the storage keys (scores are monotone in the stored
  // value within a row); NaN when no code of the row can qualify
  for (int b = threadIdx.x; b < W_t; b += blockDim.x) {
    const size_t row = (size_t)r * W_t + b;
    const float cp = cum_prime(cum, bias, row), l = lse[row];
    uint32_t lo = SKey<T>::kNegInf, hi = SKey<T>::kPosInf + 1u;  // hi: none reaches t
    while (lo < hi) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      if (orderable(score(cp, SKey<T>::value(mid), l)) >= t) hi = mid; else lo = mid + 1u;
    }
    ss.cut[row] = SKey<T>::value(lo);
  }
  __syncthreads();
  uint32_t* list = ss.tlist + (size_t)r * ss.cap_tiles;
  unsigned my_max = 0u;
  for (int i = threadIdx.x; i < n_h; i += blockDim.x) {
    const uint32_t key = on_chip ? hkeys[i] : key_of(i);
    my_max = max(my_max, key);
    if (key >= t) {
      const int pos = atomicAdd(&s_cnt, 1);
      if (pos < ss.cap_tiles) list[pos] = (uint32_t)i;
    }
  }
  for (int o = 16; o > 0; o >>= 1) my_max = max(my_max, __shfl_xor_sync(0xffffffffu, my_max, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&s_max, my_max);
  __syncthreads();
  if (threadIdx.x == 0) {
    ss.tcount[r] = s_cnt;
    ss.hmax[r] = s_max;
  }
}

// Loads the eight codes v0 .. v0+7 of row zr into zv (NaN past V).
template <typename T>
__device__ __forceinline__ void load_codes(const T* __restrict__ zr, int v0, int V, bool vec,
                                           float (&zv)[kTile / 32]) {
  constexpr int EPL = kTile / 32;
  if (vec && v0 + EPL <= V) {
    if constexpr (sizeof(T) == 2) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(zr + v0));
      const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < EPL; ++e) zv[e] = __uint_as_float(((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
    } else {
      const float4 a = __ldg(reinterpret_cast<const float4*>(zr + v0));
      const float4 c = __ldg(reinterpret_cast<const float4*>(zr + v0 + 4));
      zv[0] = a.x; zv[1] = a.y; zv[2] = a.z; zv[3] = a.w;
      zv[4] = c.x; zv[5] = c.y; zv[6] = c.z; zv[7] = c.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) zv[e] = v0 + e < V ? ldf(zr + v0 + e) : __int_as_float(0x7FC00000);
  }
}

// ---- filter: append every code of the listed tiles whose score reaches the
// bound. One warp per listed tile (256 codes, eight per lane). Codes are
// compared as stored values with the row's cutoff logit from the bound
// kernel; scores are computed only for hits.
template <typename T>
__global__ void __launch_bounds__(kFilterThreads) select_filter_kernel(
    int W_t, int V, int n_tiles, int blocks_per_req, const T* __restrict__ z,
    const float* __restrict__ lse, const float* __restrict__ cum, const float* __restrict__ bias,
    SelScratch ss) {
  constexpr int EPL = kTile / 32;          // codes per lane
  const int r = blockIdx.x / blocks_per_req;
  const int lane = threadIdx.x & 31;
  const int warps = blocks_per_req * (kFilterThreads / 32);
  const int n_list = min(ss.tcount[r], ss.cap_tiles);
  const uint32_t* list = ss.tlist + (size_t)r * ss.cap_tiles;
  uint64_t* out = ss.cand + (size_t)r * ss.cap;
  const bool vec = (V % 8) == 0 && ((uintptr_t)z & 15) == 0;
  for (int j = (blockIdx.x % blocks_per_req) * (kFilterThreads / 32) + (threadIdx.x >> 5); j < n_list;
       j += warps) {
    const uint32_t i = list[j];
    const int b = (int)(i / (uint32_t)n_tiles), tile = (int)(i % (uint32_t)n_tiles);
    const size_t row = (size_t)r * W_t + b;
    const float cp = cum_prime(cum, bias, row), l = lse[row];
    const float thr = ss.cut[row];  // NaN when no code can qualify
    const int v0 = tile * kTile + lane * EPL;
    float zv[EPL];
    load_codes<T>(z + row * (size_t)V, v0, V, vec, zv);
    unsigned hits = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if (zv[e] >= thr) hits |= 1u << e;  // NaN never compares true
    if (!__any_sync(0xffffffffu, hits != 0)) continue;
    const int mine = __popc(hits);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int base = 0;
    if (lane == 31) base = atomicAdd(ss.count + r, total);
    base = __shfl_sync(0xffffffffu, base, 31);
    int idx = base + incl - mine;
    const uint32_t flat0 = (uint32_t)b * (uint32_t)V;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (hits & (1u << e)) {
        const uint32_t o = orderable(score(cp, zv[e], l));
        if (idx < ss.cap) out[idx] = make_key(o, flat0 + (uint32_t)(v0 + e));
        ++idx;
      }
    }
  }
}

// Visits the listed tiles of request r with the whole block, one warp per
// tile. Every lane of the warp calls f(hits, o, flat0): hits masks the lane's
// eight codes whose stored value reaches the row's cutoff, o holds their
// score keys (other entries are 0) and flat0 is the flat index of code 0.
template <typename T, typename F>
__device__ __forceinline__ void for_listed_codes(int r, int W_t, int V, int n_tiles, int n_list,
                                                 const T* __restrict__ z, const float* __restrict__ lse,
                                                 const float* __restrict__ cum,
                                                 const float* __restrict__ bias, const SelScratch& ss,
                                                 F&& f) {
  constexpr int EPL = kTile / 32;
  const int lane = threadIdx.x & 31;
  const uint32_t* list = ss.tlist + (size_t)r * ss.cap_tiles;
  const bool vec = (V % 8) == 0 && ((uintptr_t)z & 15) == 0;
  for (int j = threadIdx.x >> 5; j < n_list; j += blockDim.x >> 5) {
    const uint32_t i = list[j];
    const int b = (int)(i / (uint32_t)n_tiles), tile = (int)(i % (uint32_t)n_tiles);
    const size_t row = (size_t)r * W_t + b;
    const int v0 = tile * kTile + lane * EPL;
    float zv[EPL];
    load_codes<T>(z + row * (size_t)V, v0, V, vec, zv);
    const float thr = ss.cut[row];
    unsigned hits = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if (zv[e] >= thr) hits |= 1u << e;
    uint32_t o[EPL];
    const float cp = cum_prime(cum, bias, row), l = lse[row];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = (hits >> e) & 1u ? orderable(score(cp, zv[e], l)) : 0u;
    f(hits, o, (uint32_t)b * (uint32_t)V + (uint32_t)v0);
  }
}

// ---- refine: more codes reach the bound than the buffer holds. Narrows the
// bound t over the listed codes until at most `target` codes reach it (and
// still at least W_next), then writes those codes' keys to keys[]. Each
// round histograms the score keys inside the window [lo, hi] on the 11 bits
// below the highest bit where lo and hi differ, counts the codes above hi,
// and keeps the bin holding the W_next-th largest. Returns the number of
// keys written, or -1 when the codes tying at one score are too many.
constexpr int kRefineBins = 2048;
static_assert(kRefineBins * 4 <= kFinalSmemKeys * 8, "the bins live in the final block's key area");

template <typename T>
__device__ int refine_bound(int r, int W_t, int V, int n_tiles, int W_next, int target,
                            const T* __restrict__ z, const float* __restrict__ lse,
                            const float* __restrict__ cum, const float* __restrict__ bias,
                            const SelScratch& ss, uint64_t* keys) {
  __shared__ unsigned s_above, s_cnt, s_res[4];
  uint32_t* bins = reinterpret_cast<uint32_t*>(keys);
  const int n_list = min(ss.tcount[r], ss.cap_tiles);
  const int lane = threadIdx.x & 31;
  uint32_t lo = ss.thr[r], hi = ss.hmax[r];
  bool fit = false;
  for (int round = 0; round < 8 && lo <= hi; ++round) {
    const int p = lo == hi ? 0 : 31 - __clz(lo ^ hi);
    const int shift = p >= 10 ? p - 10 : 0;
    const uint32_t base = lo >> shift;  // (hi >> shift) - base < kRefineBins
    for (int i = threadIdx.x; i < kRefineBins; i += blockDim.x) bins[i] = 0u;
    if (threadIdx.x == 0) s_above = 0u;
    __syncthreads();
    for_listed_codes<T>(r, W_t, V, n_tiles, n_list, z, lse, cum, bias, ss,
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
    if (!s_res[3]) return -1;  // fewer than W_next codes reach lo: bound inconsistent
    const uint32_t d = s_res[0];
    const unsigned total = s_above + s_res[1] + s_res[2];
    const uint32_t blo = max(lo, (uint32_t)((uint64_t)(base + d) << shift));
    const uint32_t bhi = min(hi, (uint32_t)(((uint64_t)(base + d + 1) << shift) - 1));
    __syncthreads();  // everyone has read s_res and the bins
    lo = blo;
    if (total <= (unsigned)target) {
      fit = true;
      break;
    }
    if (blo == bhi) return -1;  // more codes tie at one score than fit
    hi = bhi;
  }
  if (!fit) return -1;
  // every listed code with key >= lo, as a 64-bit selection key
  if (threadIdx.x == 0) s_cnt = 0u;
  __syncthreads();
  for_listed_codes<T>(r, W_t, V, n_tiles, n_list, z, lse, cum, bias, ss,
                      [&](unsigned hits, const uint32_t (&o)[kTile / 32], uint32_t flat0) {
    unsigned keep = 0;
#pragma unroll
    for (int e = 0; e < kTile / 32; ++e)
      if (((hits >> e) & 1u) && o[e] >= lo) keep |= 1u << e;
    const int mine = __popc(keep);
    int incl = mine;
#pragma unroll
    for (int q = 1; q < 32; q <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, q);
      if (lane >= q) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    unsigned pos = 0;
    if (lane == 31 && total) pos = atomicAdd(&s_cnt, (unsigned)total);
    pos = __shfl_sync(0xffffffffu, pos, 31) + (unsigned)(incl - mine);
#pragma unroll
    for (int e = 0; e < kTile / 32; ++e) {
      if ((keep >> e) & 1u) {
        if (pos < (unsigned)target) keys[pos] = make_key(o[e], flat0 + (uint32_t)e);
        ++pos;
      }
    }
  });
  __syncthreads();
  const unsigned n = s_cnt;
  return n >= (unsigned)W_next && n <= (unsigned)target ? (int)n : -1;
}

// ---- final: exact top-W_next of the filtered candidates, sorted
template <typename T>
__global__ void __launch_bounds__(kFinalThreads) select_final_kernel(
    int W_t, int V, int n_tiles, int W_next, const T* __restrict__ z, const float* __restrict__ lse,
    const float* __restrict__ cum, const float* __restrict__ bias, SelScratch ss,
    int32_t* __restrict__ parents, int32_t* __restrict__ tokens, float* __restrict__ cum_next) {
  extern __shared__ uint64_t keys[];  // [kFinalSmemKeys]
  __shared__ unsigned hist[256];
  __shared__ unsigned sh[4];
  __shared__ uint64_t win[kMaxSort];
  const int r = blockIdx.x;
  int n_c = ss.count[r];
  bool on_chip = false;
  if (n_c >= W_next && ss.tcount[r] <= ss.cap_tiles && n_c > ss.cap) {
    n_c = refine_bound<T>(r, W_t, V, n_tiles, W_next, min(ss.cap, kFinalSmemKeys), z, lse, cum,
                          bias, ss, keys);
    on_chip = true;
  }
  if (n_c < W_next || n_c > ss.cap || ss.tcount[r] > ss.cap_tiles) {
    if (threadIdx.x == 0) {
      ss.fb_flag[r] = 1;
      atomicOr(ss.fb_any, 1);
    }
    return;
  }
  if (threadIdx.x == 0) ss.fb_flag[r] = 0;
  const uint64_t* c = ss.cand + (size_t)r * ss.cap;
  if (!on_chip && n_c <= kFinalSmemKeys) {
    on_chip = true;
    for (int i = threadIdx.x; i < n_c; i += blockDim.x) keys[i] = c[i];
    __syncthreads();
  }
  auto get = [&](int i) { return on_chip ? keys[i] : c[i]; };
  uint64_t prefix = 0;
  if (W_next < n_c) prefix = radix_kth<uint64_t>(n_c, (unsigned)W_next, get, hist, sh);
  int P = 1;
  while (P < W_next) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) win[i] = 0;
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_c; i += blockDim.x) {
    uint64_t key = get(i);
    if (key >= prefix) {
      unsigned idx = atomicAdd(&sh[3], 1u);
      if (idx < (unsigned)W_next) win[idx] = key;
    }
  }
  __syncthreads();
  const size_t o = (size_t)r * W_next;
  sort_and_emit(win, P, W_next, V, parents + o, tokens + o, cum_next + o);
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
  // bound
  const int n_h = W_t * n_tiles;
  const int bound_keys = n_h <= 49152 ? n_h : 0;
  const size_t bound_smem = (size_t)bound_keys * 4;
  GDN_CUDA(cudaFuncSetAttribute(select_bound_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(bound_smem > 0 ? bound_smem : 4)));
  select_bound_kernel<T><<<R, kBoundThreads, bound_smem, s>>>(W_t, V, n_tiles, W_next, hint, lse,
                                                              cum, bias, ss, bound_keys, err);
  GDN_LAUNCH_CHECK();
  // filter over the listed tiles
  const int per_req = (ss.cap_tiles + kFilterThreads / 32 - 1) / (kFilterThreads / 32);
  const int bpr = per_req < kFilterBlocksPerReq ? per_req : kFilterBlocksPerReq;
  select_filter_kernel<T><<<R * bpr, kFilterThreads, 0, s>>>(W_t, V, n_tiles, bpr, z, lse, cum,
                                                              bias, ss);
  GDN_LAUNCH_CHECK();
  // final
  const size_t fin_smem = (size_t)kFinalSmemKeys * 8;
  GDN_CUDA(cudaFuncSetAttribute(select_final_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)fin_smem));
  select_final_kernel<T><<<R, kFinalThreads, fin_smem, s>>>(W_t, V, n_tiles, W_next, z, lse, cum,
                                                            bias, ss, parents, tokens, cum_next);
  GDN_LAUNCH_CHECK();
  // exact fallback for requests whose buffer was short or overflowed
  const size_t row_smem = (size_t)V * 8;
  GDN_CUDA(cudaFuncSetAttribute(select_rowcut_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)row_smem));
  const int rc_grid = n < 4 * sm_count() ? n : 4 * sm_count();
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
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev] > 0 ? sms[dev] : 132;
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
