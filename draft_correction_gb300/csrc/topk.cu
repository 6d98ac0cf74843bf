// a1. Vocabulary-wide top-K of the drafter's logits.
//
// Two Delta blog, "Keep the leading candidates": DCOCO keeps the K highest-logit
// candidates of each of the B draft positions.  Here every row (stream n, slot i) of
// [N*B, V] logits is reduced to its K largest values, sorted by value descending with
// equal values ordered by ascending token id.
//
// Design (HBM-bound; one pass over the logits):
//  * Every candidate is a 64-bit key: the order-preserving code of its float value in the
//    high word and (0xFFFFFFFF - id) in the low word, so "larger key" means "larger value,
//    then smaller id".  Keys are unique within a row, which makes every selection exact and
//    independent of scheduling.
//  * A row is split over a cluster of S thread blocks (grid.x = S, S <= 8, chosen so the
//    grid fills whole waves of the GPU).  A block streams its segment with 128-bit loads
//    (8 bf16 per lane), the next iteration's loads in flight while the current one is
//    filtered.  The streaming loop has no barrier.
//  * Threshold: the K-th largest of the block's 256 lane maxima over its first 2 iterations
//    (each warp sorts its 32 maxima with shuffles; ranks come from binary searches in the 8
//    sorted lists).  K values reach it, so anything smaller is not in the top K.
//  * Streaming loop, no barrier: a lane tests the packed max of its vectors against the
//    threshold and, if it may hold a candidate, records the vectors' position (a "suspect").
//    After the loop the block keys the suspect vectors element by element, keeps the keys above
//    the threshold, selects its K largest by rank counting, pushes them into block 0 of the
//    cluster (distributed shared memory), and block 0 ranks the S sorted lists by binary search.
//  * Rows that defeat the threshold (all values equal, sorted rows, NaN rows) overflow the
//    buffer; the block then recomputes its segment exactly with per-warp register lists.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;          // 16-byte vectors per lane per iteration
constexpr int kMaxSplit = 8;
constexpr int kMaxK = 64;
constexpr int kCap = 1024;     // candidate buffer (keys), kCap / kWarps per warp
constexpr int kSusCap = 2048;  // lanes that may hold a candidate (per block), kSusCap / kWarps per warp
constexpr int kCapW = kCap / kWarps;
constexpr int kSusW = kSusCap / kWarps;
constexpr unsigned kFull = 0xFFFFFFFFu;

template <bool kBf16>
constexpr int kEpv = kBf16 ? 8 : 4;  // elements per 16-byte vector

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 32 bytes at a 32-byte aligned address, streamed (not kept in L1).
__device__ __forceinline__ void ld_stream32(const uint4* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}

// 32 bytes of a suspect, read again after the stream: the access hands the line back to L2's
// normal eviction order as one to evict first (the stream marked it to keep).
__device__ __forceinline__ void ld_release32(const uint4* p, uint4& a, uint4& b) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], pol;\n\t}"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p));
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Element e of a 16-byte vector as float bits.
template <bool kBf16>
__device__ __forceinline__ uint32_t elem_bits(const uint4& v, int e) {
  if constexpr (kBf16) {
    const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
    return (e & 1) ? (w & 0xFFFF0000u) : (w << 16);
  } else {
    return (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
  }
}

// Element-wise max of two 16-byte vectors (packed bf16 pairs or f32); a NaN operand is dropped.
template <bool kBf16>
__device__ __forceinline__ uint4 vmax(const uint4& a, const uint4& b) {
  if constexpr (kBf16) {
    return make_uint4(bmax2(a.x, b.x), bmax2(a.y, b.y), bmax2(a.z, b.z), bmax2(a.w, b.w));
  } else {
    return make_uint4(__float_as_uint(fmaxf(__uint_as_float(a.x), __uint_as_float(b.x))),
                      __float_as_uint(fmaxf(__uint_as_float(a.y), __uint_as_float(b.y))),
                      __float_as_uint(fmaxf(__uint_as_float(a.z), __uint_as_float(b.z))),
                      __float_as_uint(fmaxf(__uint_as_float(a.w), __uint_as_float(b.w))));
  }
}

// Largest element of a vector as float bits (NaN only if every element is NaN).
template <bool kBf16>
__device__ __forceinline__ uint32_t vec_max_bits(const uint4& v) {
  if constexpr (kBf16) {
    const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
    return __float_as_uint(fmaxf(__uint_as_float(m & 0xFFFF0000u), __uint_as_float(m << 16)));
  } else {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
  }
}

// Descending bitonic sort of one key per lane across the warp.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t y = __shfl_xor_sync(kFull, x, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
    }
  }
  return x;
}

// Descending bitonic sort of 64 keys across a warp, two per lane: key i = lane + 32 h is x[h];
// afterwards x[0] of lane r is the r-th largest.
__device__ __forceinline__ void warp_sort64_desc(uint64_t (&x)[2], int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partners in the same lane (k == 64: the larger goes to the lower index)
        const uint64_t hi = x[0] > x[1] ? x[0] : x[1], lo = x[0] > x[1] ? x[1] : x[0];
        x[0] = hi;
        x[1] = lo;
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = lane + 32 * h;
          const uint64_t y = __shfl_xor_sync(kFull, x[h], j);
          const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
          x[h] = keep_max ? (x[h] > y ? x[h] : y) : (x[h] < y ? x[h] : y);
        }
      }
    }
  }
}

// Number of keys above x in nl (<= NL) descending lists of len keys each (list w at
// lists[w * len]).  The binary searches of all lists advance together, one probe of each per
// step, so their shared-memory loads overlap; in a descending list the keys above x form a
// prefix, and pos[w] grows to its length.
template <int NL>
__device__ __forceinline__ int rank_in_lists(const uint64_t* lists, int nl, int len, uint64_t x) {
  int top = 1;  // the largest power of two not above len
  while (top * 2 <= len) top *= 2;
  int pos[NL];
#pragma unroll
  for (int w = 0; w < NL; ++w) pos[w] = 0;
  for (int step = top; step > 0; step >>= 1) {
#pragma unroll
    for (int w = 0; w < NL; ++w) {
      const int i = pos[w] + step - 1;
      if (w < nl && i < len && lists[w * len + i] > x) pos[w] += step;
    }
  }
  int above = 0;
#pragma unroll
  for (int w = 0; w < NL; ++w) above += pos[w];
  return above;
}

// Merge the kWarps descending, 0-padded lists of K keys in s_wl[w * K ..] into the K largest,
// s_keep[0, K) (descending; 0 where fewer exist): every key's rank is the sum of binary-search
// counts over the lists.  Called by every thread of the block.
__device__ __forceinline__ void merge_lists(const uint64_t* s_wl, int K, uint64_t* s_keep) {
  for (int t = threadIdx.x; t < K; t += kThreads) s_keep[t] = 0;
  __syncthreads();
  for (int t = threadIdx.x; t < kWarps * K; t += kThreads) {
    const uint64_t x = s_wl[t];
    if (x == 0) continue;
    const int above = rank_in_lists<kWarps>(s_wl, kWarps, K, x);
    if (above < K) s_keep[above] = x;
  }
  __syncthreads();
}

// Keep the K largest keys of s_buf[0, cnt) (cnt <= kCap) in s_keep[0, K) (descending; 0 where
// cnt < K).  Called by every thread of the block; s_wl ([kWarps * K]) is scratch and may be
// s_buf itself.  Thread t holds candidates t, t + kThreads, ... in registers, so each warp owns
// an eighth of them; a warp extracts its K largest one per round with two warp max reductions
// (value word, then index word among equal values) and the lists are merged.
__device__ __forceinline__ void select_top(const uint64_t* s_buf, int cnt, int K, uint64_t* s_wl, uint64_t* s_keep) {
  constexpr int PER = kCap / kThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t e[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int c = static_cast<int>(threadIdx.x) + j * kThreads;
    e[j] = c < cnt ? s_buf[c] : 0ull;
  }
  __syncthreads();  // every candidate is in registers: s_wl (possibly s_buf) may be overwritten
  auto lane_best = [&]() {
    uint64_t b = e[0];
#pragma unroll
    for (int j = 1; j < PER; ++j) b = e[j] > b ? e[j] : b;
    return b;
  };
  uint64_t b = lane_best();
  for (int r = 0; r < K; ++r) {
    const uint32_t hi = static_cast<uint32_t>(b >> 32), lo = static_cast<uint32_t>(b);
    const uint32_t mhi = __reduce_max_sync(kFull, hi);
    const uint32_t tie = __ballot_sync(kFull, hi == mhi);
    uint32_t mlo = 0;
    if (hi == mhi) mlo = __reduce_max_sync(tie, lo);
    mlo = __shfl_sync(kFull, mlo, __ffs(tie) - 1);
    const uint64_t win = (static_cast<uint64_t>(mhi) << 32) | mlo;  // 0 once the warp runs out
    if (lane == 0) s_wl[warp * K + r] = win;
    if (win != 0 && b == win) {  // keys are unique: exactly one lane holds the winner
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (e[j] == win) e[j] = 0;
      b = lane_best();
    }
  }
  __syncthreads();
  merge_lists(s_wl, K, s_keep);
}

// The K largest of buf[0, cnt) (cnt <= kCapW) into out[0, K) (descending, 0-padded), by one warp:
// lane l holds buf[l], buf[l + 32], ... in registers and each round extracts the largest key
// with two warp max reductions (value word, then index word among equal values).
__device__ __forceinline__ void warp_top(const uint64_t* buf, int cnt, int K, uint64_t* out, int lane) {
  if (cnt <= 32) {  // the common case: one key per lane, one warp sort
    const uint64_t x = warp_sort_desc(lane < cnt ? buf[lane] : 0ull, lane);
    for (int r = lane; r < K; r += 32) out[r] = r < 32 ? (r == lane ? x : 0ull) : 0ull;
    return;
  }
  if (cnt <= 64) {  // two keys per lane, one 64-key warp sort
    uint64_t x[2] = {buf[lane], lane + 32 < cnt ? buf[lane + 32] : 0ull};
    warp_sort64_desc(x, lane);
    for (int r = lane; r < K; r += 32) out[r] = r < 32 ? x[0] : x[1];
    return;
  }
  constexpr int PER = kCapW / 32;
  uint64_t e[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) e[j] = lane + 32 * j < cnt ? buf[lane + 32 * j] : 0ull;
  auto lane_best = [&]() {
    uint64_t b = e[0];
#pragma unroll
    for (int j = 1; j < PER; ++j) b = e[j] > b ? e[j] : b;
    return b;
  };
  uint64_t b = lane_best();
  for (int r = 0; r < K; ++r) {
    const uint32_t hi = static_cast<uint32_t>(b >> 32), lo = static_cast<uint32_t>(b);
    const uint32_t mhi = __reduce_max_sync(kFull, hi);
    const uint32_t tie = __ballot_sync(kFull, hi == mhi);
    uint32_t mlo = 0;
    if (hi == mhi) mlo = __reduce_max_sync(tie, lo);
    mlo = __shfl_sync(kFull, mlo, __ffs(tie) - 1);
    const uint64_t win = (static_cast<uint64_t>(mhi) << 32) | mlo;  // 0 once the candidates run out
    if (lane == 0) out[r] = win;
    if (win != 0 && b == win) {  // keys are unique: exactly one lane holds the winner
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (e[j] == win) e[j] = 0;
      b = lane_best();
    }
  }
}

// Exact fallback for rows the threshold cannot thin out: a descending top-K list per warp in
// registers (entry j*32 + lane in e[j] of `lane`), one insertion per surviving key.
template <int KW>
struct WarpTopK {
  uint64_t e[KW];
  int K;
  uint64_t kth;  // entry K-1 (0 while the list is not full)

  __device__ __forceinline__ void init(int k) {
#pragma unroll
    for (int j = 0; j < KW; ++j) e[j] = 0;
    K = k;
    kth = 0;
  }
  __device__ __forceinline__ void insert(uint64_t x, int lane) {
    int pos = 0;
#pragma unroll
    for (int j = 0; j < KW; ++j) pos += __popc(__ballot_sync(kFull, e[j] > x));
    uint64_t prev[KW];
#pragma unroll
    for (int j = 0; j < KW; ++j) {
      const uint64_t up = __shfl_up_sync(kFull, e[j], 1);
      const uint64_t wrap = (j > 0) ? __shfl_sync(kFull, e[j > 0 ? j - 1 : 0], 31) : 0ull;
      prev[j] = (lane == 0) ? wrap : up;
    }
#pragma unroll
    for (int j = 0; j < KW; ++j) {
      const int idx = j * 32 + lane;
      e[j] = (idx < pos) ? e[j] : (idx == pos ? x : prev[j]);
    }
    const int last = K - 1;
    uint64_t t = 0;
#pragma unroll
    for (int j = 0; j < KW; ++j) {
      const uint64_t v = __shfl_sync(kFull, e[j], last & 31);
      if ((last >> 5) == j) t = v;
    }
    kth = t;
  }
  // Offer one key per lane (0 = none), lowest lane first.
  __device__ __forceinline__ void offer(uint64_t mine, int lane) {
    uint32_t pend = __ballot_sync(kFull, mine > kth);
    while (pend) {
      const int src = __ffs(pend) - 1;
      pend &= pend - 1;
      const uint64_t x = __shfl_sync(kFull, mine, src);
      if (x > kth) insert(x, lane);
    }
  }
};

struct Segment {
  const char* rowp;  // first element of the row
  const uint4* vp;   // first 32-byte aligned vector of the row
  int head, nvec, tail, vbeg, vend;  // nvec (the row's vectors) and every split point are even
};

template <bool kBf16, int KW>
__device__ __noinline__ void exact_segment_topk(const Segment& g, int K, int rank, int S, uint64_t* s_wl,
                                                uint64_t* s_keep) {
  constexpr int EPV = kEpv<kBf16>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpTopK<KW> L;
  L.init(K);
  for (int vi = g.vbeg + static_cast<int>(threadIdx.x); vi - lane < g.vend; vi += kThreads) {  // warp-uniform trip count
    const bool valid = vi < g.vend;
    const uint4 v = valid ? ld_stream(g.vp + vi) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int e = 0; e < EPV; ++e) L.offer(valid ? make_key(elem_bits<kBf16>(v, e), g.head + vi * EPV + e) : 0ull, lane);
  }
  if (warp == 0) {
    int idx = -1;
    if (rank == 0 && lane < g.head) idx = lane;
    if (rank == S - 1 && lane >= 16 && lane - 16 < g.tail) idx = g.head + g.nvec * EPV + (lane - 16);
    uint64_t k = 0;
    if (idx >= 0) {
      const uint32_t bits = kBf16 ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(g.rowp)[idx]) << 16
                                  : reinterpret_cast<const uint32_t*>(g.rowp)[idx];
      k = make_key(bits, idx);
    }
    L.offer(k, lane);
  }
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    const int idx = j * 32 + lane;
    if (idx < K) s_wl[warp * K + idx] = L.e[j];
  }
  __syncthreads();
  select_top(s_wl, kWarps * K, K, s_wl, s_keep);
}

template <bool kBf16, int KW>
__global__ void __launch_bounds__(kThreads, 4) topk_kernel(const void* __restrict__ logits, int V, int K, int S,
                                                        float* __restrict__ vals, int32_t* __restrict__ ids,
                                                        int wait_prior) {
  constexpr int EPV = kEpv<kBf16>;
  __shared__ uint64_t s_buf[kCap];
  __shared__ uint64_t s_sorted[kThreads];  // each warp's lane maxima, sorted
  __shared__ uint64_t s_wl[kWarps * kMaxK];
  __shared__ uint64_t s_keep[kMaxK];
  __shared__ uint64_t s_cluster[kMaxSplit * kMaxK];
  __shared__ int s_sus[kSusCap];  // first vector index of lanes that may hold a candidate
  __shared__ uint64_t s_thr;
  __shared__ int s_overflow;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int rank = blockIdx.x;  // == rank in the cluster (the cluster spans grid.x)
  const int64_t row = blockIdx.y;
  if (threadIdx.x == 0) {
    s_overflow = 0;
    s_thr = 0;
  }

  Segment g;
  const int64_t e0 = row * static_cast<int64_t>(V);
  g.rowp = static_cast<const char*>(logits) + e0 * (kBf16 ? 2 : 4);
  // Elements before the first 32-byte boundary form the head, and the last odd vector plus the
  // leftover elements the tail (each at most 15 elements), so that every lane can fetch its 64
  // contiguous bytes with two 32-byte loads.
  constexpr int ESZ = kBf16 ? 2 : 4;
  g.head = static_cast<int>(((32 - (reinterpret_cast<uintptr_t>(g.rowp) & 31)) & 31) / ESZ);
  if (g.head > V) g.head = V;
  g.nvec = ((V - g.head) / EPV) & ~1;
  g.tail = V - g.head - g.nvec * EPV;
  g.vp = reinterpret_cast<const uint4*>(g.rowp + static_cast<int64_t>(g.head) * ESZ);
  g.vbeg = 2 * static_cast<int>(static_cast<int64_t>(rank) * (g.nvec / 2) / S);
  g.vend = 2 * static_cast<int>(static_cast<int64_t>(rank + 1) * (g.nvec / 2) / S);
  constexpr int CH = kWarps * kU * 32;  // vectors per block iteration
  const int iters = (g.vend - g.vbeg + CH - 1) / CH;
  // lane t of the block owns kU consecutive vectors (64 bytes) of every iteration
  auto vidx = [&](int it, int u) { return g.vbeg + it * CH + static_cast<int>(threadIdx.x) * kU + u; };

  // Lanes past the end of the segment see -inf.
  const uint4 neg_inf = kBf16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                              : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
  // Three iterations of vectors in registers: the current one and two in flight.
  uint4 c0[kU], c1[kU], c2[kU];
  auto load = [&](int it, uint4(&v)[kU]) {
    const int vi0 = vidx(it, 0);
    if (it < iters && vi0 + kU <= g.vend) {
      ld_stream32(g.vp + vi0, v[0], v[1]);
      ld_stream32(g.vp + vi0 + 2, v[2], v[3]);
    } else {
#pragma unroll
      for (int u = 0; u < kU; ++u) v[u] = (it < iters && vi0 + u < g.vend) ? ld_stream(g.vp + vi0 + u) : neg_inf;
    }
  };

  if (wait_prior) grid_dep_wait();  // the logits may come from the preceding kernel
  grid_dep_launch();
  // Seed threshold: the K-th largest of the block's lane maxima over the first two iterations
  // (already in registers).  K elements reach that value, so nothing below it is in the top K.
  load(0, c0);
  load(1, c1);
  // While the block ranks its lane maxima (two barriers, no loads in flight), keep HBM busy:
  // ask L2 for the next two iterations, which the hot loop then reads from L2.
#pragma unroll
  for (int it = 2; it < 4; ++it) {
    const int vi0 = vidx(it, 0);
    if (it < iters && vi0 < g.vend) {
      prefetch_l2(g.vp + vi0);
      if (vi0 + kU - 1 < g.vend) prefetch_l2(g.vp + vi0 + kU - 1);
    }
  }
  {
    uint32_t mb = 0xFF800000u;  // -inf
    bool any = false;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (iters > 0 && vidx(0, u) < g.vend) {
        mb = __float_as_uint(fmaxf(__uint_as_float(mb), __uint_as_float(vec_max_bits<kBf16>(c0[u]))));
        any = true;
      }
      if (iters > 1 && vidx(1, u) < g.vend) {
        mb = __float_as_uint(fmaxf(__uint_as_float(mb), __uint_as_float(vec_max_bits<kBf16>(c1[u]))));
        any = true;
      }
    }
    const uint64_t mk = any ? (static_cast<uint64_t>(ord32(mb)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - threadIdx.x)
                            : 0ull;
    s_sorted[threadIdx.x] = warp_sort_desc(mk, lane);
    __syncthreads();
    const uint64_t x = s_sorted[threadIdx.x];
    if (x != 0 && K <= kThreads) {
      const int above = rank_in_lists<kWarps>(s_sorted, kWarps, 32, x);
      if (above == K - 1) s_thr = x & 0xFFFFFFFF00000000ull;  // value part only: keeps ties
    }
    __syncthreads();
  }
  const uint64_t thr = s_thr;
  const float tval = key_value(thr);
  const bool fast = thr != 0 && tval > -INFINITY;

  // Hot loop: one packed max over the lane's vectors and one compare per iteration.  A lane
  // that may hold a key above the threshold only records where its vectors are.
  int nsus = 0;  // this warp's suspect lanes so far (warp-uniform)
  for (int it = 0; it < iters; ++it) {
    load(it + 2, c2);
    bool maybe = vidx(it, 0) < g.vend;
    if (fast) {
      uint4 mx = c0[0];
#pragma unroll
      for (int u = 1; u < kU; ++u) mx = vmax<kBf16>(mx, c0[u]);
      maybe = !(__uint_as_float(vec_max_bits<kBf16>(mx)) < tval);
    }
    const uint32_t bal = __ballot_sync(kFull, maybe);
    if (maybe) {
      const int pos = nsus + __popc(bal & ((1u << lane) - 1));
      if (pos < kSusW) s_sus[warp * kSusW + pos] = vidx(it, 0);
      // the suspect's 64 bytes are read again after the loop: keep them in L2 past the stream
      // (whole 64-byte chunks only: those are the ones read back with the matching release)
      if (vidx(it, 0) + kU <= g.vend) prefetch_l2_keep(g.vp + vidx(it, 0));
    }
    nsus += __popc(bal);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      c0[u] = c1[u];
      c1[u] = c2[u];
    }
  }

  // Each warp, without waiting for the others: key every element of its suspect lanes'
  // vectors, keep the keys above the threshold, and extract its K largest.  Warps that finish
  // streaming early do this while the others still stream.
  {
    uint64_t* wbuf = s_buf + warp * kCapW;
    int ncand = 0;  // warp-uniform
    bool over = nsus > kSusW;
    auto append = [&](bool keep, uint64_t key) {
      const uint32_t b = __ballot_sync(kFull, keep);
      if (keep) {
        const int pos = ncand + __popc(b & ((1u << lane) - 1));
        if (pos < kCapW) wbuf[pos] = key;
      }
      ncand += __popc(b);
    };
    if (!over) {
      // one suspect per lane per round; the next round's 64 bytes are requested before this
      // round's are keyed, so the rounds' memory latencies overlap
      auto fetch = [&](int vi0, uint4(&v)[kU]) {
        if (vi0 + kU <= g.vend) {  // the lane's 64 contiguous bytes, one burst
          ld_release32(g.vp + vi0, v[0], v[1]);
          ld_release32(g.vp + vi0 + 2, v[2], v[3]);
        } else {
#pragma unroll
          for (int u = 0; u < kU; ++u) v[u] = vi0 + u < g.vend ? ld_stream(g.vp + vi0 + u) : neg_inf;
        }
      };
      int vi_next = lane < nsus ? s_sus[warp * kSusW + lane] : g.vend;
      uint4 v_next[kU];
      if (nsus > 0) fetch(vi_next, v_next);
      for (int j0 = 0; j0 < nsus; j0 += 32) {  // warp-uniform trip count
        const int vi0 = vi_next;
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = v_next[u];
        if (j0 + 32 < nsus) {
          const int jn = j0 + 32 + lane;
          vi_next = jn < nsus ? s_sus[warp * kSusW + jn] : g.vend;
          fetch(vi_next, v_next);
        }
        // Only values reaching the threshold value can have a key above it: mark them (a rolled
        // loop over the lane's 16 words, so that this code stays a few instruction-cache lines),
        // give every lane its output range with one warp scan, and key the marked values.  A value
        // at the threshold whose key is not above it stays a zero key, which every later step
        // ignores.
        auto word_at = [&](int w) -> uint32_t {
          const uint4 q = (w >> 2) == 0 ? v[0] : (w >> 2) == 1 ? v[1] : (w >> 2) == 2 ? v[2] : v[3];
          const int c = w & 3;
          return c == 0 ? q.x : c == 1 ? q.y : c == 2 ? q.z : q.w;
        };
        constexpr int EPW = kBf16 ? 2 : 1;  // elements per 32-bit word
        uint32_t mark = 0;
#pragma unroll 1
        for (int w = 0; w < 4 * kU; ++w) {
          const uint32_t x = word_at(w);
#pragma unroll
          for (int h = 0; h < EPW; ++h) {
            const int e = w * EPW + h;  // element of the lane's 64 bytes
            const uint32_t bits = kBf16 ? (h ? (x & 0xFFFF0000u) : (x << 16)) : x;
            if (vi0 + e / EPV < g.vend && !(__uint_as_float(bits) < tval)) mark |= 1u << e;
          }
        }
        const int cnt = __popc(mark);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        int pos = ncand + incl - cnt;
        while (mark != 0) {
          const int e = __ffs(mark) - 1;
          mark &= mark - 1;
          const uint32_t x = word_at(e / EPW);
          const uint32_t bits = kBf16 ? ((e & 1) ? (x & 0xFFFF0000u) : (x << 16)) : x;
          const uint64_t key = make_key(bits, g.head + vi0 * EPV + e);
          if (pos < kCapW) wbuf[pos] = key > thr ? key : 0ull;
          ++pos;
        }
        ncand += __shfl_sync(kFull, incl, 31);
      }
    }
    if (warp == 0) {
      // Unaligned head (rank 0) and tail (last rank) elements, one per lane.
      int idx = -1;
      if (rank == 0 && lane < g.head) idx = lane;
      if (rank == S - 1 && lane >= 16 && lane - 16 < g.tail) idx = g.head + g.nvec * EPV + (lane - 16);
      uint64_t key = 0;
      if (idx >= 0) {
        const uint32_t bits = kBf16 ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(g.rowp)[idx]) << 16
                                    : reinterpret_cast<const uint32_t*>(g.rowp)[idx];
        key = make_key(bits, idx);
      }
      append(idx >= 0, key);
    }
    over = over || ncand > kCapW;
    if (over) {
      if (lane == 0) s_overflow = 1;
    } else {
      __syncwarp();
      warp_top(wbuf, ncand, K, s_wl + warp * K, lane);
    }
  }
  __syncthreads();
  if (s_overflow)
    exact_segment_topk<kBf16, KW>(g, K, rank, S, s_wl, s_keep);
  else
    merge_lists(s_wl, K, s_keep);

  if (S > 1) {
    // Push this block's K keys into block 0 of the cluster; block 0 ranks every key among the
    // S sorted lists with binary searches.
    if (threadIdx.x < K) {
      const uint32_t dst = map_to_rank(smem_u32(&s_cluster[rank * K + threadIdx.x]), 0);
      st_cluster_u64(dst, s_keep[threadIdx.x]);
    }
    cluster_sync();
    if (rank != 0) return;
    for (int c = threadIdx.x; c < S * K; c += kThreads) {
      const uint64_t x = s_cluster[c];
      if (x == 0) continue;
      const int above = rank_in_lists<kMaxSplit>(s_cluster, S, K, x);
      if (above < K) {
        vals[row * K + above] = key_value(x);
        ids[row * K + above] = static_cast<int32_t>(key_index(x));
      }
    }
    return;
  }
  if (threadIdx.x < K) {
    const uint64_t x = s_keep[threadIdx.x];
    vals[row * K + threadIdx.x] = key_value(x);
    ids[row * K + threadIdx.x] = static_cast<int32_t>(key_index(x));
  }
}

template <bool kBf16, int KW>
cudaError_t launch_topk_t(const void* logits, int rows, int V, int K, int S, float* vals, int32_t* ids,
                          cudaStream_t stream, bool after_unrelated) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S > 1 ? 1 : 0;
  if (after_unrelated) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  } else {
    cfg.numAttrs += pdl_attr(&attr[cfg.numAttrs]);
  }
  return cudaLaunchKernelEx(&cfg, topk_kernel<kBf16, KW>, logits, V, K, S, vals, ids, after_unrelated ? 0 : 1);
}

// Blocks per row: one block per row once there are at least two rows per SM (more blocks per
// row only add per-block overhead); fewer rows are split until there are about four blocks per
// SM, at most 8 ways, keeping every segment at 16 KB or more.
int auto_split(int rows, int V, bool bf16) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
  }
  if (rows >= 2 * sms) return 1;
  const int64_t row_bytes = static_cast<int64_t>(V) * (bf16 ? 2 : 4);
  int s = (4 * sms + rows - 1) / rows;
  if (s > kMaxSplit) s = kMaxSplit;
  while (s > 1 && row_bytes / s < 16 * 1024) --s;
  return s;
}

}  // namespace

int topk_ctas_per_row(int rows, int V, bool is_bf16, int ctas_per_row) {
  const int S = ctas_per_row > 0 ? ctas_per_row : auto_split(rows, V, is_bf16);
  return S < 1 ? 1 : (S > kMaxSplit ? kMaxSplit : S);
}

cudaError_t launch_topk(const void* logits, bool is_bf16, int rows, int V, int K, int ctas_per_row, float* vals,
                        int32_t* ids, cudaStream_t stream, bool after_unrelated) {
  if (rows > 65535 || K > kMaxK) return cudaErrorInvalidConfiguration;
  const int S = topk_ctas_per_row(rows, V, is_bf16, ctas_per_row);
  if (is_bf16)
    return K <= 32 ? launch_topk_t<true, 1>(logits, rows, V, K, S, vals, ids, stream, after_unrelated)
                   : launch_topk_t<true, 2>(logits, rows, V, K, S, vals, ids, stream, after_unrelated);
  return K <= 32 ? launch_topk_t<false, 1>(logits, rows, V, K, S, vals, ids, stream, after_unrelated)
                 : launch_topk_t<false, 2>(logits, rows, V, K, S, vals, ids, stream, after_unrelated);
}

}  // namespace dcoco
