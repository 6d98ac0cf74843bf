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
//    then smaller id".  Keys are unique within a row, which makes every merge exact and
//    independent of scheduling.
//  * A row is split over a cluster of `S` thread blocks (grid.x = S).  Each warp streams
//    its share with 128-bit loads (8 bf16 per lane) and keeps a sorted top-K list in
//    registers (one or two entries per lane).  A vector is rejected with three packed
//    bf16 max instructions when all 8 values fall below the current threshold; only
//    survivors are keyed and inserted.
//  * The threshold is the largest K-th entry any warp of the block has seen (shared
//    memory atomicMax), seeded per warp from the K-th largest of its first 32 lane maxima.
//  * Warp lists are merged in shared memory by rank counting, then the S block results are
//    pushed into block 0's shared memory over the cluster (DSMEM) and merged the same way.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr int kMaxSplit = 8;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

// Element-wise max of two 16-byte vectors (packed bf16 pairs or f32).
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

// True when every element of the vector is strictly below `tval` (NaN never rejects).
template <bool kBf16>
__device__ __forceinline__ bool all_below(const uint4& v, float tval) {
  if constexpr (kBf16) {
    const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
    return (__uint_as_float(m & 0xFFFF0000u) < tval) && (__uint_as_float(m << 16) < tval);
  } else {
    const float m = fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                          fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    return m < tval;  // fmaxf drops a NaN operand; a vector of all NaN fails the test
  }
}

// A descending top-K list spread over a warp: entry j*32 + lane lives in e[j] of `lane`.
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
  // Insert key x (warp-uniform call).
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
};

// Offer this lane's candidate keys (bit e of `pend` marks keys[e]) to the warp list.
template <int KW, int EPV>
__device__ __forceinline__ void offer(WarpTopK<KW>& L, const uint64_t (&keys)[EPV], uint32_t pend, uint64_t& filt,
                                      int lane, unsigned long long* s_thresh) {
  for (;;) {
    const uint32_t any = __ballot_sync(kFull, pend != 0);
    if (!any) break;
    const int src = __ffs(any) - 1;
    uint64_t mine = 0;
    if (pend) {
      const int e = __ffs(pend) - 1;
#pragma unroll
      for (int t = 0; t < EPV; ++t)
        if (t == e) mine = keys[t];
    }
    const uint64_t x = __shfl_sync(kFull, mine, src);
    if (lane == src) pend &= pend - 1;
    if (x > filt) {
      L.insert(x, lane);
      if (L.kth > filt) {
        filt = L.kth;
        if (lane == 0) atomicMax(s_thresh, static_cast<unsigned long long>(filt));
      }
    }
  }
}

template <bool kBf16, int KW>
__global__ void __launch_bounds__(kThreads) topk_kernel(const void* __restrict__ logits, int V, int K, int S,
                                                        float* __restrict__ vals, int32_t* __restrict__ ids) {
  constexpr int EPV = kBf16 ? 8 : 4;  // elements per 16-byte vector
  __shared__ uint64_t s_warp[kWarps * 32 * KW];
  __shared__ uint64_t s_block[32 * KW];
  __shared__ uint64_t s_cluster[kMaxSplit * 32 * KW];
  __shared__ unsigned long long s_thresh;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int rank = blockIdx.x;  // == rank in the cluster (the cluster spans grid.x)
  const int64_t row = blockIdx.y;

  if (threadIdx.x == 0) s_thresh = 0;
  __syncthreads();

  const int64_t e0 = row * static_cast<int64_t>(V);
  int head = static_cast<int>((EPV - (e0 % EPV)) % EPV);
  if (head > V) head = V;
  const int nvec = (V - head) / EPV;
  const int tail = V - head - nvec * EPV;
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(logits) + (e0 + head) * (kBf16 ? 2 : 4));
  const int vbeg = static_cast<int>(static_cast<int64_t>(rank) * nvec / S);
  const int vend = static_cast<int>(static_cast<int64_t>(rank + 1) * nvec / S);

  WarpTopK<KW> L;
  L.init(K);
  uint64_t filt = 0;  // keys <= filt cannot be in the row's top K

  auto key_of = [&](const uint4& v, int e, int elem0) { return make_key(elem_bits<kBf16>(v, e), elem0 + e); };

  // Lanes past the end of the segment see a vector of -inf (bf16 and f32 bit patterns).
  const uint4 neg_inf = kBf16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                              : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
  bool first = true;
  for (int base = vbeg + warp * (kUnroll * 32); base < vend; base += kWarps * kUnroll * 32) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = base + u * 32 + lane;
      v[u] = (vi < vend) ? ld_stream(vp + vi) : neg_inf;
    }
    const uint64_t shared_t = *reinterpret_cast<volatile unsigned long long*>(&s_thresh);
    if (shared_t > filt) filt = shared_t;
    if (first && KW == 1) {
      // Seed the threshold: the K-th largest of the 32 lane maxima of the first vector is a
      // lower bound for the K-th largest key of the warp's data, so anything below it can go.
      const int vi = base + lane;
      uint64_t m = 0;
      if (vi < vend) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const uint64_t k = key_of(v[0], e, head + vi * EPV);
          m = k > m ? k : m;
        }
      }
      int above = 0;  // keys are unique, so exactly one lane has K-1 larger maxima
      for (int o = 0; o < 32; ++o) above += (__shfl_sync(kFull, m, o) > m);
      const uint32_t is_kth = __ballot_sync(kFull, m != 0 && above == K - 1);
      if (is_kth) {
        const uint64_t t0 = __shfl_sync(kFull, m, __ffs(is_kth) - 1);
        if (t0 - 1 > filt) filt = t0 - 1;
      }
      first = false;
    }
    // Common case: one packed max over all kUnroll vectors of the lane, one compare, one vote.
    const float tval = key_value(filt);
    const bool fast = filt != 0 && tval > -INFINITY;
    bool maybe = true;
    if (fast) {
      uint4 mx = v[0];
#pragma unroll
      for (int u = 1; u < kUnroll; ++u) mx = vmax<kBf16>(mx, v[u]);
      maybe = !all_below<kBf16>(mx, tval);
    }
    if (!__any_sync(kFull, maybe)) continue;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = base + u * 32 + lane;
      const float tv = key_value(filt);
      const bool fst = filt != 0 && tv > -INFINITY;
      const bool slow = vi < vend && !(fst && all_below<kBf16>(v[u], tv));
      if (!__any_sync(kFull, slow)) continue;
      uint32_t pend = 0;
      uint64_t keys[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        keys[e] = slow ? key_of(v[u], e, head + vi * EPV) : 0ull;
        if (keys[e] > filt) pend |= 1u << e;
      }
      offer<KW, EPV>(L, keys, pend, filt, lane, &s_thresh);
    }
  }

  // Unaligned head (rank 0) and tail (last rank) elements, one per lane.
  if (warp == 0) {
    uint64_t keys[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) keys[e] = 0;
    uint32_t pend = 0;
    const char* rowp = static_cast<const char*>(logits) + e0 * (kBf16 ? 2 : 4);
    auto scalar_key = [&](int idx) {
      uint32_t bits;
      if constexpr (kBf16) {
        bits = static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rowp)[idx]) << 16;
      } else {
        bits = reinterpret_cast<const uint32_t*>(rowp)[idx];
      }
      return make_key(bits, idx);
    };
    if (rank == 0 && lane < head) {
      keys[0] = scalar_key(lane);
      pend = keys[0] > filt ? 1u : 0u;
    }
    offer<KW, EPV>(L, keys, pend, filt, lane, &s_thresh);
    pend = 0;
    keys[0] = 0;
    if (rank == S - 1 && lane < tail) {
      keys[0] = scalar_key(head + nvec * EPV + lane);
      pend = keys[0] > filt ? 1u : 0u;
    }
    offer<KW, EPV>(L, keys, pend, filt, lane, &s_thresh);
  }

  // Block merge: rank every warp entry among all of them.
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    const int idx = j * 32 + lane;
    if (idx < K) s_warp[warp * K + idx] = L.e[j];
  }
  if (threadIdx.x < K) s_block[threadIdx.x] = 0;
  __syncthreads();
  const int total = kWarps * K;
  for (int c = threadIdx.x; c < total; c += kThreads) {
    const uint64_t x = s_warp[c];
    if (x == 0) continue;
    int above = 0;
    for (int o = 0; o < total; ++o) above += (s_warp[o] > x);
    if (above < K) s_block[above] = x;
  }
  __syncthreads();

  const uint64_t* final_keys = s_block;
  if (S > 1) {
    // Push this block's K keys into block 0 of the cluster, then block 0 merges S*K keys.
    if (threadIdx.x < K) {
      const uint32_t dst = map_to_rank(smem_u32(&s_cluster[rank * K + threadIdx.x]), 0);
      st_cluster_u64(dst, s_block[threadIdx.x]);
    }
    cluster_sync();
    if (rank != 0) return;
    if (threadIdx.x < K) s_block[threadIdx.x] = 0;
    __syncthreads();
    const int tot = S * K;
    for (int c = threadIdx.x; c < tot; c += kThreads) {
      const uint64_t x = s_cluster[c];
      if (x == 0) continue;
      int above = 0;
      for (int o = 0; o < tot; ++o) above += (s_cluster[o] > x);
      if (above < K) s_block[above] = x;
    }
    __syncthreads();
    final_keys = s_block;
  }
  if (threadIdx.x < K) {
    const uint64_t x = final_keys[threadIdx.x];
    vals[row * K + threadIdx.x] = key_value(x);
    ids[row * K + threadIdx.x] = static_cast<int32_t>(key_index(x));
  }
}

template <bool kBf16, int KW>
cudaError_t launch_topk_t(const void* logits, int rows, int V, int K, int S, float* vals, int32_t* ids,
                          cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_kernel<kBf16, KW>, logits, V, K, S, vals, ids);
}

}  // namespace

cudaError_t launch_topk(const void* logits, bool is_bf16, int rows, int V, int K, int ctas_per_row, float* vals,
                        int32_t* ids, cudaStream_t stream) {
  const int S = ctas_per_row < 1 ? 1 : (ctas_per_row > kMaxSplit ? kMaxSplit : ctas_per_row);
  if (rows > 65535) return cudaErrorInvalidConfiguration;
  if (is_bf16) {
    return K <= 32 ? launch_topk_t<true, 1>(logits, rows, V, K, S, vals, ids, stream)
                   : launch_topk_t<true, 2>(logits, rows, V, K, S, vals, ids, stream);
  }
  return K <= 32 ? launch_topk_t<false, 1>(logits, rows, V, K, S, vals, ids, stream)
                 : launch_topk_t<false, 2>(logits, rows, V, K, S, vals, ids, stream);
}

}  // namespace dcoco
