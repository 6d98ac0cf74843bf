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
//    filtered.
//  * Filtering is against one block-wide key threshold: a lane rejects its 16 values with
//    packed bf16 max instructions when all fall below it.  Survivors are appended to a
//    block-wide candidate buffer in shared memory.  At the end of an iteration, if the
//    buffer holds more than 128 keys, the block keeps its K largest (rank counting) and
//    the K-th becomes the new threshold.  The first iteration is seeded per warp with the
//    K-th largest of its 32 lane maxima, a valid lower bound on the K-th value.
//  * The buffer can take one full iteration of appends on top of 128 entries, so it never
//    overflows.  At the end each block selects its K largest keys, pushes them into block
//    0 of the cluster (distributed shared memory), and block 0 merges S*K keys.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 2;          // 16-byte vectors per lane per iteration
constexpr int kMaxSplit = 8;
constexpr int kMaxK = 64;
constexpr int kCapLow = 128;   // compaction trigger
constexpr unsigned kFull = 0xFFFFFFFFu;

template <bool kBf16>
constexpr int kEpv = kBf16 ? 8 : 4;  // elements per 16-byte vector
template <bool kBf16>
constexpr int kCap = kCapLow + kThreads * kU * kEpv<kBf16> + 32;  // + one warp of head/tail

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
    const float hi = __uint_as_float(m & 0xFFFF0000u), lo = __uint_as_float(m << 16);
    return __float_as_uint(fmaxf(hi, lo));
  } else {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
  }
}

// True when every element of the vector is strictly below `tval` (NaN never rejects).
template <bool kBf16>
__device__ __forceinline__ bool all_below(const uint4& v, float tval) {
  return __uint_as_float(vec_max_bits<kBf16>(v)) < tval;
}

// Keep the K largest keys of s_buf[0, cnt) in s_keep[0, K) (descending; 0 where cnt < K).
// Called by every thread of the block.
__device__ __forceinline__ void select_top(const uint64_t* s_buf, int cnt, int K, uint64_t* s_keep) {
  if (threadIdx.x < K) s_keep[threadIdx.x] = 0;
  __syncthreads();
  for (int c = threadIdx.x; c < cnt; c += kThreads) {
    const uint64_t x = s_buf[c];
    int above = 0;
    for (int o = 0; o < cnt; ++o) above += (s_buf[o] > x);
    if (above < K) s_keep[above] = x;
  }
  __syncthreads();
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) topk_kernel(const void* __restrict__ logits, int V, int K, int S,
                                                        float* __restrict__ vals, int32_t* __restrict__ ids) {
  constexpr int EPV = kEpv<kBf16>;
  constexpr int CAP = kCap<kBf16>;
  __shared__ uint64_t s_buf[CAP];
  __shared__ uint64_t s_keep[kMaxK];
  __shared__ uint64_t s_cluster[kMaxSplit * kMaxK];
  __shared__ uint64_t s_thr;
  __shared__ int s_cnt;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int rank = blockIdx.x;  // == rank in the cluster (the cluster spans grid.x)
  const int64_t row = blockIdx.y;
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_thr = 0;
  }

  const int64_t e0 = row * static_cast<int64_t>(V);
  int head = static_cast<int>((EPV - (e0 % EPV)) % EPV);
  if (head > V) head = V;
  const int nvec = (V - head) / EPV;
  const int tail = V - head - nvec * EPV;
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(logits) + (e0 + head) * (kBf16 ? 2 : 4));
  const int vbeg = static_cast<int>(static_cast<int64_t>(rank) * nvec / S);
  const int vend = static_cast<int>(static_cast<int64_t>(rank + 1) * nvec / S);
  constexpr int CH = kWarps * kU * 32;  // vectors per block iteration
  const int iters = (vend - vbeg + CH - 1) / CH;

  const uint4 neg_inf = kBf16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                              : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
  auto vidx = [&](int it, int u) { return vbeg + it * CH + (warp * kU + u) * 32 + lane; };
  uint4 cur[kU], nxt[kU];
  if (iters > 0) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int vi = vidx(0, u);
      cur[u] = vi < vend ? ld_stream(vp + vi) : neg_inf;
    }
  }
  __syncthreads();

  uint64_t warp_thr = 0;
  for (int it = 0; it < iters; ++it) {
    if (it + 1 < iters) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int vi = vidx(it + 1, u);
        nxt[u] = vi < vend ? ld_stream(vp + vi) : neg_inf;
      }
    }
    uint64_t thr = s_thr;
    if (it == 0 && K <= 32) {
      // Seed: the K-th largest of the warp's 32 lane maxima.  At least K elements reach that
      // value, so a key threshold with that value and index part 0 drops only elements that
      // cannot be in the top K.
      uint32_t mb = vec_max_bits<kBf16>(cur[0]);
#pragma unroll
      for (int u = 1; u < kU; ++u) mb = __float_as_uint(fmaxf(__uint_as_float(mb), __uint_as_float(vec_max_bits<kBf16>(cur[u]))));
      const uint64_t m = (static_cast<uint64_t>(ord32(mb)) << 32) | static_cast<uint64_t>(31 - lane);
      int above = 0;
      for (int o = 0; o < 32; ++o) above += (__shfl_sync(kFull, m, o) > m);
      const uint32_t is_kth = __ballot_sync(kFull, above == K - 1);
      const uint64_t kth = __shfl_sync(kFull, m, __ffs(is_kth) - 1);
      warp_thr = kth & 0xFFFFFFFF00000000ull;
    }
    if (it == 0 && warp_thr > thr) thr = warp_thr;
    const float tval = key_value(thr);
    const bool fast = thr != 0 && tval > -INFINITY;
    bool maybe = true;
    if (fast) {
      uint4 mx = cur[0];
#pragma unroll
      for (int u = 1; u < kU; ++u) mx = vmax<kBf16>(mx, cur[u]);
      maybe = !all_below<kBf16>(mx, tval);
    }
    if (__any_sync(kFull, maybe)) {
      uint32_t mask = 0;  // bit u*EPV + e: element e of vector u is a candidate
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int vi = vidx(it, u);
        if (maybe && vi < vend) {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            if (make_key(elem_bits<kBf16>(cur[u], e), head + vi * EPV + e) > thr) mask |= 1u << (u * EPV + e);
        }
      }
      const int n = __popc(mask);
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const int total = __shfl_sync(kFull, incl, 31);
      int start = 0;
      if (lane == 31 && total > 0) start = atomicAdd(&s_cnt, total);
      int pos = __shfl_sync(kFull, start, 31) + incl - n;
      while (mask) {
        const int b = __ffs(mask) - 1;
        mask &= mask - 1;
        const int u = b / EPV, e = b % EPV;
        uint4 vv = cur[0];
#pragma unroll
        for (int q = 1; q < kU; ++q)
          if (q == u) vv = cur[q];
        s_buf[pos++] = make_key(elem_bits<kBf16>(vv, e), head + vidx(it, u) * EPV + e);
      }
    }
    __syncthreads();
    const int cnt = s_cnt;
    __syncthreads();  // every thread has read the count before the next appends
    if (cnt > kCapLow) {
      select_top(s_buf, cnt, K, s_keep);
      if (threadIdx.x < K) s_buf[threadIdx.x] = s_keep[threadIdx.x];
      if (threadIdx.x == 0) {
        s_cnt = K;
        s_thr = s_keep[K - 1];
      }
      __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) cur[u] = nxt[u];
  }

  // Unaligned head (rank 0) and tail (last rank) elements, one per lane of warp 0.
  if (warp == 0) {
    const char* rowp = static_cast<const char*>(logits) + e0 * (kBf16 ? 2 : 4);
    int idx = -1;
    if (rank == 0 && lane < head) idx = lane;
    if (rank == S - 1 && lane >= 16 && lane - 16 < tail) idx = head + nvec * EPV + (lane - 16);
    const bool has = idx >= 0;
    const uint32_t bal = __ballot_sync(kFull, has);
    int start = 0;
    if (lane == 0 && bal) start = atomicAdd(&s_cnt, __popc(bal));
    start = __shfl_sync(kFull, start, 0);
    if (has) {
      uint32_t bits;
      if constexpr (kBf16) {
        bits = static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rowp)[idx]) << 16;
      } else {
        bits = reinterpret_cast<const uint32_t*>(rowp)[idx];
      }
      s_buf[start + __popc(bal & ((1u << lane) - 1))] = make_key(bits, idx);
    }
  }
  __syncthreads();
  select_top(s_buf, s_cnt, K, s_keep);

  if (S > 1) {
    // Push this block's K keys into block 0 of the cluster, then block 0 merges S*K keys.
    if (threadIdx.x < K) {
      const uint32_t dst = map_to_rank(smem_u32(&s_cluster[rank * K + threadIdx.x]), 0);
      st_cluster_u64(dst, s_keep[threadIdx.x]);
    }
    cluster_sync();
    if (rank != 0) return;
    int tot = S * K;
    // drop empty slots (blocks whose segment held fewer than K elements) before ranking
    select_top(s_cluster, tot, K, s_keep);
  }
  if (threadIdx.x < K) {
    const uint64_t x = s_keep[threadIdx.x];
    vals[row * K + threadIdx.x] = key_value(x);
    ids[row * K + threadIdx.x] = static_cast<int32_t>(key_index(x));
  }
}

template <bool kBf16>
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
  return cudaLaunchKernelEx(&cfg, topk_kernel<kBf16>, logits, V, K, S, vals, ids);
}

// Blocks per row: the split (<= 8) whose grid fills the most of its last wave, preferring
// fewer blocks on ties and keeping every segment at 16 KB or more.
int auto_split(int rows, int V, bool bf16) {
  static int slots = 0;
  if (slots == 0) {
    int dev = 0, sms = 152, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (bf16)
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<true>, kThreads, 0);
    else
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<false>, kThreads, 0);
    slots = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t row_bytes = static_cast<int64_t>(V) * (bf16 ? 2 : 4);
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= kMaxSplit; ++s) {
    if (s > 1 && row_bytes / s < 16 * 1024) break;
    const double waves = static_cast<double>(rows) * s / slots;
    const double eff = waves / std::ceil(waves);
    if (eff > best_eff + 1e-3) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_topk(const void* logits, bool is_bf16, int rows, int V, int K, int ctas_per_row, float* vals,
                        int32_t* ids, cudaStream_t stream) {
  if (rows > 65535 || K > kMaxK) return cudaErrorInvalidConfiguration;
  int S = ctas_per_row > 0 ? ctas_per_row : auto_split(rows, V, is_bf16);
  S = S < 1 ? 1 : (S > kMaxSplit ? kMaxSplit : S);
  return is_bf16 ? launch_topk_t<true>(logits, rows, V, K, S, vals, ids, stream)
                 : launch_topk_t<false>(logits, rows, V, K, S, vals, ids, stream);
}

}  // namespace dcoco
