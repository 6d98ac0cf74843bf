// a5. Prefix-first greedy walk and a6. verification of the corrected block.
//
// Walk (Two Delta blog, "Select using the realized token identities"; jaehun.me review of
// arXiv 2610.12570 §3.3): slot 0 keeps the drafter's top candidate, every later slot takes
// the best-scoring successor of the candidate actually chosen before it.  It is the only
// sequential step: one warp per stream, the stream's score grid staged in shared memory,
// each step a warp argmax over the K successors (ties to the lower candidate index).
//
// Verification (review §3.1, App. D):
//  greedy      accept while the draft equals the verifier's greedy token; commit the
//              accepted prefix and the verifier's token at the first rejection.
//  stochastic  the corrected draft is a point-mass proposal, so slot j is accepted with
//              probability q_j(y_j) (u < q), and the first rejection draws from the residual
//              q(v) 1[v != y_j] / (1 - q(y_j)) by inverse CDF in vocabulary order.
//  speculative a general draft distribution p: accept iff u p(y) < q(y) (exact in float64),
//              residual max(0, q - p).
// Residual masses are summed exactly in 62-bit fixed point (integer additions, so the order
// does not matter and float64 -- slow on this GPU -- is not needed): super-block sums with
// coalesced loads, one warp's prefix over them, and one warp scan of the crossing super-block.
// For the two sampling modes a stream's vocabulary row is shared by a cluster of up to 8 CTAs,
// each summing a contiguous range of super-blocks; rank 0 reads the others' sums through
// distributed shared memory and makes the draw (integer sums: the same result for any split).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxB = 64;
constexpr int kStageFloats = 8 * 1024;  // score grid staged in shared memory up to 32 KB
constexpr int kIdsStage = 2048;         // candidate ids staged with it (in the draw's 8 KB buffer)
constexpr unsigned kFull = 0xFFFFFFFFu;

// argmax over the order codes row[0..K) (K <= 64; 0 marks no entry): the largest code, the
// lowest index among equal ones.  One warp reduction and a ballot.
__device__ __forceinline__ int warp_argmax_ord(uint32_t a, uint32_t b, int lane) {
  const uint32_t m = __reduce_max_sync(kFull, a > b ? a : b);
  const uint32_t ba = __ballot_sync(kFull, a == m);
  if (ba) return __ffs(ba) - 1;
  return 32 + __ffs(__ballot_sync(kFull, b == m)) - 1;
}
__device__ __forceinline__ float canon(float x) { return x != x ? -INFINITY : x; }  // NaN ranks lowest

constexpr int kMaxSB = 1024;  // super-blocks of a vocabulary row in the residual draw
constexpr int kDrawU = 8;     // loads per row in flight per lane while summing them

// A probability as unsigned fixed point with 62 fractional bits (range [0, 4)): exact for every
// float32 at or above 2^-38; smaller values round down (by less than 2^-62); NaN, negatives and
// zero give 0; values of 4 or more saturate.
__device__ __forceinline__ uint64_t to_fx(float x) {
  if (!(x > 0.f)) return 0;
  if (x >= 4.f) return ~0ull >> 1;
  const uint32_t b = __float_as_uint(x);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  const uint64_t m = (b & 0x7FFFFFu) | (e != 0 ? 0x800000u : 0u);
  const int sh = (e != 0 ? e : 1) - 150 + 62;  // x = m 2^(e-150); fixed = m 2^(e-150+62)
  return sh >= 0 ? (m << sh) : (sh <= -64 ? 0ull : (m >> -sh));
}
// floor(R u) for u in [0, 1) given as float32 (exact: 64 x 24-bit product).
__device__ __forceinline__ uint64_t mul_floor(uint64_t R, float u) {
  if (!(u > 0.f)) return 0;
  const uint32_t b = __float_as_uint(u);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  const uint64_t m = (b & 0x7FFFFFu) | (e != 0 ? 0x800000u : 0u);
  const int s = 150 - (e != 0 ? e : 1);  // u = m 2^-s, s >= 24 for u < 1
  const uint64_t lo = R * m, hi = __umul64hi(R, m);
  if (s >= 128) return 0;
  if (s >= 64) return hi >> (s - 64);
  return (hi << (64 - s)) | (lo >> s);
}
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
__device__ __forceinline__ float warp_sum_f32(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
// inclusive prefix sum across the warp
__device__ __forceinline__ uint64_t warp_scan_u64(uint64_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
__device__ __forceinline__ int warp_argmax(const float* row, int K, int lane) {
  const uint32_t a = lane < K ? ord32(__float_as_uint(row[lane])) : 0u;
  const uint32_t b = lane + 32 < K ? ord32(__float_as_uint(row[lane + 32])) : 0u;
  return warp_argmax_ord(a, b, lane);
}

// kSampling: the instance that also holds the stochastic and speculative draw (modes 1, 2); the
// other instance (walk, path rules, greedy verification) is compiled without it.
template <bool kSampling>
__global__ void __launch_bounds__(kThreads) select_verify_kernel(const SelectVerifyArgs a) {
  __shared__ uint32_t s_S[kStageFloats];  // order codes of the stream's scores
  __shared__ int32_t s_draft[kMaxB];
  __shared__ int32_t s_k[kMaxB];       // walk: chosen candidate per slot
  __shared__ uint8_t s_back[kMaxB][64];  // whole-path rule: best predecessor of each candidate
  __shared__ int32_t s_t[kMaxB + 1];   // greedy verification: the verifier's tokens
  __shared__ int s_A;
  __shared__ uint64_t s_sb[kMaxSB];       // residual mass of each super-block (fixed point)
  __shared__ float s_fsum[kThreads / 32];
  __shared__ uint64_t s_draw[6];  // R, T, found, crossing super-block, mass before it, flag

  const int n = blockIdx.y;
  const int C = gridDim.x, rank = blockIdx.x;  // CTAs of this stream's cluster (1 unless sampling)
  const int B = a.B, K = a.K, V = a.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait();  // scores, logits and ids come from preceding kernels
  grid_dep_launch();

  // ------------------------------------------------------------------ walk
  if (a.S != nullptr) {
    const size_t grid_floats = static_cast<size_t>(B - 1) * K * K;
    const float* Sn = a.S + static_cast<size_t>(n) * grid_floats;
    const bool staged = grid_floats <= static_cast<size_t>(kStageFloats);
    const bool greedy = a.rule == 0;
    // first-slot logits and candidate ids staged with the grid (greedy walk, B K <= kIdsStage)
    const bool pre = staged && greedy && B * K <= kIdsStage;
    uint32_t* s_v0 = reinterpret_cast<uint32_t*>(s_draft);  // read by warp 0 before it writes s_draft
    int32_t* s_ids = reinterpret_cast<int32_t*>(s_sb);      // the residual draw uses s_sb only later
    if (staged) {
      // greedy walk: order codes (argmax by integer max); whole-path rule: values, NaN as -inf.
      // Every thread issues all its loads before storing any, so they are in flight together;
      // for the greedy walk the first slot's logits and the stream's candidate ids come in the
      // same batch, so the walk and the token look-up touch only shared memory.
      constexpr int kPer = kStageFloats / kThreads;
      constexpr int kIdPer = kIdsStage / kThreads;
      float x[kPer];
      int32_t idv[kIdPer];
      float v0 = 0.f;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const size_t i = threadIdx.x + static_cast<size_t>(q) * kThreads;
        x[q] = i < grid_floats ? Sn[i] : 0.f;
      }
      if (pre) {
        const size_t base = static_cast<size_t>(n) * B * K;
        if (static_cast<int>(threadIdx.x) < K) v0 = a.vals[base + threadIdx.x];
#pragma unroll
        for (int q = 0; q < kIdPer; ++q) {
          const int i = static_cast<int>(threadIdx.x) + q * kThreads;
          idv[q] = i < B * K ? a.ids[base + i] : 0;
        }
      }
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const size_t i = threadIdx.x + static_cast<size_t>(q) * kThreads;
        if (i < grid_floats) s_S[i] = greedy ? ord32(__float_as_uint(x[q])) : __float_as_uint(canon(x[q]));
      }
      if (pre) {
        if (static_cast<int>(threadIdx.x) < K) s_v0[threadIdx.x] = ord32(__float_as_uint(v0));
#pragma unroll
        for (int q = 0; q < kIdPer; ++q) {
          const int i = static_cast<int>(threadIdx.x) + q * kThreads;
          if (i < B * K) s_ids[i] = idv[q];
        }
      }
    }
    __syncthreads();
    if (warp == 0 && !greedy) {
      // Discounted max-sum over all paths (lambda = 1: Global-Sum): lane l owns candidates l and
      // l + 32; V_{p+1}(b) = max_a V_p(a) + lambda^(p+1) S_p(a, b), lowest a among equal values.
      float v0 = lane < K ? canon(a.vals[static_cast<size_t>(n) * B * K + lane]) : -INFINITY;
      float v1 = lane + 32 < K ? canon(a.vals[static_cast<size_t>(n) * B * K + lane + 32]) : -INFINITY;
      float w = 1.f;
      for (int p = 0; p + 1 < B; ++p) {
        w *= a.lam;
        const size_t base = static_cast<size_t>(p) * K * K;
        float best[2] = {-INFINITY, -INFINITY};
        int arg[2] = {0, 0};
        auto S_at = [&](int q, int b) -> float {
          return staged ? __uint_as_float(s_S[base + static_cast<size_t>(q) * K + b])
                        : canon(Sn[base + static_cast<size_t>(q) * K + b]);
        };
        if (K <= 32) {
#pragma unroll 4
          for (int q = 0; q < K; ++q) {
            const float vq = __shfl_sync(kFull, v0, q);  // the best score ending at candidate q
            const float c = vq + w * (lane < K ? S_at(q, lane) : 0.f);
            if (c > best[0]) {
              best[0] = c;
              arg[0] = q;
            }
          }
        } else {
#pragma unroll 2
          for (int q = 0; q < K; ++q) {
            const float vq = __shfl_sync(kFull, q < 32 ? v0 : v1, q & 31);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int b = lane + 32 * h;
              const float c = vq + w * (b < K ? S_at(q, b) : 0.f);
              if (c > best[h]) {
                best[h] = c;
                arg[h] = q;
              }
            }
          }
        }
        if (lane < K) s_back[p + 1][lane] = static_cast<uint8_t>(arg[0]);
        if (lane + 32 < K) s_back[p + 1][lane + 32] = static_cast<uint8_t>(arg[1]);
        v0 = lane < K ? best[0] : -INFINITY;
        v1 = lane + 32 < K ? best[1] : -INFINITY;
      }
      __syncwarp();
      int k = warp_argmax_ord(lane < K ? ord32(__float_as_uint(v0)) : 0u, lane + 32 < K ? ord32(__float_as_uint(v1)) : 0u,
                              lane);
      if (lane == 0) {
        s_k[B - 1] = k;
        for (int p = B - 1; p > 0; --p) {
          k = s_back[p][k];
          s_k[p - 1] = k;
        }
      }
      __syncwarp();
    } else if (warp == 0) {
      // The chain of argmaxes touches only shared memory (and registers); the token ids of
      // the chosen candidates are looked up together afterwards.
      int k = pre ? warp_argmax_ord(lane < K ? s_v0[lane] : 0u, lane + 32 < K ? s_v0[lane + 32] : 0u, lane)
                  : warp_argmax(a.vals + static_cast<size_t>(n) * B * K, K, lane);
      if (lane == 0) s_k[0] = k;
      for (int p = 0; p + 1 < B; ++p) {
        const size_t row = (static_cast<size_t>(p) * K + k) * K;
        if (staged) {
          const uint32_t x = lane < K ? s_S[row + lane] : 0u;
          const uint32_t y = lane + 32 < K ? s_S[row + lane + 32] : 0u;
          k = warp_argmax_ord(x, y, lane);
        } else {
          k = warp_argmax(Sn + row, K, lane);
        }
        if (lane == 0) s_k[p + 1] = k;
      }
      __syncwarp();
    }
    if (warp == 0) {
      const int32_t* idn = a.ids + static_cast<size_t>(n) * B * K;
      for (int j = lane; j < B; j += 32) {
        const int kj = s_k[j];
        const int32_t tok = pre ? s_ids[j * K + kj] : idn[static_cast<size_t>(j) * K + kj];
        s_draft[j] = tok;
        if (rank == 0) {
          a.k_sel[static_cast<size_t>(n) * B + j] = kj;
          a.tokens[static_cast<size_t>(n) * B + j] = tok;
        }
      }
    } else if (warp == 1 && a.mode == 0) {
      // the verifier's greedy tokens, fetched while the walk runs
      for (int j = lane; j <= B; j += 32) s_t[j] = a.t[static_cast<size_t>(n) * (B + 1) + j];
    }
  } else if (a.mode >= 0) {
    for (int j = threadIdx.x; j < B; j += kThreads) s_draft[j] = a.draft[static_cast<size_t>(n) * B + j];
    if (a.mode == 0)
      for (int j = threadIdx.x; j <= B; j += kThreads) s_t[j] = a.t[static_cast<size_t>(n) * (B + 1) + j];
  }
  __syncthreads();
  if (a.mode < 0) return;

  // ------------------------------------------------------------------ accept length
  if (warp == 0) {
    uint64_t acc_mask = 0;  // bit j set when slot j is accepted
    for (int base = 0; base < B; base += 32) {
      const int j = base + lane;
      bool ok = false;
      if (j < B) {
        const int32_t y = s_draft[j];
        if (a.mode == 0) {
          ok = (y == s_t[j]);
        } else {
          const float uq = a.u[(static_cast<size_t>(n) * (B + 1) + j) * 2];
          const float qy = (y >= 0 && y < V) ? a.q[(static_cast<size_t>(n) * (B + 1) + j) * V + y] : 0.f;
          if (a.mode == 1) {
            ok = uq < qy;
          } else {  // general draft distribution: u p(y) < q(y), the product exact in float64
            const float py = (y >= 0 && y < V) ? a.p[(static_cast<size_t>(n) * B + j) * V + y] : 0.f;
            ok = static_cast<double>(uq) * static_cast<double>(py) < static_cast<double>(qy);
          }
        }
      }
      acc_mask |= static_cast<uint64_t>(__ballot_sync(kFull, ok)) << base;
    }
    if (lane == 0) {
      const uint64_t rej = ~acc_mask;  // bits >= B are set too
      s_A = (rej == 0) ? 64 : __ffsll(static_cast<long long>(rej)) - 1;
      if (s_A > B) s_A = B;
    }
  }
  __syncthreads();
  const int A = s_A;
  int32_t* com = a.committed + static_cast<size_t>(n) * (B + 1);

  if (a.mode == 0) {
    for (int j = threadIdx.x; j <= B; j += kThreads)
      com[j] = j < A ? s_draft[j] : (j == A ? s_t[A] : -1);
    if (threadIdx.x == 0) {
      a.accept_len[n] = A;
      a.n_commit[n] = A + 1;
    }
    return;
  }
  if constexpr (kSampling) {
  // ------------------------------------------------------------------ stochastic draw
  // Row A of q: the residual at the first rejected slot, or the bonus position B (q itself) when
  // every slot was accepted.  Point-mass proposal: q without the draft token; general draft
  // distribution: max(0, q - p).  Masses are summed exactly in 62-bit fixed point (every
  // probability at or above 2^-38 converts exactly, smaller ones round down by less than 2^-62),
  // so any order of addition gives the same sums: coalesced super-block sums, one warp's prefix
  // over them, then one warp scans the crossing super-block.
  const int fallback = A < B ? s_draft[A] : -1;  // kept when there is no residual mass
  const int excl = (A < B && a.mode == 1) ? s_draft[A] : -1;
  const float* row = a.q + (static_cast<size_t>(n) * (B + 1) + A) * V;
  const float* prow = (A < B && a.mode == 2) ? a.p + (static_cast<size_t>(n) * B + A) * V : nullptr;
  auto mass = [&](int v) -> uint64_t {
    if (v >= V) return 0;
    const uint64_t qq = to_fx(row[v]);
    if (prow != nullptr) {
      const uint64_t pp = to_fx(prow[v]);
      return qq > pp ? qq - pp : 0;
    }
    return v == excl ? 0 : qq;
  };
  const int sb_len = max(1024, (V + kMaxSB - 1) / kMaxSB + 31) & ~31;  // elements per super-block
  const int nsb = (V + sb_len - 1) / sb_len;                             // <= kMaxSB
  auto sb_owner = [&](int sb) { return static_cast<int>((static_cast<int64_t>(sb) * C) / nsb); };
  const int sb_lo = static_cast<int>((static_cast<int64_t>(rank) * nsb + C - 1) / C);  // first sb with owner rank
  const int sb_hi = static_cast<int>((static_cast<int64_t>(rank + 1) * nsb + C - 1) / C);
  float fsum = 0.f;  // plain float total, to flag rows that are not probability vectors
  for (int sb = sb_lo + warp; sb < sb_hi; sb += kThreads / 32) {
    uint64_t acc = 0;
    for (int k = 0; k < sb_len; k += 32 * kDrawU) {  // kDrawU loads of each row in flight per lane
      float qv[kDrawU], pv[kDrawU];
#pragma unroll
      for (int i = 0; i < kDrawU; ++i) {
        const int v = sb * sb_len + k + i * 32 + lane;
        qv[i] = (k + i * 32 < sb_len && v < V) ? row[v] : 0.f;
        pv[i] = (prow != nullptr && k + i * 32 < sb_len && v < V) ? prow[v] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < kDrawU; ++i) {
        const int v = sb * sb_len + k + i * 32 + lane;
        const uint64_t qq = to_fx(qv[i]);
        uint64_t m;
        if (prow != nullptr) {
          const uint64_t pp = to_fx(pv[i]);
          m = qq > pp ? qq - pp : 0;
        } else {
          m = v == excl ? 0 : qq;
        }
        acc += m;
        fsum += qv[i];
      }
    }
    acc = warp_sum_u64(acc);
    if (lane == 0) s_sb[sb] = acc;
  }
  fsum = warp_sum_f32(fsum);
  if (lane == 0) s_fsum[warp] = fsum;
  __syncthreads();
  if (C > 1) {
    // rank 0 collects the other ranks' super-block sums and float partial totals
    cluster_sync();
    if (rank == 0) {
      for (int sb = threadIdx.x; sb < nsb; sb += kThreads) {
        const int o = sb_owner(sb);
        if (o != 0) s_sb[sb] = ld_cluster_u64(map_to_rank(smem_u32(&s_sb[sb]), o));
      }
      if (threadIdx.x < kThreads / 32) {
        float f = s_fsum[threadIdx.x];
        for (int o = 1; o < C; ++o) f += ld_cluster_f32(map_to_rank(smem_u32(&s_fsum[threadIdx.x]), o));
        s_fsum[threadIdx.x] = f;
      }
    }
    cluster_sync();  // no rank leaves while rank 0 reads its shared memory
    if (rank != 0) return;
    __syncthreads();
  }
  if (warp == 0) {
    // prefix over the super-blocks: lane l takes a contiguous run of them
    const int per = (nsb + 31) / 32, s0 = min(nsb, lane * per), s1 = min(nsb, s0 + per);
    uint64_t mine = 0;
    for (int i = s0; i < s1; ++i) mine += s_sb[i];
    const uint64_t incl = warp_scan_u64(mine, lane);
    const uint64_t R = __shfl_sync(kFull, incl, 31);
    float ftot = lane < kThreads / 32 ? s_fsum[lane] : 0.f;
    ftot = warp_sum_f32(ftot);
    const uint64_t T = mul_floor(R, a.u[(static_cast<size_t>(n) * (B + 1) + A) * 2 + 1]);
    // the first super-block whose inclusive prefix exceeds T
    uint64_t run = incl - mine;
    int found = -1;
    uint64_t found_base = 0;
    for (int i = s0; i < s1 && R > 0; ++i) {
      if (run + s_sb[i] > T) {
        found = i;
        found_base = run;
        break;
      }
      run += s_sb[i];
    }
    const uint32_t has = __ballot_sync(kFull, found >= 0);
    if (lane == 0) {
      s_draw[0] = R;
      s_draw[1] = T;
      s_draw[2] = has ? 1u : 0u;
      s_draw[5] = (R < (1ull << 47) || !(ftot < 3.5f)) ? 1u : 0u;  // flag: tiny mass or not a distribution
    }
    if (has) {
      const int src = __ffs(has) - 1;
      const int sb = __shfl_sync(kFull, found, src);
      const uint64_t base = __shfl_sync(kFull, found_base, src);
      if (lane == 0) {
        s_draw[3] = static_cast<uint64_t>(sb);
        s_draw[4] = base;
      }
    }
  }
  __syncthreads();
  if (s_draw[2] != 0) {
    // The crossing super-block: every warp sums 32-element chunks of it (one memory round trip
    // each, in parallel), warp 0 scans the chunk sums and then the one chunk that crosses.
    const uint64_t R = s_draw[0], T = s_draw[1];
    const int sb = static_cast<int>(s_draw[3]);
    const int nch = sb_len / 32;
    if (nch <= kMaxSB) {
      for (int c = warp; c < nch; c += kThreads / 32) {
        const uint64_t cs = warp_sum_u64(mass(sb * sb_len + c * 32 + lane));
        if (lane == 0) s_sb[c] = cs;
      }
    }
    __syncthreads();
    if (warp == 0) {
      uint64_t base = s_draw[4];
      int v_pick = fallback;
      bool near = true;
      const uint64_t tol = R >> 30;  // about 0.93e-9 R
      int c_lo = 0, c_hi = nch;
      if (nch <= kMaxSB) {
        // first chunk whose inclusive prefix exceeds T (lane l takes a contiguous run)
        const int per = (nch + 31) / 32, s0 = min(nch, lane * per), s1 = min(nch, s0 + per);
        uint64_t mine = 0;
        for (int i = s0; i < s1; ++i) mine += s_sb[i];
        const uint64_t incl = warp_scan_u64(mine, lane);
        uint64_t run = base + incl - mine;
        int found = -1;
        uint64_t fb = 0;
        for (int i = s0; i < s1; ++i) {
          if (run + s_sb[i] > T) {
            found = i;
            fb = run;
            break;
          }
          run += s_sb[i];
        }
        const uint32_t hc = __ballot_sync(kFull, found >= 0);
        if (hc) {
          const int src = __ffs(hc) - 1;
          c_lo = __shfl_sync(kFull, found, src);
          c_hi = c_lo + 1;
          base = __shfl_sync(kFull, fb, src);
        }
      }
      for (int c = c_lo; c < c_hi; ++c) {
        const int v = sb * sb_len + c * 32 + lane;
        const uint64_t m = mass(v);
        const uint64_t in = warp_scan_u64(m, lane);
        const uint32_t cross = __ballot_sync(kFull, m > 0 && base + in > T);
        if (cross) {
          const int l = __ffs(cross) - 1;
          const uint64_t after = base + __shfl_sync(kFull, in, l);
          const uint64_t before = after - __shfl_sync(kFull, m, l);
          v_pick = sb * sb_len + c * 32 + l;
          near = (after - T <= tol) || (T >= before ? T - before <= tol : before - T <= tol);
          break;
        }
        base += __shfl_sync(kFull, in, 31);
      }
      // residual mass below 2^-15 (relative truncation error above 1e-9) or rows that are not
      // probability vectors (sums beyond the fixed-point range) are flagged, not trusted
      if (s_draw[5] != 0) near = true;
      if (lane == 0) {
        com[A] = v_pick;
        if (a.near_tie) a.near_tie[n] = near ? 1 : 0;
      }
    }
  } else if (threadIdx.x == 0) {
    com[A] = fallback;
    if (a.near_tie) a.near_tie[n] = 1;
  }
  if (threadIdx.x == 0) {
    a.accept_len[n] = A;
    a.n_commit[n] = A + 1;
  }
  for (int j = threadIdx.x; j < A; j += kThreads) com[j] = s_draft[j];
  for (int j = A + 1 + static_cast<int>(threadIdx.x); j <= B; j += kThreads) com[j] = -1;
  }
}

}  // namespace

cudaError_t launch_select_verify(const SelectVerifyArgs& a, cudaStream_t stream) {
  // Sampling modes read whole vocabulary rows: spread each stream over a cluster so that up to
  // two CTAs per SM (what registers allow) stream them.  The walk and greedy verification stay
  // one CTA per stream.
  const int sms = sm_count();
  int C = 1;
  if (a.mode >= 1)
    while (C < 8 && static_cast<int64_t>(a.N) * C * 2 <= 2 * static_cast<int64_t>(sms)) C *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.N, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  cfg.numAttrs += pdl_attr(&attr[cfg.numAttrs]);
  return a.mode >= 1 ? cudaLaunchKernelEx(&cfg, select_verify_kernel<true>, a)
                     : cudaLaunchKernelEx(&cfg, select_verify_kernel<false>, a);
}

}  // namespace dcoco
