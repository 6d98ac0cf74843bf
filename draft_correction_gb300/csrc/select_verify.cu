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
//              q(v) 1[v != y_j] / (1 - q(y_j)) by inverse CDF in vocabulary order.  Running
//              sums are in float64: each thread sums one contiguous chunk of the row, the
//              chunk totals are prefixed in chunk order, and only the chunk holding the
//              crossing is rescanned, with the same additions.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxB = 64;
constexpr int kStageFloats = 8 * 1024;  // score grid staged in shared memory up to 32 KB
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
__device__ __forceinline__ int warp_argmax(const float* row, int K, int lane) {
  const uint32_t a = lane < K ? ord32(__float_as_uint(row[lane])) : 0u;
  const uint32_t b = lane + 32 < K ? ord32(__float_as_uint(row[lane + 32])) : 0u;
  return warp_argmax_ord(a, b, lane);
}

__global__ void __launch_bounds__(kThreads) select_verify_kernel(const SelectVerifyArgs a) {
  __shared__ uint32_t s_S[kStageFloats];  // order codes of the stream's scores
  __shared__ int32_t s_draft[kMaxB];
  __shared__ int32_t s_k[kMaxB];       // walk: chosen candidate per slot
  __shared__ float s_V[64];            // whole-path rule: best path score ending at each candidate
  __shared__ uint8_t s_back[kMaxB][64];  // whole-path rule: best predecessor of each candidate
  __shared__ int32_t s_t[kMaxB + 1];   // greedy verification: the verifier's tokens
  __shared__ int s_A;
  __shared__ double s_part[kThreads];
  __shared__ double s_pre[kThreads];
  __shared__ int s_pick;
  __shared__ double s_R, s_target;

  const int n = blockIdx.x;
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
    if (staged) {
      // greedy walk: order codes (argmax by integer max); whole-path rule: values, NaN as -inf
      for (size_t i = threadIdx.x; i < grid_floats; i += kThreads)
        s_S[i] = greedy ? ord32(__float_as_uint(Sn[i])) : __float_as_uint(canon(Sn[i]));
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
        s_V[lane] = v0;
        s_V[lane + 32] = v1;
        __syncwarp();
        const size_t base = static_cast<size_t>(p) * K * K;
        float best[2] = {-INFINITY, -INFINITY};
        int arg[2] = {0, 0};
        for (int q = 0; q < K; ++q) {
          const float vq = s_V[q];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int b = lane + 32 * h;
            if (b < K) {
              const float sv = staged ? __uint_as_float(s_S[base + static_cast<size_t>(q) * K + b])
                                      : canon(Sn[base + static_cast<size_t>(q) * K + b]);
              const float c = vq + w * sv;
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
        __syncwarp();
      }
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
      int k = warp_argmax(a.vals + static_cast<size_t>(n) * B * K, K, lane);
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
        const int32_t tok = idn[static_cast<size_t>(j) * K + kj];
        s_draft[j] = tok;
        a.k_sel[static_cast<size_t>(n) * B + j] = kj;
        a.tokens[static_cast<size_t>(n) * B + j] = tok;
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

  // ------------------------------------------------------------------ stochastic draw
  // Row A of q: the residual at the first rejected slot, or the bonus position B (q itself) when
  // every slot was accepted.  Point-mass proposal: q without the draft token; general draft
  // distribution: max(0, q - p), each difference exact in float64.
  const int fallback = A < B ? s_draft[A] : -1;  // kept when there is no residual mass
  const int excl = (A < B && a.mode == 1) ? s_draft[A] : -1;
  const float* row = a.q + (static_cast<size_t>(n) * (B + 1) + A) * V;
  const float* prow = (A < B && a.mode == 2) ? a.p + (static_cast<size_t>(n) * B + A) * V : nullptr;
  auto mass = [&](int v) -> double {
    if (prow != nullptr) return fmax(0.0, static_cast<double>(row[v]) - static_cast<double>(prow[v]));
    return v == excl ? 0.0 : static_cast<double>(row[v]);
  };
  const double u1 = static_cast<double>(a.u[(static_cast<size_t>(n) * (B + 1) + A) * 2 + 1]);
  const int chunk = (V + kThreads - 1) / kThreads;
  const int c0 = min(V, static_cast<int>(threadIdx.x) * chunk), c1 = min(V, c0 + chunk);
  double part = 0.0;
  for (int v = c0; v < c1; ++v) part += mass(v);
  s_part[threadIdx.x] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    double run = 0.0;
    for (int t = 0; t < kThreads; ++t) {
      s_pre[t] = run;
      run += s_part[t];
    }
    const double R = run, target = u1 * R;
    int pick = -1;
    if (R > 0.0) {
      for (int t = 0; t < kThreads; ++t) {
        if (s_part[t] > 0.0 && target - s_pre[t] < s_part[t]) {
          pick = t;
          break;
        }
      }
    }
    s_R = R;
    s_target = target;
    s_pick = pick;
  }
  __syncthreads();
  const int pick = s_pick;
  const double R = s_R, target = s_target;
  if (pick >= 0 && static_cast<int>(threadIdx.x) == pick) {
    // Rescan the crossing chunk with the same additions as its partial sum: a crossing exists
    // because the chunk's full sum exceeds target - prefix.
    const double d = target - s_pre[pick];
    double run = 0.0, before = 0.0;
    int v_pick = c1 - 1;
    for (int v = c0; v < c1; ++v) {
      const double m = mass(v);
      if (m == 0.0) continue;  // no mass: cannot be the crossing (the running sum is unchanged)
      before = run;
      run += m;
      if (run > d) {
        v_pick = v;
        break;
      }
    }
    const double tol = 1e-9 * R;
    const bool near = fabs(s_pre[pick] + run - target) <= tol || fabs(s_pre[pick] + before - target) <= tol;
    com[A] = v_pick;
    if (a.near_tie) a.near_tie[n] = near ? 1 : 0;
  } else if (pick < 0 && threadIdx.x == 0) {
    // R <= 0: no residual mass, the draft token stays.  Otherwise the crossing was lost to
    // rounding at the end of the row: the last token with mass.
    int v = fallback;
    if (R > 0.0) {
      for (int w = V - 1; w >= 0; --w)
        if (mass(w) > 0.0) {
          v = w;
          break;
        }
    }
    com[A] = v;
    if (a.near_tie) a.near_tie[n] = 1;
  }
  if (threadIdx.x == 0) {
    a.accept_len[n] = A;
    a.n_commit[n] = A + 1;
  }
  for (int j = threadIdx.x; j < A; j += kThreads) com[j] = s_draft[j];
  for (int j = A + 1 + static_cast<int>(threadIdx.x); j <= B; j += kThreads) com[j] = -1;
}

}  // namespace

cudaError_t launch_select_verify(const SelectVerifyArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.N, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return cudaLaunchKernelEx(&cfg, select_verify_kernel, a);
}

}  // namespace dcoco
