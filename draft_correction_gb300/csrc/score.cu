// a4. Transition scores of every candidate pair of neighbouring slots.
//
// Two Delta blog, "Score neighboring candidates in parallel", and jaehun.me review of
// arXiv 2610.12570 §3.2: all (B-1)K^2 transitions are scored at once with one shared
// two-layer MLP,
//   S_p(a,b) = l_{p+1}(b) + w2 . SiLU(U z_{p,a} + V z_{p+1,b} + W s_p + u_a l_p(a) + u_b l_{p+1}(b) + b1) + b2.
// The per-candidate (U z, V z) and per-pair (W s) blocks of the first layer are computed
// once upstream; this kernel forms the K x K broadcast sum on chip and never writes the
// [K, K, H] hidden layer to memory.
//
// One thread block handles one transition (n, p) and AB predecessor rows a.  Per chunk of
// HC hidden units it stages, in shared memory,
//   P[a][h] = (uz[n,p,a,h] + ws[n,p,h] + u_a[h] l_p(a) + b1[h]) / 2
//   Q[b][h] = (vz[n,p+1,b,h] + u_b[h] l_{p+1}(b)) / 2
// so that with x = 2(P + Q):  SiLU(x) = x sigmoid(x) = y + y tanh(y), y = P + Q.
// The tanh uses the SFU's tanh.approx.f32 (one instruction per hidden unit and pair).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 128;
constexpr int kAB = 4;    // predecessor rows per block
constexpr int kHC = 256;  // hidden units per shared-memory chunk
constexpr int kPad = 4;   // row padding (floats): neighbouring rows start in different banks

template <bool kBf16>
__device__ __forceinline__ float ldv(const void* p, size_t i) {
  if constexpr (kBf16) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  } else {
    return static_cast<const float*>(p)[i];
  }
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) score_kernel(const ScoreArgs a) {
  extern __shared__ float sm[];
  const int K = a.K, H = a.H, B = a.B;
  const int np = blockIdx.x;  // n * (B-1) + p
  const int n = np / (B - 1), p = np % (B - 1);
  const int a0 = blockIdx.y * kAB;
  const int na = min(kAB, K - a0);
  const int hc = min(H, kHC);
  const int ld = hc + kPad;
  float* P = sm;            // [kAB][ld]
  float* Q = P + kAB * ld;  // [K][ld]
  float* w2c = Q + K * ld;  // [hc]
  float* red = w2c + hc;    // [HS][nout], HS * nout <= kThreads

  // Work split: nout = na*K outputs.  With nout < kThreads, HS threads share one output and
  // split its hidden units; otherwise each thread owns outputs o, o + kThreads (at most 2).
  const int nout = na * K;
  const int HS = nout >= kThreads ? 1 : kThreads / nout;
  const int o = threadIdx.x % nout, hs = threadIdx.x / nout;
  const int n_mine = (hs < HS) ? (HS == 1 ? (nout - o + kThreads - 1) / kThreads : 1) : 0;

  const size_t row_p = (static_cast<size_t>(n) * B + p) * K;      // candidate rows of slot p
  const size_t row_q = (static_cast<size_t>(n) * B + p + 1) * K;  // candidate rows of slot p+1
  const float* vals_p = a.vals + row_p;
  const float* vals_q = a.vals + row_q;
  const float* wsp = a.wsp + static_cast<size_t>(np) * H;

  float acc0 = 0.f, acc1 = 0.f;
  for (int h0 = 0; h0 < H; h0 += hc) {
    __syncthreads();
    for (int i = threadIdx.x; i < kAB * hc; i += kThreads) {
      const int r = i / hc, c = i % hc, h = h0 + c;
      float v = 0.f;
      if (r < na) {
        v = ldv<kBf16>(a.uz, (row_p + a0 + r) * H + h) + wsp[h] + ldv<kBf16>(a.u_a, h) * vals_p[a0 + r] +
            ldv<kBf16>(a.b1, h);
      }
      P[r * ld + c] = 0.5f * v;
    }
    for (int i = threadIdx.x; i < K * hc; i += kThreads) {
      const int r = i / hc, c = i % hc, h = h0 + c;
      Q[r * ld + c] = 0.5f * (ldv<kBf16>(a.vz, (row_q + r) * H + h) + ldv<kBf16>(a.u_b, h) * vals_q[r]);
    }
    for (int i = threadIdx.x; i < hc; i += kThreads) w2c[i] = ldv<kBf16>(a.w2, h0 + i);
    __syncthreads();
    for (int t = 0; t < n_mine; ++t) {
      const int oo = o + t * kThreads;
      const float4* p4 = reinterpret_cast<const float4*>(P + (oo / K) * ld);
      const float4* q4 = reinterpret_cast<const float4*>(Q + (oo % K) * ld);
      const float4* w4 = reinterpret_cast<const float4*>(w2c);
      float s = 0.f;
      for (int c = hs; c < hc / 4; c += HS) {
        const float4 pp = p4[c], qq = q4[c], ww = w4[c];
        float y;
        y = pp.x + qq.x; s = fmaf(ww.x, fmaf(y, tanh_fast(y), y), s);
        y = pp.y + qq.y; s = fmaf(ww.y, fmaf(y, tanh_fast(y), y), s);
        y = pp.z + qq.z; s = fmaf(ww.z, fmaf(y, tanh_fast(y), y), s);
        y = pp.w + qq.w; s = fmaf(ww.w, fmaf(y, tanh_fast(y), y), s);
      }
      if (t == 0) acc0 += s; else acc1 += s;
    }
  }

  const float b2 = ldv<kBf16>(a.b2, 0);
  float* Sp = a.S + (static_cast<size_t>(np) * K + a0) * K;  // rows a0.. of this transition
  if (HS > 1) {
    // Combine the HS partial sums of each output in a fixed order.
    if (hs < HS) red[hs * nout + o] = acc0;
    __syncthreads();
    if (threadIdx.x < nout) {
      float s = 0.f;
      for (int j = 0; j < HS; ++j) s += red[j * nout + threadIdx.x];
      Sp[threadIdx.x] = vals_q[threadIdx.x % K] + s + b2;
    }
  } else {
    if (n_mine > 0) Sp[o] = vals_q[o % K] + acc0 + b2;
    if (n_mine > 1) Sp[o + kThreads] = vals_q[(o + kThreads) % K] + acc1 + b2;
  }
}

}  // namespace

cudaError_t launch_scores(const ScoreArgs& a, bool is_bf16, cudaStream_t stream) {
  const int hc = a.H < kHC ? a.H : kHC;
  const int ld = hc + kPad;
  // P, Q, the w2 chunk, and kThreads floats for combining partial sums (HS * nout <= kThreads)
  const size_t smem = (static_cast<size_t>(kAB + a.K) * ld + hc + kThreads) * sizeof(float);
  dim3 grid(a.N * (a.B - 1), (a.K + kAB - 1) / kAB);
  // The dynamic shared memory ceiling is raised once per device to the largest this kernel
  // can need (K = 64), so later calls enqueue only the launch (CUDA-graph friendly).
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const int most = static_cast<int>((static_cast<size_t>(kAB + 64) * (kHC + kPad) + kHC + kThreads) * sizeof(float));
    e = cudaFuncSetAttribute(score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  if (is_bf16)
    score_kernel<true><<<grid, kThreads, smem, stream>>>(a);
  else
    score_kernel<false><<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dcoco
