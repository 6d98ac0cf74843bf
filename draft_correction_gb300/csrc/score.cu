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
// One thread block handles one transition (n, p) and AB = 8 predecessor rows a.  Per chunk of
// HC hidden units it stages, in shared memory,
//   P[a][h] = (uz[n,p,a,h] + ws[n,p,h] + u_a[h] l_p(a) + b1[h]) / 2
//   Q[b][h] = (vz[n,p+1,b,h] + u_b[h] l_{p+1}(b)) / 2
// so that with x = 2(P + Q):  SiLU(x) = x sigmoid(x) = y + y tanh(y), y = P + Q.
// Each thread owns a 2 x 4 tile of (a, b) outputs over a strided subset of the hidden units
// (7 shared-memory vector loads per 32 SiLUs); the partial sums are then added in a fixed
// order.  For bf16 inputs the tanh runs as packed half-precision SFU instructions (two values
// each; pre-activations and sums stay fp32); for f32 inputs as tanh.approx.f32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 256;
constexpr int kAB = 8;    // predecessor rows per block
constexpr int kTA = 2;    // predecessor rows per thread tile
constexpr int kTB = 4;    // successor rows per thread tile
constexpr int kHC = 128;  // hidden units per shared-memory chunk (at most)
constexpr int kPad = 4;   // row padding (floats): neighbouring rows start in different banks

// Hidden units per shared-memory chunk: all of H up to 128, else 128 or 64, whichever divides H
// (H is a multiple of 64), so every chunk is full.
__host__ __device__ __forceinline__ int score_chunk(int H) {
  return H <= kHC ? H : (H % 128 == 0 ? 128 : 64);
}

template <bool kBf16>
__device__ __forceinline__ float ldv(const void* p, size_t i) {
  if constexpr (kBf16) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  } else {
    return static_cast<const float*>(p)[i];
  }
}

// Eight consecutive activations (16 bytes of bf16 or 32 bytes of f32) widened to float.
template <bool kBf16>
__device__ __forceinline__ void ld8(const void* p, size_t i, float (&x)[8]) {
  if constexpr (kBf16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(u[j] << 16);
      x[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Eight consecutive activations of a shared-memory row widened to float.
template <bool kBf16, typename Act>
__device__ __forceinline__ void ld8_smem(const Act* p, float (&x)[8]) {
  if constexpr (kBf16) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(u[j] << 16);
      x[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// sum over 8 hidden units of w * SiLU(2y) / 2 ... written as w * (y + y tanh(y)) with y = p + q,
// in packed half precision; returns the two interleaved partial sums.
__device__ __forceinline__ __half2 silu_dot8(const uint4& p, const uint4& q, const uint4& w) {
  const uint32_t pp[4] = {p.x, p.y, p.z, p.w}, qq[4] = {q.x, q.y, q.z, q.w}, ww[4] = {w.x, w.y, w.z, w.w};
  __half2 acc = __float2half2_rn(0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 y = __hadd2(*reinterpret_cast<const __half2*>(&pp[k]), *reinterpret_cast<const __half2*>(&qq[k]));
    uint32_t t;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&y)));
    const __half2 sv = __hfma2(y, *reinterpret_cast<const __half2*>(&t), y);
    acc = __hfma2(*reinterpret_cast<const __half2*>(&ww[k]), sv, acc);
  }
  return acc;
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh of four floats with two packed half-precision SFU instructions.  Inputs beyond the half
// range round to +-inf, whose tanh is the exact limit +-1, so no input is out of range.
__device__ __forceinline__ void tanh4_f16(float a, float b, float c, float d, float& ta, float& tb, float& tc,
                                          float& td) {
  uint32_t p0, p1, r0, r1;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(p0) : "f"(b), "f"(a));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(p1) : "f"(d), "f"(c));
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(r0) : "r"(p0));
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(r1) : "r"(p1));
  const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&r0));
  const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&r1));
  ta = f0.x;
  tb = f0.y;
  tc = f1.x;
  td = f1.y;
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) score_kernel(const ScoreArgs a) {
  using Act = typename std::conditional<kBf16, __nv_bfloat16, float>::type;
  extern __shared__ __align__(16) float sm[];
  const int K = a.K, H = a.H, B = a.B;
  const int np = blockIdx.x;  // n * (B-1) + p
  const int n = np / (B - 1), p = np % (B - 1);
  const int a0 = blockIdx.y * kAB;
  const int na = min(kAB, K - a0);
  const int Kp = (K + kTB - 1) / kTB * kTB;  // successor rows padded to the thread tile
  const int hc = score_chunk(H);  // 64 or 128
  const int hc_shift = hc == 128 ? 7 : 6;
  const int ld = hc + kPad;   // row pitch of P and Q in floats (f32 path)
  const int ldh = hc + 8;     // row pitch in halves (bf16 path): rows start on 16-byte boundaries
  const int rows = kAB + Kp;
  float* w2v = sm;            // [H]  output weights
  float* uav = w2v + H;       // [H]  u_a
  float* ubv = uav + H;       // [H]  u_b
  float* bwv = ubv + H;       // [H]  b1 + W s_p
  __half* w2h = reinterpret_cast<__half*>(bwv + H);  // [H] output weights in half precision
  float* P = bwv + H + H / 2;  // [kAB][ld]   current chunk (halves on the bf16 path)
  float* Q = P + kAB * ld;    // [Kp][ld]
  float* red = Q + Kp * ld;   // [kThreads][kTA * kTB] partial sums
  Act* raw = reinterpret_cast<Act*>(red + kThreads * kTA * kTB);  // [rows][hc] next chunk, as stored

  // Thread tiles: OT = (kAB/kTA) x (Kp/kTB); HS threads share a tile and split the hidden units.
  // Tile (ta, tb) holds predecessor rows ta*kTA + i and successor rows tb + j*tiles_b (strided, so
  // that neighbouring threads read rows in different shared-memory banks).
  const int tiles_b = Kp / kTB;
  const int OT = (kAB / kTA) * tiles_b;
  const int HS = kThreads / OT;  // OT <= 64 (K <= 64), so HS >= 4
  const int ot = threadIdx.x % OT, hs = threadIdx.x / OT;
  const bool active = hs < HS;
  const int ta = ot / tiles_b, tb = ot % tiles_b;

  const size_t row_p = (static_cast<size_t>(n) * B + p) * K;      // candidate rows of slot p
  const size_t row_q = (static_cast<size_t>(n) * B + p + 1) * K;  // candidate rows of slot p+1
  const float* vals_p = a.vals + row_p;
  const float* vals_q = a.vals + row_q;
  const float* wsp = a.wsp + static_cast<size_t>(np) * H;
  const int cpr = hc * static_cast<int>(sizeof(Act)) / 16;  // 16-byte pieces per row and chunk

  // Raw rows of one chunk (predecessor rows from uz, successor rows from vz) by cp.async.
  auto fetch = [&](int h0) {
    const uint32_t base = smem_u32(raw);
    for (int i = threadIdx.x; i < rows * cpr; i += kThreads) {
      const int r = i / cpr, c = i - r * cpr;
      const Act* src = nullptr;
      if (r < kAB) {
        if (r < na) src = static_cast<const Act*>(a.uz) + (row_p + a0 + r) * H + h0;
      } else if (r - kAB < K) {
        src = static_cast<const Act*>(a.vz) + (row_q + r - kAB) * H + h0;
      }
      if (src != nullptr) cp_async16(base + (r * hc) * sizeof(Act) + c * 16, reinterpret_cast<const char*>(src) + c * 16, 16);
    }
    cp_async_commit();
  };
  fetch(0);
  for (int i = threadIdx.x; i < H; i += kThreads) {
    w2v[i] = ldv<kBf16>(a.w2, i);
    uav[i] = ldv<kBf16>(a.u_a, i);
    ubv[i] = ldv<kBf16>(a.u_b, i);
    bwv[i] = ldv<kBf16>(a.b1, i) + wsp[i];
    w2h[i] = __float2half_rn(w2v[i]);
  }

  float acc[kTA][kTB];
#pragma unroll
  for (int i = 0; i < kTA; ++i)
#pragma unroll
    for (int j = 0; j < kTB; ++j) acc[i][j] = 0.f;

  for (int h0 = 0; h0 < H; h0 += hc) {
    cp_async_wait(0);
    __syncthreads();  // this chunk's raw rows and the vectors are visible; P/Q are free
    // P[a][h] = (uz + b1 + W s + u_a l_p(a)) / 2 and Q[b][h] = (vz + u_b l_{p+1}(b)) / 2; rows
    // past na (P) or K (Q) are zero.
    for (int i = threadIdx.x; i < (rows << hc_shift) / 8; i += kThreads) {
      const int r = (i * 8) >> hc_shift, c = (i * 8) & (hc - 1), h = h0 + c;
      float x[8];
      float* dst;
      if (r < kAB) {
        dst = kBf16 ? reinterpret_cast<float*>(reinterpret_cast<__half*>(P) + r * ldh + c) : P + r * ld + c;
        if (r < na) {
          ld8_smem<kBf16>(raw + r * hc + c, x);
          const float l = vals_p[a0 + r];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.5f * (x[e] + bwv[h + e] + uav[h + e] * l);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
      } else {
        const int rb = r - kAB;
        dst = kBf16 ? reinterpret_cast<float*>(reinterpret_cast<__half*>(Q) + rb * ldh + c) : Q + rb * ld + c;
        if (rb < K) {
          ld8_smem<kBf16>(raw + r * hc + c, x);
          const float l = vals_q[rb];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.5f * (x[e] + ubv[h + e] * l);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
      }
      if constexpr (kBf16) {
        // half precision, clamped to +-30000 so that a sum of two never overflows
        __half2* d16 = reinterpret_cast<__half2*>(dst);  // rows of ld halves
        uint4 w;
        __half2 hh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          hh[e] = __floats2half2_rn(fminf(fmaxf(x[2 * e], -30000.f), 30000.f),
                                    fminf(fmaxf(x[2 * e + 1], -30000.f), 30000.f));
        w.x = *reinterpret_cast<uint32_t*>(&hh[0]);
        w.y = *reinterpret_cast<uint32_t*>(&hh[1]);
        w.z = *reinterpret_cast<uint32_t*>(&hh[2]);
        w.w = *reinterpret_cast<uint32_t*>(&hh[3]);
        *reinterpret_cast<uint4*>(d16) = w;
      } else {
        *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
      }
    }
    __syncthreads();  // P/Q ready; the raw buffer is free for the next chunk
    if (h0 + hc < H) fetch(h0 + hc);
    if (active) {
      if constexpr (kBf16) {
        // Packed half precision: 8 hidden units per step, two per instruction.  Each output keeps
        // an f16 pair of partial sums for the step and adds it to its fp32 total.
        const uint4* p8 = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(P) + ta * kTA * ldh);
        const uint4* q8 = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(Q) + tb * ldh);
        const uint4* w8 = reinterpret_cast<const uint4*>(w2h + h0);
        const int ld8 = ldh / 8;
        for (int c = hs; c < hc / 8; c += HS) {
          const uint4 w = w8[c];
          uint4 pv[kTA], qv[kTB];
#pragma unroll
          for (int i = 0; i < kTA; ++i) pv[i] = p8[i * ld8 + c];
#pragma unroll
          for (int j = 0; j < kTB; ++j) qv[j] = q8[j * tiles_b * ld8 + c];
#pragma unroll
          for (int i = 0; i < kTA; ++i) {
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
              __half2 sacc = silu_dot8(pv[i], qv[j], w);
              const float2 f = __half22float2(sacc);
              acc[i][j] += f.x + f.y;
            }
          }
        }
      } else {
        const float4* w4 = reinterpret_cast<const float4*>(w2v + h0);
        const float4* p4 = reinterpret_cast<const float4*>(P + ta * kTA * ld);
        const float4* q4 = reinterpret_cast<const float4*>(Q + tb * ld);
        const int ld4 = ld / 4;
        for (int c = hs; c < hc / 4; c += HS) {
          const float4 w = w4[c];
          float4 pv[kTA], qv[kTB];
#pragma unroll
          for (int i = 0; i < kTA; ++i) pv[i] = p4[i * ld4 + c];
#pragma unroll
          for (int j = 0; j < kTB; ++j) qv[j] = q4[j * tiles_b * ld4 + c];
#pragma unroll
          for (int i = 0; i < kTA; ++i) {
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
              const float y0 = pv[i].x + qv[j].x, y1 = pv[i].y + qv[j].y;
              const float y2 = pv[i].z + qv[j].z, y3 = pv[i].w + qv[j].w;
              float s = acc[i][j];
              s = fmaf(w.x, fmaf(y0, tanh_fast(y0), y0), s);
              s = fmaf(w.y, fmaf(y1, tanh_fast(y1), y1), s);
              s = fmaf(w.z, fmaf(y2, tanh_fast(y2), y2), s);
              s = fmaf(w.w, fmaf(y3, tanh_fast(y3), y3), s);
              acc[i][j] = s;
            }
          }
        }
      }
    }
  }

  // Add the HS partial sums of every output in a fixed order.
#pragma unroll
  for (int i = 0; i < kTA; ++i)
#pragma unroll
    for (int j = 0; j < kTB; ++j) red[threadIdx.x * (kTA * kTB) + i * kTB + j] = active ? acc[i][j] : 0.f;
  __syncthreads();
  const float b2 = ldv<kBf16>(a.b2, 0);
  float* Sp = a.S + (static_cast<size_t>(np) * K + a0) * K;  // rows a0.. of this transition
  for (int o = threadIdx.x; o < na * K; o += kThreads) {
    const int ar = o / K, bc = o % K;
    const int t = (ar / kTA) * tiles_b + bc % tiles_b;
    const int idx = (ar % kTA) * kTB + bc / tiles_b;
    float s = 0.f;
    for (int h = 0; h < HS; ++h) s += red[(h * OT + t) * (kTA * kTB) + idx];
    Sp[o] = vals_q[bc] + s + b2;
  }
}

}  // namespace

size_t score_smem_bytes(int H, int K, bool is_bf16) {
  const int hc = score_chunk(H);
  const int ld = hc + kPad;
  const int Kp = (K + kTB - 1) / kTB * kTB;
  // vectors, P and Q, partial sums, and one chunk of raw rows
  return (4 * static_cast<size_t>(H) + H / 2 + static_cast<size_t>(kAB + Kp) * ld + kThreads * kTA * kTB) * sizeof(float) +
         static_cast<size_t>(kAB + Kp) * hc * (is_bf16 ? 2 : 4);
}

cudaError_t launch_scores(const ScoreArgs& a, bool is_bf16, cudaStream_t stream) {
  const size_t smem = score_smem_bytes(a.H, a.K, is_bf16);
  dim3 grid(a.N * (a.B - 1), (a.K + kAB - 1) / kAB);
  // The dynamic shared memory ceiling is raised once per device to the largest this kernel
  // can need (K = 64), so later calls enqueue only the launch (CUDA-graph friendly).
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const int most = 227 * 1024;
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
