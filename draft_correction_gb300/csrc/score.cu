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
// One thread block handles one transition (n, p) and AB predecessor rows a (8 in score_kernel,
// 4 in the cycle's score_prepped_kernel).  Per chunk of HC hidden units it stages, in shared
// memory,
//   P[a][h] = (uz[n,p,a,h] + ws[n,p,h] + u_a[h] l_p(a) + b1[h]) / 2
//   Q[b][h] = (vz[n,p+1,b,h] + u_b[h] l_{p+1}(b)) / 2
// so that with x = 2(P + Q):  SiLU(x) = x sigmoid(x) = y + y tanh(y), y = P + Q.
// Each thread owns a 2 x 4 tile of (a, b) outputs over a strided subset of the hidden units
// (7 shared-memory vector loads per 32 SiLUs); the partial sums are then added in a fixed
// order.  For bf16 inputs P and Q are kept in half precision, and their sum, the tanh (packed
// half-precision SFU instructions, two values each) and the 8-term partial sums are half
// precision too, each partial sum then added to the output's fp32 total; for f32 inputs
// everything is fp32, with tanh.approx.f32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int kThreads = 256;
constexpr int kAB = 8;    // predecessor rows per block of score_kernel
constexpr int kABP = 4;   // predecessor rows per block of score_prepped_kernel (about two waves at the headline shape)
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

// Thread tiles: OT = (AB/kTA) x (Kp/kTB) for AB predecessor rows per block; HS threads share a
// tile and split the hidden units.
// Tile (ta, tb) holds predecessor rows ta*kTA + i and successor rows tb + j*tiles_b (strided, so
// that neighbouring threads read rows in different shared-memory banks).
struct Tile {
  int tiles_b, OT, HS, hs, ta, tb;
  bool active;
};
template <int NT, int AB>
__device__ __forceinline__ Tile make_tile(int Kp) {
  Tile t;
  t.tiles_b = Kp / kTB;
  t.OT = (AB / kTA) * t.tiles_b;
  t.HS = NT / t.OT;  // OT <= 64 (K <= 64), so HS >= NT / 64
  const int ot = threadIdx.x % t.OT;
  t.hs = threadIdx.x / t.OT;
  t.active = t.hs < t.HS;
  t.ta = ot / t.tiles_b;
  t.tb = ot % t.tiles_b;
  return t;
}

// Adds hc hidden units of w . (y + y tanh y), y = P[a] + Q[b], to the thread's kTA x kTB outputs.
// bf16 path: P, Q and w in half precision (rows of ld halves), 8 units per step, two per
// instruction, with an f16 pair of partial sums per step added to the fp32 total.  f32 path:
// fp32 throughout (rows of ld floats).
template <bool kBf16>
__device__ __forceinline__ void accumulate(float (&acc)[kTA][kTB], const void* P, const void* Q, int ld, const void* w,
                                           int hc, const Tile& t) {
  if (!t.active) return;
  if constexpr (kBf16) {
    const uint4* p8 = reinterpret_cast<const uint4*>(static_cast<const __half*>(P) + t.ta * kTA * ld);
    const uint4* q8 = reinterpret_cast<const uint4*>(static_cast<const __half*>(Q) + t.tb * ld);
    const uint4* w8 = static_cast<const uint4*>(w);
    const int ld8 = ld / 8, qs = t.tiles_b * ld8;
    for (int c = t.hs; c < hc / 8; c += t.HS) {
      const uint4 wv = w8[c];
      uint4 pv[kTA], qv[kTB];
#pragma unroll
      for (int i = 0; i < kTA; ++i) pv[i] = p8[i * ld8 + c];
#pragma unroll
      for (int j = 0; j < kTB; ++j) qv[j] = q8[j * qs + c];
#pragma unroll
      for (int i = 0; i < kTA; ++i) {
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
          const float2 f = __half22float2(silu_dot8(pv[i], qv[j], wv));
          acc[i][j] += f.x + f.y;
        }
      }
    }
  } else {
    const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(P) + t.ta * kTA * ld);
    const float4* q4 = reinterpret_cast<const float4*>(static_cast<const float*>(Q) + t.tb * ld);
    const float4* w4 = static_cast<const float4*>(w);
    const int ld4 = ld / 4, qs = t.tiles_b * ld4;
    for (int c = t.hs; c < hc / 4; c += t.HS) {
      const float4 wv = w4[c];
      float4 pv[kTA], qv[kTB];
#pragma unroll
      for (int i = 0; i < kTA; ++i) pv[i] = p4[i * ld4 + c];
#pragma unroll
      for (int j = 0; j < kTB; ++j) qv[j] = q4[j * qs + c];
#pragma unroll
      for (int i = 0; i < kTA; ++i) {
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
          const float y0 = pv[i].x + qv[j].x, y1 = pv[i].y + qv[j].y;
          const float y2 = pv[i].z + qv[j].z, y3 = pv[i].w + qv[j].w;
          float s = acc[i][j];
          s = fmaf(wv.x, fmaf(y0, tanh_fast(y0), y0), s);
          s = fmaf(wv.y, fmaf(y1, tanh_fast(y1), y1), s);
          s = fmaf(wv.z, fmaf(y2, tanh_fast(y2), y2), s);
          s = fmaf(wv.w, fmaf(y3, tanh_fast(y3), y3), s);
          acc[i][j] = s;
        }
      }
    }
  }
}

// Adds the HS partial sums of every output in a fixed order and writes
// S[n,p,a0+ar,bc] = l_{p+1}(bc) + sum + b2 for the block's na predecessor rows.
template <int NT>
__device__ __forceinline__ void finish(const float (&acc)[kTA][kTB], float* red, const Tile& t, float* Sp,
                                       const float* vals_q, float b2, int na, int K) {
#pragma unroll
  for (int i = 0; i < kTA; ++i)
#pragma unroll
    for (int j = 0; j < kTB; ++j) red[threadIdx.x * (kTA * kTB) + i * kTB + j] = t.active ? acc[i][j] : 0.f;
  __syncthreads();
  for (int o = threadIdx.x; o < na * K; o += NT) {
    const int ar = o / K, bc = o % K;
    const int ti = (ar / kTA) * t.tiles_b + bc % t.tiles_b;
    const int idx = (ar % kTA) * kTB + bc / t.tiles_b;
    float s = 0.f;
    for (int h = 0; h < t.HS; ++h) s += red[(h * t.OT + ti) * (kTA * kTB) + idx];
    Sp[o] = vals_q[bc] + s + b2;
  }
}

// ------------------------------------------------------------------ from uz, vz and W s
// One thread block handles one transition (n, p) and kAB predecessor rows.  Per chunk of HC
// hidden units it stages, in shared memory,
//   P[a][h] = (uz[n,p,a,h] + ws[n,p,h] + u_a[h] l_p(a) + b1[h]) / 2
//   Q[b][h] = (vz[n,p+1,b,h] + u_b[h] l_{p+1}(b)) / 2
// (the raw rows of the next chunk arrive by cp.async while the current chunk computes).
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
  const int ld = kBf16 ? hc + 8 : hc + kPad;  // P/Q row pitch (halves or floats): 16-byte aligned rows
  const int rows = kAB + Kp;
  float* w2v = sm;            // [H]  output weights
  float* uav = w2v + H;       // [H]  u_a
  float* ubv = uav + H;       // [H]  u_b
  float* bwv = ubv + H;       // [H]  b1 + W s_p
  __half* w2h = reinterpret_cast<__half*>(bwv + H);  // [H] output weights in half precision
  float* P = bwv + H + H / 2;  // [kAB][ld]   current chunk (halves on the bf16 path)
  float* Q = P + kAB * (hc + kPad);  // [Kp][ld]
  float* red = Q + Kp * (hc + kPad);  // [kThreads][kTA * kTB] partial sums
  Act* raw = reinterpret_cast<Act*>(red + kThreads * kTA * kTB);  // [rows][hc] next chunk, as stored
  const Tile t = make_tile<kThreads, kAB>(Kp);

  const size_t row_p = (static_cast<size_t>(n) * B + p) * K;      // candidate rows of slot p
  const size_t row_q = (static_cast<size_t>(n) * B + p + 1) * K;  // candidate rows of slot p+1
  const float* vals_p = a.vals + row_p;
  const float* vals_q = a.vals + row_q;
  const float* wsp = a.wsp + static_cast<size_t>(np) * H;
  const int cpr = hc * static_cast<int>(sizeof(Act)) / 16;  // 16-byte pieces per row and chunk
  grid_dep_wait();  // uz, vz, W s and the logits come from preceding kernels
  grid_dep_launch();

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
    // Rows past na (P) or K (Q) are zero.
    for (int i = threadIdx.x; i < (rows << hc_shift) / 8; i += kThreads) {
      const int r = (i * 8) >> hc_shift, c = (i * 8) & (hc - 1), h = h0 + c;
      float x[8];
      const bool is_p = r < kAB;
      const int rr = is_p ? r : r - kAB;
      if (is_p ? r < na : rr < K) {
        ld8_smem<kBf16>(raw + r * hc + c, x);
        if (is_p) {
          const float l = vals_p[a0 + r];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.5f * (x[e] + bwv[h + e] + uav[h + e] * l);
        } else {
          const float l = vals_q[rr];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.5f * (x[e] + ubv[h + e] * l);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
      if constexpr (kBf16) {
        // half precision, clamped to +-30000 so that a sum of two never overflows
        __half* dst = reinterpret_cast<__half*>(is_p ? P : Q) + rr * ld + c;
        uint32_t hw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hh = __floats2half2_rn(fminf(fmaxf(x[2 * e], -30000.f), 30000.f),
                                               fminf(fmaxf(x[2 * e + 1], -30000.f), 30000.f));
          hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      } else {
        float* dst = (is_p ? P : Q) + rr * ld + c;
        *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
      }
    }
    __syncthreads();  // P/Q ready; the raw buffer is free for the next chunk
    if (h0 + hc < H) fetch(h0 + hc);
    accumulate<kBf16>(acc, P, Q, ld, kBf16 ? static_cast<const void*>(w2h + h0) : static_cast<const void*>(w2v + h0),
                      hc, t);
  }
  finish<kThreads>(acc, red, t, a.S + (static_cast<size_t>(np) * K + a0) * K, vals_q, ldv<kBf16>(a.b2, 0), na, K);
}

// ------------------------------------------------------------------ from prepared operands
// P and Q rows come ready-made from the epilogue of the U z / V z projection (f16 for bf16
// weights, f32 otherwise; P rows are indexed like uz, Q rows like vz), so a block only copies
// them into shared memory: all H hidden units at once when they fit in kPrepBudget bytes, else
// chunks of 64 or 128.  Blocks of 128 threads keep ~7 blocks resident per SM, so the whole grid
// of a typical batch runs in one wave; the partial sums reuse the operand buffers at the end.
constexpr int kPrepThreads = 128;
constexpr int kPrepBudget = 96 * 1024;

template <bool kBf16>
__host__ __device__ __forceinline__ int prep_chunk(int H, int K) {
  const int esz = kBf16 ? 2 : 4;
  const int Kp = (K + kTB - 1) / kTB * kTB;
  return (kABP + Kp) * (H * esz + 16) <= kPrepBudget ? H : score_chunk(H);
}

template <bool kBf16>
__global__ void __launch_bounds__(kPrepThreads, 8) score_prepped_kernel(const ScoreArgs a) {
  using Op = typename std::conditional<kBf16, __half, float>::type;
  constexpr int esz = sizeof(Op);
  extern __shared__ __align__(16) float sm[];
  const int K = a.K, H = a.H, B = a.B;
  const int np = blockIdx.x;  // n * (B-1) + p
  const int n = np / (B - 1), p = np % (B - 1);
  const int a0 = blockIdx.y * kABP;
  const int na = min(kABP, K - a0);
  const int Kp = (K + kTB - 1) / kTB * kTB;
  const int hc = prep_chunk<kBf16>(H, K);
  const int ld = hc + 16 / esz;  // row pitch (elements): rows start on 16-byte boundaries
  const int rows = kABP + Kp;
  Op* wv = reinterpret_cast<Op*>(sm);  // [H] output weights
  Op* P = wv + H;                      // [kABP][ld]
  Op* Q = P + kABP * ld;                // [Kp][ld]
  // partial sums [kPrepThreads][kTA * kTB], over P/Q once every thread is done with them
  float* red = reinterpret_cast<float*>(P);
  const Tile t = make_tile<kPrepThreads, kABP>(Kp);

  const size_t row_p = (static_cast<size_t>(n) * B + p) * K + a0;  // first predecessor row
  const size_t row_q = (static_cast<size_t>(n) * B + p + 1) * K;   // first successor row
  const int ppr = hc * esz / 16;  // 16-byte pieces per row and chunk
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Rows past na (P) or K (Q) are zero-filled.
  auto fetch = [&](int h0) {
    for (int r = warp; r < rows; r += kPrepThreads / 32) {
      const bool is_p = r < kABP;
      const int rr = is_p ? r : r - kABP;
      const bool live = is_p ? rr < na : rr < K;
      const Op* src = static_cast<const Op*>(is_p ? a.uz : a.vz) +
                      (live ? (is_p ? row_p : row_q) + rr : 0) * static_cast<size_t>(H) + h0;
      const uint32_t dst = smem_u32((is_p ? P : Q) + rr * ld);
      for (int c = lane; c < ppr; c += 32)
        cp_async16(dst + c * 16, reinterpret_cast<const char*>(src) + c * 16, live ? 16u : 0u);
    }
    cp_async_commit();
  };
  for (int i = threadIdx.x; i < H; i += kPrepThreads) {
    if constexpr (kBf16)
      wv[i] = __float2half_rn(ldv<true>(a.w2, i));
    else
      wv[i] = ldv<false>(a.w2, i);
  }
  grid_dep_wait();  // P and Q come from the preceding kernel
  fetch(0);

  float acc[kTA][kTB];
#pragma unroll
  for (int i = 0; i < kTA; ++i)
#pragma unroll
    for (int j = 0; j < kTB; ++j) acc[i][j] = 0.f;

  for (int h0 = 0; h0 < H; h0 += hc) {
    if (h0 > 0) {
      __syncthreads();  // every thread is done with the previous chunk
      fetch(h0);
    }
    cp_async_wait(0);
    __syncthreads();
    accumulate<kBf16>(acc, P, Q, ld, wv + h0, hc, t);
  }
  grid_dep_launch();
  __syncthreads();  // P/Q are free for the partial sums
  finish<kPrepThreads>(acc, red, t, a.S + (static_cast<size_t>(np) * K + a0) * K, a.vals + row_q,
                       ldv<kBf16>(a.b2, 0), na, K);
}

}  // namespace

size_t score_smem_bytes(int H, int K, bool is_bf16) {
  const int hc = score_chunk(H);
  const int ld = hc + kPad;
  const int Kp = (K + kTB - 1) / kTB * kTB;
  // vectors (four f32, one f16), P and Q, partial sums, and one chunk of raw rows
  return (4 * static_cast<size_t>(H) + H / 2 + static_cast<size_t>(kAB + Kp) * ld + kThreads * kTA * kTB) * sizeof(float) +
         static_cast<size_t>(kAB + Kp) * hc * (is_bf16 ? 2 : 4);
}

size_t score_prepped_smem_bytes(int H, int K, bool is_bf16) {
  const size_t esz = is_bf16 ? 2 : 4;
  const int hc = is_bf16 ? prep_chunk<true>(H, K) : prep_chunk<false>(H, K);
  const int Kp = (K + kTB - 1) / kTB * kTB;
  // the partial sums reuse the P/Q buffers; the chunk of a small H may leave them shorter
  return static_cast<size_t>(H) * esz +
         std::max(static_cast<size_t>(kABP + Kp) * (hc * esz + 16),
                  static_cast<size_t>(kPrepThreads) * kTA * kTB * sizeof(float));
}

namespace {
// The dynamic shared memory ceiling of both kernels is raised once per device to the most they
// can need, so later calls enqueue only the launch (CUDA-graph friendly).
cudaError_t configure_once() {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev]) return cudaSuccess;
  const void* fns[] = {reinterpret_cast<const void*>(score_kernel<true>), reinterpret_cast<const void*>(score_kernel<false>),
                       reinterpret_cast<const void*>(score_prepped_kernel<true>),
                       reinterpret_cast<const void*>(score_prepped_kernel<false>)};
  for (const void* f : fns) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, f);
    if (e != cudaSuccess) return e;
    // the dynamic ceiling plus the kernel's static shared memory stays within 227 KB
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024 - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
  }
  configured[dev] = true;
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_scores(const ScoreArgs& a, bool is_bf16, cudaStream_t stream) {
  const size_t smem = score_smem_bytes(a.H, a.K, is_bf16);
  if (smem > 226 * 1024) return cudaErrorInvalidValue;
  const dim3 grid(a.N * (a.B - 1), (a.K + kAB - 1) / kAB);
  cudaError_t e = configure_once();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return is_bf16 ? cudaLaunchKernelEx(&cfg, score_kernel<true>, a) : cudaLaunchKernelEx(&cfg, score_kernel<false>, a);
}

cudaError_t launch_scores_prepped(const ScoreArgs& a, bool is_bf16, cudaStream_t stream) {
  const size_t smem = score_prepped_smem_bytes(a.H, a.K, is_bf16);
  if (smem > 226 * 1024) return cudaErrorInvalidValue;
  const dim3 grid(a.N * (a.B - 1), (a.K + kABP - 1) / kABP);
  cudaError_t e = configure_once();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPrepThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return is_bf16 ? cudaLaunchKernelEx(&cfg, score_prepped_kernel<true>, a)
                 : cudaLaunchKernelEx(&cfg, score_prepped_kernel<false>, a);
}

}  // namespace dcoco
