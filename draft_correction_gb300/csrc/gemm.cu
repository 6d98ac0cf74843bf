// Dense projections of the corrector on the 5th-generation tensor cores.
//
// jaehun.me review of arXiv 2610.12570, §3.2: every projection and MLP parameter of the
// corrector is shared across slots and transitions, so each projection is one GEMM over
// all streams' rows: C[m, n] = sum_k A[m, k] B[n, k] with B a weight stored out x in.
//
// Kernel shape (one 128-row x BN-column output tile per CTA, 10 warps):
//   warp 0     TMA producer.  B tiles come from a 2-D tensor map, and so do A tiles of
//              activations.  For the candidate embeddings the epilogue warps gather the A
//              rows Emb[c] themselves while the main loop runs (32-byte register loads, stored
//              into the swizzled operand layout) -- the embedding table is never copied to a
//              dense matrix.
//   warp 1     allocates tensor memory; lane 0 issues tcgen05.mma (bf16 -> kind::f16,
//              f32 -> kind::tf32) into an fp32 accumulator of 128 lanes x BN columns and
//              commits each stage back to the producer.
//   warps 2-9  epilogue: tcgen05.ld of the accumulator, then the fused op of the group
//              (LayerNorm over the full row, SiLU with a per-slot bias, the scorer operands,
//              or a plain store).  Two warps share each 32-lane quarter of the accumulator
//              and split its columns; LayerNorm exchanges row partial sums in shared memory.
// Split-K: with split_k > 1 the CTAs of one tile form a cluster along z and each reduces a
// K range.  Each CTA owns a slice of the tile's rows: every CTA writes its partial rows into
// the owner's shared memory (distributed shared memory stores), and the owner adds them in
// rank order -- deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int BM = 128;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each with half of the tile's columns
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kGatherThreads = kEpiThreads;  // epilogue warps that gather the A operand
constexpr int kGatherDepth = 4;              // k-blocks of gathered rows in flight per thread
constexpr int kBiasStageBytes = 20 * 1024;  // per-slot bias rows of one tile (SiLU epilogue)
constexpr int SPLIT_RP = BM + 1;            // split-K buffer: float4 slots per column group

__device__ unsigned int g_status_word;

template <bool kBf16>
struct Elt {
  static constexpr int BK = kBf16 ? 64 : 32;  // elements per 128-byte row of a stage
  static constexpr int UK = kBf16 ? 16 : 8;   // K of one MMA instruction (32 bytes)
  static constexpr uint32_t fmt = kBf16 ? 1u : 2u;
};

// SiLU(x) = x sigmoid(x) = h + h tanh(h), h = x/2 (one SFU instruction).
__device__ __forceinline__ float silu(float x) {
  const float h = 0.5f * x;
  return fmaf(h, tanh_approx(h), h);
}

// One thread's row of a 128-byte-wide output sub-tile into the 128-byte swizzled staging
// layout a tensor-map store expects (16-byte chunk c of row r at r*128 + (c ^ (r & 7))*16).
// kOut: 0 f32, 1 bf16, 2 f16.
template <int kOut>
__device__ __forceinline__ void stage_row(uint8_t* buf, int r, const float* v) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 w;
    if constexpr (kOut == 1) {
      __nv_bfloat162 t0 = __floats2bfloat162_rn(v[8 * c + 0], v[8 * c + 1]);
      __nv_bfloat162 t1 = __floats2bfloat162_rn(v[8 * c + 2], v[8 * c + 3]);
      __nv_bfloat162 t2 = __floats2bfloat162_rn(v[8 * c + 4], v[8 * c + 5]);
      __nv_bfloat162 t3 = __floats2bfloat162_rn(v[8 * c + 6], v[8 * c + 7]);
      w = make_uint4(*reinterpret_cast<uint32_t*>(&t0), *reinterpret_cast<uint32_t*>(&t1),
                     *reinterpret_cast<uint32_t*>(&t2), *reinterpret_cast<uint32_t*>(&t3));
    } else if constexpr (kOut == 2) {
      // half precision clamped to +-30000 (so that a sum of two stays finite)
      const __half2 lim = __float2half2_rn(30000.f), nlim = __float2half2_rn(-30000.f);
      __half2 t0 = __hmax2(__hmin2(__floats2half2_rn(v[8 * c + 0], v[8 * c + 1]), lim), nlim);
      __half2 t1 = __hmax2(__hmin2(__floats2half2_rn(v[8 * c + 2], v[8 * c + 3]), lim), nlim);
      __half2 t2 = __hmax2(__hmin2(__floats2half2_rn(v[8 * c + 4], v[8 * c + 5]), lim), nlim);
      __half2 t3 = __hmax2(__hmin2(__floats2half2_rn(v[8 * c + 6], v[8 * c + 7]), lim), nlim);
      w = make_uint4(*reinterpret_cast<uint32_t*>(&t0), *reinterpret_cast<uint32_t*>(&t1),
                     *reinterpret_cast<uint32_t*>(&t2), *reinterpret_cast<uint32_t*>(&t3));
    } else {
      w = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                     __float_as_uint(v[4 * c + 3]));
    }
    *reinterpret_cast<uint4*>(buf + r * 128 + ((c ^ (r & 7)) << 4)) = w;
  }
}

// Eight values as bf16, round to nearest even.
__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 t1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 t2 = __floats2bfloat162_rn(v[4], v[5]);
  __nv_bfloat162 t3 = __floats2bfloat162_rn(v[6], v[7]);
  return make_uint4(*reinterpret_cast<uint32_t*>(&t0), *reinterpret_cast<uint32_t*>(&t1),
                    *reinterpret_cast<uint32_t*>(&t2), *reinterpret_cast<uint32_t*>(&t3));
}

// Four consecutive entries of a weight-dtype vector as float.
template <bool kBf16>
__device__ __forceinline__ float4 ldw4(const void* p, int i) {
  if constexpr (kBf16) {
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + i);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
  } else {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
  }
}

template <bool kBf16>
__device__ __forceinline__ void store_act1(void* out, size_t idx, float v) {
  if constexpr (kBf16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<float*>(out)[idx] = v;
  }
}

// 32 bytes (two 16-byte halves) from a 32-byte aligned address of data no kernel writes while
// this one runs, not kept in L1; not volatile, so the compiler may schedule the loads freely.
__device__ __forceinline__ void ld_nc32(const void* p, uint4& a, uint4& b) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p));
}
__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <bool kBf16, int BN, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs args, int stages,
                                                          int split_k, int bias_stage_offset) {
  using T = Elt<kBf16>;
  constexpr int A_BYTES = BM * 128;
  constexpr int B_BYTES = BN * 128;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int NH = BN > 256 ? 2 : 1;         // MMA instructions per K step (N <= 256 each)
  constexpr int NMMA = BN / NH;
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  constexpr uint32_t IDESC = mma_idesc(T::fmt, BM, NMMA);

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int s_rows[BM];
  __shared__ float s_ln[2][BM];  // LayerNorm partial row sums of the two column halves

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x;
  int gi = 0, nt = blockIdx.y;
  while (gi + 1 < args.n_groups && nt >= args.g[gi].n_tiles) {
    nt -= args.g[gi].n_tiles;
    ++gi;
  }
  const GemmGroup& grp = args.g[gi];
  // The group's scalars in registers: gi is not a compile-time index, so every read through
  // grp is a generic load from parameter memory, which stores through other pointers force the
  // compiler to repeat (one memory round trip each).
  const int g_epi = grp.epi;
  void* const g_out = grp.out;
  const int g_ldo = grp.ldo;
  const void* const g_col_u = grp.col_u;
  const void* const g_col_b = grp.col_b;
  const float* const g_row_bias = grp.row_bias;
  const int ks = blockIdx.z;
  const int nkb_total = (args.K + T::BK - 1) / T::BK;
  const int per = (nkb_total + split_k - 1) / split_k;
  const int kb0 = ks * per;
  const int nk = std::max(0, std::min(nkb_total, kb0 + per) - kb0);

  const bool gather = args.gather != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      // gathered A: the B tile's transaction count plus one arrival per gathering thread
      mbar_init(smem_u32(&full_bar[s]), gather ? 1 + kGatherThreads : 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    fence_mbar_init();
    prefetch_tmap(&args.a_map);
    prefetch_tmap(&grp.b_map);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), TMEM_COLS);
  tc_fence_before();
  __syncthreads();  // barriers initialised, accumulator allocated
  tc_fence_after();
  // The weight (B) tiles of the first stages do not depend on the preceding kernel: request them
  // before waiting for it.
  const int pre = std::min(nk, stages);
  if (threadIdx.x == 0) {
    for (int i = 0; i < pre; ++i) {
      const uint32_t fb = smem_u32(&full_bar[i]);
      const uint32_t b_s = smem_u32(smem) + i * STAGE_BYTES + A_BYTES;
      const int kx = (kb0 + i) * T::BK;
      mbar_expect_tx(fb, gather ? B_BYTES : STAGE_BYTES);
#pragma unroll
      for (int h = 0; h < NH; ++h) tma_load_2d(b_s + h * NMMA * 128, &grp.b_map, kx, nt * BN + h * NMMA, fb);
    }
  }
  if (args.early_dependents) grid_dep_launch();
  grid_dep_wait();
  if (args.gather != nullptr && threadIdx.x < BM) {
    const int m = m_tile * BM + threadIdx.x;
    int row = 0;
    if (m < args.M) {
      row = args.gather[m];
      if (row < 0 || row >= args.gather_limit) {
        atomicOr(args.status, DEV_BAD_INDEX);
        row = 0;
      }
    }
    s_rows[threadIdx.x] = row;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t smem0 = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    for (int i = 0; i < nk; ++i) {
      const int s = i % stages;
      const uint32_t ph = (i / stages) & 1;
      const uint32_t fb = smem_u32(&full_bar[s]);
      const uint32_t a_s = smem0 + s * STAGE_BYTES;
      const uint32_t b_s = a_s + A_BYTES;
      const int kx = (kb0 + i) * T::BK;
      if (i >= pre) {  // the first `pre` stages are fresh and already expect their bytes
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1))) {
          if (lane == 0) atomicOr(args.status, DEV_TIMEOUT_MMA);
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(fb, gather ? B_BYTES : STAGE_BYTES);
#pragma unroll
          for (int h = 0; h < NH; ++h) tma_load_2d(b_s + h * NMMA * 128, &grp.b_map, kx, nt * BN + h * NMMA, fb);
        }
      }
      if (!gather && lane == 0) tma_load_2d(a_s, &args.a_map, kx, m_tile * BM, fb);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = (i / stages) & 1;
        if (!mbar_wait(smem_u32(&full_bar[s]), ph)) {
          atomicOr(args.status, DEV_TIMEOUT_TMA);
          break;
        }
        tc_fence_after();
        const uint32_t a_s = smem0 + s * STAGE_BYTES;
        const uint32_t b_s = a_s + A_BYTES;
#pragma unroll
        for (int j = 0; j < T::BK / T::UK; ++j) {
          const uint64_t ad = sw128_desc(a_s + j * 32);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const uint64_t bd = sw128_desc(b_s + h * NMMA * 128 + j * 32);
            tc_mma<!kBf16>(tmem + h * NMMA, ad, bd, IDESC, (i > 0 || j > 0) ? 1u : 0u);
          }
        }
        tc_commit(smem_u32(&empty_bar[s]));
      }
      tc_commit(smem_u32(&acc_bar));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    if (gather) {
      // Gathered A operand: while the main loop runs these 256 threads copy Emb[c] rows into the
      // stages through registers.  Thread t owns the 32-byte piece t % 4 of tile rows t / 4 and
      // 64 + t / 4 in every k-block (the 8 threads of a row pair cover 2 x 128 bytes, coalesced),
      // loads kGatherDepth k-blocks ahead with 32-byte non-caching loads, and stores each k-block
      // into the 128-byte swizzled operand layout once its stage is free; a generic-to-async
      // proxy fence and one arrival per thread hand the stage to the tensor core.  (Measured on
      // this GPU with clean L2 lines: this access pattern alone reads 8192 random 8 KB rows at
      // 3.4 to 4 TB/s, whole rows per warp at about 4.2 TB/s; TMA bulk copies of 128 or 512
      // bytes per row are issue-bound near 0.6 and 2 TB/s.)
      const int t = threadIdx.x - 64;
      const int pc = t & 3;                    // 32-byte piece of the 128-byte row
      const int rA = t >> 2, rB = 64 + (t >> 2);
      constexpr int esz = kBf16 ? 2 : 4;
      constexpr int EPP = 32 / esz;            // elements per piece
      const char* base = static_cast<const char*>(args.gather_base);
      const char* pA = base + static_cast<size_t>(s_rows[rA]) * args.gather_pitch_bytes + kb0 * 128 + pc * 32;
      const char* pB = base + static_cast<size_t>(s_rows[rB]) * args.gather_pitch_bytes + kb0 * 128 + pc * 32;
      const int kel0 = kb0 * T::BK + pc * EPP;  // first element of this thread's piece in k-block 0
      // 32-byte loads need 32-byte aligned rows; the ABI promises 16 (then two 16-byte loads)
      const bool wide = ((reinterpret_cast<uintptr_t>(base) | static_cast<uintptr_t>(args.gather_pitch_bytes)) & 31) == 0;
      uint4 ra[kGatherDepth][2], rb[kGatherDepth][2];
      // The piece of k-block i, 16 bytes at a time: a row ends on a 16-byte boundary, so each half
      // lies wholly inside the row or wholly past its end (zero).
      auto fetch = [&](int i, uint4(&a)[2], uint4(&b)[2]) {
        const int kcol = kel0 + i * T::BK;
        const size_t off = static_cast<size_t>(i) * 128;
        const bool lo = i < nk && kcol < args.K;
        const bool hi = i < nk && kcol + EPP / 2 < args.K;
        if (wide && hi) {
          ld_nc32(pA + off, a[0], a[1]);
          ld_nc32(pB + off, b[0], b[1]);
        } else {
          const uint4 z = make_uint4(0, 0, 0, 0);
          a[0] = lo ? ld_nc16(pA + off) : z;
          b[0] = lo ? ld_nc16(pB + off) : z;
          a[1] = hi ? ld_nc16(pA + off + 16) : z;
          b[1] = hi ? ld_nc16(pB + off + 16) : z;
        }
      };
      // swizzled positions of the piece's two 16-byte chunks in rows rA and rB (rA & 7 == rB & 7)
      const int sw = rA & 7;
      const uint32_t offA0 = rA * 128 + (((2 * pc) ^ sw) << 4), offA1 = rA * 128 + (((2 * pc + 1) ^ sw) << 4);
      const uint32_t offB0 = offA0 + 64 * 128, offB1 = offA1 + 64 * 128;
#pragma unroll
      for (int d = 0; d < kGatherDepth; ++d) fetch(d, ra[d], rb[d]);
      bool alive = true;
      for (int i0 = 0; i0 < nk && alive; i0 += kGatherDepth) {
#pragma unroll
        for (int d = 0; d < kGatherDepth; ++d) {
          const int i = i0 + d;
          if (i >= nk || !alive) break;  // warp-uniform
          const int s = i % stages;
          const uint32_t ph = (i / stages) & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1))) {
            if (lane == 0) atomicOr(args.status, DEV_TIMEOUT_MMA);
            alive = false;
            break;
          }
          uint8_t* a_s = smem + s * STAGE_BYTES;
          *reinterpret_cast<uint4*>(a_s + offA0) = ra[d][0];
          *reinterpret_cast<uint4*>(a_s + offA1) = ra[d][1];
          *reinterpret_cast<uint4*>(a_s + offB0) = rb[d][0];
          *reinterpret_cast<uint4*>(a_s + offB1) = rb[d][1];
          fence_proxy_async();
          mbar_arrive(smem_u32(&full_bar[s]));
          fetch(i + kGatherDepth, ra[d], rb[d]);
        }
      }
    }
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the tile's columns (when split)
    const int row_local = q * 32 + lane;
    const int m = m_tile * BM + row_local;
    // tcgen05.ld is warp-collective: every lane of the warp takes the same path below and
    // only the stores are predicated on the row being inside M.
    // While the main loop runs, stage this tile's per-slot bias rows in shared memory.
    const float* sbias = nullptr;
    int first_slot = 0, prep_nslots = 0;
    if (g_epi == EPI_SILU_BIAS) {
      first_slot = (m_tile * BM) / args.bias_div;
      const int last_slot = (min(args.M, m_tile * BM + BM) - 1) / args.bias_div;
      const int nslots = last_slot - first_slot + 1;
      if (nslots * BN * 4 <= kBiasStageBytes) {
        float* dst = reinterpret_cast<float*>(smem + bias_stage_offset);
        for (int i = threadIdx.x - 64; i < nslots * (BN / 4); i += kEpiThreads) {
          const int sl = i / (BN / 4), c4 = i % (BN / 4);
          *reinterpret_cast<float4*>(dst + sl * BN + c4 * 4) = *reinterpret_cast<const float4*>(
              args.bias + static_cast<size_t>(first_slot + sl) * args.ld_bias + nt * BN + c4 * 4);
        }
        sbias = dst;
      }
      named_barrier_sync(1, kEpiThreads);
    } else if (g_epi == EPI_PREP) {
      // Rows 0..nslots-1: (col_b + the slot's pair-bias row) / 2; row nslots: col_u / 2.
      first_slot = (m_tile * BM) / args.bias_div;
      const int last_slot = (min(args.M, m_tile * BM + BM) - 1) / args.bias_div;
      const int nslots = last_slot - first_slot + 1;
      if ((nslots + 1) * BN * 4 <= kBiasStageBytes) {
        float* dst = reinterpret_cast<float*>(smem + bias_stage_offset);
        for (int i = threadIdx.x - 64; i < (nslots + 1) * (BN / 4); i += kEpiThreads) {
          const int sl = i / (BN / 4), c4 = i % (BN / 4);
          const int col = nt * BN + c4 * 4;
          float4 v;
          if (sl == nslots) {
            v = ldw4<kBf16>(g_col_u, col);
          } else {
            v = g_col_b != nullptr ? ldw4<kBf16>(g_col_b, col) : make_float4(0.f, 0.f, 0.f, 0.f);
            const int qs = first_slot + sl, stream_i = qs / args.slots;
            if (g_row_bias != nullptr && qs - stream_i * args.slots < args.slots - 1) {
              const float4 rb = *reinterpret_cast<const float4*>(
                  g_row_bias + static_cast<size_t>(qs - stream_i) * args.ld_bias + col);
              v.x += rb.x;
              v.y += rb.y;
              v.z += rb.z;
              v.w += rb.w;
            }
          }
          *reinterpret_cast<float4*>(dst + sl * BN + c4 * 4) = make_float4(0.5f * v.x, 0.5f * v.y, 0.5f * v.z, 0.5f * v.w);
        }
        sbias = dst;
        prep_nslots = nslots;
      }
      named_barrier_sync(1, kEpiThreads);
    }
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&acc_bar), 0));
    if (!ok && lane == 0) atomicOr(args.status, DEV_TIMEOUT_ACC);
    grid_dep_launch();  // main loop done: the next kernel may start its prologue
    const bool live = m < args.M;
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    if constexpr (kSplit) {
      // Every CTA of the cluster is past its main loop, so its pipeline buffers are free, before
      // any partial row is written into them.  Row rr of the slice owned by rank o receives this
      // CTA's partial at slot row (rank * rpc + rr) of o's buffer: stores only, no round trips.
      // The buffer is column-group major (four columns of every slot row, then the next four),
      // so the 32 lanes of a warp (32 consecutive rows) store 512 contiguous bytes.
      cluster_arrive();
      cluster_wait();
      const int rank = static_cast<int>(cluster_rank());  // the cluster spans grid.z
      const int rpc = BM / split_k;
      const int owner = row_local / rpc;
      const uint32_t dst = map_to_rank(smem_u32(smem), static_cast<uint32_t>(owner)) +
                           static_cast<uint32_t>(rank * rpc + row_local - owner * rpc) * 16u;
      constexpr int SH = BN >= 64 ? 2 : 1;  // warps per quarter sharing the columns
      constexpr int CW = BN / SH;           // columns per warp
      if (half < SH) {
#pragma unroll 1
        for (int c = half * CW; c < (half + 1) * CW; c += 64) {
          uint32_t v[2][32];
          const int n2 = c + 32 < (half + 1) * CW ? 2 : 1;  // two 32-column loads in flight
          tmem_ld32_nowait(trow + c, v[0]);
          if (n2 == 2) tmem_ld32_nowait(trow + c + 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= n2) break;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              st_cluster_f32x4(dst + static_cast<uint32_t>((c + 32 * u + i) >> 2) * (SPLIT_RP * 16u),
                               __uint_as_float(v[u][i]), __uint_as_float(v[u][i + 1]), __uint_as_float(v[u][i + 2]),
                               __uint_as_float(v[u][i + 3]));
          }
        }
      }
    } else {
      // Row-per-thread values go through a swizzled staging buffer per warp (two 32 x 128-byte
      // halves, reusing the drained pipeline buffers) and leave with tensor-map stores, which
      // write whole rows coalesced and clip rows past M.  Every epilogue warp runs this block,
      // even after a timed-out wait (then nothing is stored), so the named barriers always
      // see all of them.
      const bool out_bf16 = kBf16 && g_epi != EPI_F32;
      const int cps = out_bf16 ? 64 : 32;  // output columns per 128-byte sub-tile
      const int nsub = BN / cps;           // 128-byte sub-tiles in the tile's columns
      const int halves = nsub >= 2 ? 2 : 1;
      const int j0 = half * nsub / halves, j1 = (half + 1) * nsub / halves;  // this warp's sub-tiles
      uint8_t* stg = smem + (warp - 2) * 8192;
      const int y0 = m_tile * BM + q * 32;
      const bool any_rows = y0 < args.M;
      float mean = 0.f, rstd = 1.f;
      if (g_epi == EPI_LN) {
        // Two-pass row statistics over the full row: each warp sums its columns, the two
        // warps of a quarter exchange their partial sums.
        const int c0 = half < halves ? j0 * cps : 0, c1 = half < halves ? j1 * cps : 0;
        float sum = 0.f;
        for (int c = c0; c < c1; c += 32) {
          float v[32];
          tmem_ld32(trow + c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) sum += v[i];
        }
        if (halves == 2) {
          s_ln[half][row_local] = sum;
          named_barrier_sync(2, kEpiThreads);
          sum = s_ln[0][row_local] + s_ln[1][row_local];
        }
        mean = sum / BN;
        float ss = 0.f;
        for (int c = c0; c < c1; c += 32) {
          float v[32];
          tmem_ld32(trow + c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) ss += (v[i] - mean) * (v[i] - mean);
        }
        if (halves == 2) {
          named_barrier_sync(2, kEpiThreads);  // everyone has read the first exchange
          s_ln[half][row_local] = ss;
          named_barrier_sync(2, kEpiThreads);
          ss = s_ln[0][row_local] + s_ln[1][row_local];
        }
        rstd = rsqrtf(ss / BN + args.ln_eps);
      }
      const float* bias = nullptr;
      if (g_epi == EPI_SILU_BIAS && live) {
        bias = sbias != nullptr ? sbias + (m / args.bias_div - first_slot) * BN
                                : args.bias + static_cast<size_t>(m / args.bias_div) * args.ld_bias + nt * BN;
      }
      // EPI_PREP: this row's scale and pair-bias row
      float row_l = 0.f;
      const float* rbias = nullptr;
      if (g_epi == EPI_PREP && live) {
        row_l = args.row_l[m];
        const int q_slot = m / args.bias_div;  // stream * slots + slot
        const int stream_i = q_slot / args.slots, slot = q_slot - stream_i * args.slots;
        if (g_row_bias != nullptr && slot < args.slots - 1)
          rbias = g_row_bias + static_cast<size_t>(q_slot - stream_i) * args.ld_bias + nt * BN;
      }
      // The fused op on 32 consecutive columns starting at `col` (compile-time trip counts).
      auto apply32 = [&](float(&x)[32], int col) {
        if (g_epi == EPI_LN) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = (x[i] - mean) * rstd;
        } else if (bias != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 bb = *reinterpret_cast<const float4*>(bias + col + i);
            x[i] = silu(x[i] + bb.x);
            x[i + 1] = silu(x[i + 1] + bb.y);
            x[i + 2] = silu(x[i + 2] + bb.z);
            x[i + 3] = silu(x[i + 3] + bb.w);
          }
        } else if (g_epi == EPI_PREP && sbias != nullptr) {
          const float* add = sbias + (m / args.bias_div - first_slot) * BN + col;
          const float* uu = sbias + prep_nslots * BN + col;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 a4 = live ? *reinterpret_cast<const float4*>(add + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 u4 = *reinterpret_cast<const float4*>(uu + i);
            x[i] = fmaf(0.5f, x[i], fmaf(u4.x, row_l, a4.x));
            x[i + 1] = fmaf(0.5f, x[i + 1], fmaf(u4.y, row_l, a4.y));
            x[i + 2] = fmaf(0.5f, x[i + 2], fmaf(u4.z, row_l, a4.z));
            x[i + 3] = fmaf(0.5f, x[i + 3], fmaf(u4.w, row_l, a4.w));
          }
        } else if (g_epi == EPI_PREP) {
          const int c0 = nt * BN + col;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 uu = ldw4<kBf16>(g_col_u, c0 + i);
            float4 add = g_col_b != nullptr ? ldw4<kBf16>(g_col_b, c0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (rbias != nullptr) {
              const float4 rb = *reinterpret_cast<const float4*>(rbias + col + i);
              add.x += rb.x;
              add.y += rb.y;
              add.z += rb.z;
              add.w += rb.w;
            }
            x[i] = 0.5f * (x[i] + add.x + uu.x * row_l);
            x[i + 1] = 0.5f * (x[i + 1] + add.y + uu.y * row_l);
            x[i + 2] = 0.5f * (x[i + 2] + add.z + uu.z * row_l);
            x[i + 3] = 0.5f * (x[i + 3] + add.w + uu.w * row_l);
          }
        }
      };
      for (int j = j0; half < halves && j < j1; ++j) {
        float v[64];
        float(&lo)[32] = *reinterpret_cast<float(*)[32]>(v);
        float(&hi)[32] = *reinterpret_cast<float(*)[32]>(v + 32);
        tmem_ld32(trow + j * cps, lo);
        apply32(lo, j * cps);
        if (out_bf16) {
          tmem_ld32(trow + j * cps + 32, hi);
          apply32(hi, j * cps + 32);
        }
        uint8_t* buf = stg + ((j - j0) & 1) * 4096;
        if (j - j0 >= 2) {
          if (lane == 0) bulk_wait_read<1>();  // the store that used this half has read it
          __syncwarp();
        }
        if (g_epi == EPI_PREP && kBf16)
          stage_row<2>(buf, lane, v);
        else if (out_bf16)
          stage_row<1>(buf, lane, v);
        else
          stage_row<0>(buf, lane, v);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0 && any_rows && ok) {
          tma_store_2d(&grp.out_map, nt * BN + j * cps, y0, smem_u32(buf));
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait<0>();
    }
  }

  if constexpr (kSplit) {
    // The producer and MMA warps take the first cluster barrier of the epilogue warps here; the
    // second one makes every pushed partial row visible to its owner.
    if (warp < 2) {
      cluster_arrive();
      cluster_wait();
    }
    tc_fence_before();
    cluster_sync();
    const int rank = static_cast<int>(cluster_rank());
    const int rpc = BM / split_k;
    // partial rows, column-group major: column c of slot row sr at ((c / 4) * SPLIT_RP + sr) * 4 + c % 4
    const float* red = reinterpret_cast<const float*>(smem);
    if (g_epi == EPI_LN) {
      // LayerNorm rows: four threads per row, each with a quarter of the columns in registers
      // (the partials added in rank order: deterministic).  Lane = quarter * 8 + row within the
      // warp's 8 rows, so a warp's loads cover 8 consecutive slot rows of 4 column groups
      // (conflict-free) and the row sums need two shuffles.  Each thread stores its quarter of
      // the row with 16-byte stores.
      constexpr int CQ = BN / 4;  // columns per thread
      const int t = threadIdx.x;
      const int rr = (t >> 5) * 8 + (t & 7), q = (t >> 3) & 3;
      const bool on = t < rpc * 4;  // rpc is a multiple of 8
      const int m = m_tile * BM + rank * rpc + rr;
      float v[CQ];
#pragma unroll
      for (int i = 0; i < CQ; ++i) v[i] = 0.f;
      if (on) {
        for (int src = 0; src < split_k; ++src) {
#pragma unroll
          for (int k = 0; k < CQ / 4; ++k) {
            const float4 x = *reinterpret_cast<const float4*>(red + ((q * (CQ / 4) + k) * SPLIT_RP + src * rpc + rr) * 4);
            v[4 * k] += x.x;
            v[4 * k + 1] += x.y;
            v[4 * k + 2] += x.z;
            v[4 * k + 3] += x.w;
          }
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < CQ; ++i) sum += v[i];
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 8);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 16);
      const float mean = sum / BN;
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < CQ; ++i) ss += (v[i] - mean) * (v[i] - mean);
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 8);
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 16);
      const float rstd = rsqrtf(ss / BN + args.ln_eps);
      if (on && m < args.M) {
        const size_t obase = static_cast<size_t>(m) * g_ldo + static_cast<size_t>(nt) * BN + q * CQ;
#pragma unroll
        for (int i = 0; i < CQ; ++i) v[i] = (v[i] - mean) * rstd;
        if constexpr (kBf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g_out) + obase);
#pragma unroll
          for (int k = 0; k < CQ / 8; ++k) dst[k] = pack8_bf16(v + 8 * k);
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(g_out) + obase);
#pragma unroll
          for (int k = 0; k < CQ / 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
      }
    } else {
    // Other epilogues: one warp per owned row, two rows at a time so that their loads and
    // reductions overlap; the partials are added in rank order (deterministic).
    constexpr int NW = kThreads / 32;
    constexpr int NJ = (BN + 31) / 32;
    for (int rr0 = warp; rr0 < rpc; rr0 += 2 * NW) {
      float v[2][NJ];
      int mm[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int rr = rr0 + u * NW;
        mm[u] = rr < rpc ? m_tile * BM + rank * rpc + rr : args.M;  // args.M: nothing to write
#pragma unroll
        for (int j = 0; j < NJ; ++j) v[u][j] = 0.f;
        if (rr >= rpc) continue;
        for (int src = 0; src < split_k; ++src) {
          const float* part = red + (src * rpc + rr) * 4;
#pragma unroll
          for (int j = 0; j < NJ; ++j) {
            const int c = lane + 32 * j;  // lanes read 32 different banks (SPLIT_RP * 4 = 4 mod 32)
            if (c < BN) v[u][j] += part[(c >> 2) * (SPLIT_RP * 4) + (c & 3)];
          }
        }
      }
      if (g_epi == EPI_LN) {
        float mean[2], rstd[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < NJ; ++j) sum += v[u][j];
          mean[u] = warp_sum(sum) / BN;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float ss = 0.f;
#pragma unroll
          for (int j = 0; j < NJ; ++j)
            if (lane + 32 * j < BN) ss += (v[u][j] - mean[u]) * (v[u][j] - mean[u]);
          rstd[u] = rsqrtf(warp_sum(ss) / BN + args.ln_eps);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < NJ; ++j)
            if (mm[u] < args.M && lane + 32 * j < BN)
              store_act1<kBf16>(g_out, static_cast<size_t>(mm[u]) * g_ldo + static_cast<size_t>(nt) * BN + lane + 32 * j,
                                (v[u][j] - mean[u]) * rstd[u]);
      } else {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int m = mm[u];
          if (m >= args.M) continue;
          const size_t obase = static_cast<size_t>(m) * g_ldo + static_cast<size_t>(nt) * BN;
          if (g_epi == EPI_F32) {
#pragma unroll
            for (int j = 0; j < NJ; ++j)
              if (lane + 32 * j < BN) static_cast<float*>(g_out)[obase + lane + 32 * j] = v[u][j];
          } else {
            const float* bias = (g_epi == EPI_SILU_BIAS)
                                    ? args.bias + static_cast<size_t>(m / args.bias_div) * args.ld_bias + nt * BN
                                    : nullptr;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              if (lane + 32 * j >= BN) continue;
              float x = v[u][j];
              if (bias != nullptr) x = silu(x + bias[lane + 32 * j]);
              store_act1<kBf16>(g_out, obase + lane + 32 * j, x);
            }
          }
        }
      }
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <bool kBf16, int BN, bool kSplit>
cudaError_t launch_gemm_t(const GemmArgs& args, int split_k, cudaStream_t stream) {
  // The split-K reduction has no scorer-operand epilogue.
  auto any_group = [&](auto pred) {
    for (int i = 0; i < args.n_groups; ++i)
      if (pred(args.g[i].epi)) return true;
    return false;
  };
  if (args.n_groups < 1 || args.n_groups > 3) return cudaErrorInvalidValue;
  if (kSplit && any_group([](int epi) { return epi == EPI_PREP; })) return cudaErrorInvalidValue;
  constexpr int STAGE_BYTES = BM * 128 + BN * 128;
  int stages = std::min(kMaxStages, kSmemBudget / STAGE_BYTES);
  // split-K reuses the pipeline buffers for the partial rows it receives (BN / 4 column groups
  // of SPLIT_RP float4 slots)
  const int split_bytes = kSplit ? (BN / 4) * SPLIT_RP * 16 : 0;
  auto staged = [](int epi) { return epi == EPI_SILU_BIAS || epi == EPI_PREP; };
  const bool has_bias = any_group(staged);
  if (has_bias) stages = std::min(stages, 4);
  const int bias_off = std::max(stages * STAGE_BYTES, split_bytes);
  const int smem = bias_off + (has_bias ? kBiasStageBytes : 0) + 1024;
  auto kern = gemm_kernel<kBf16, BN, kSplit>;
  // Function attributes are set once per instantiation (and device), so that later calls
  // enqueue nothing but the launch and can be captured into a CUDA graph.
  static int configured[64] = {};  // largest dynamic shared memory size set so far, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  int n_tiles = 0;
  for (int i = 0; i < args.n_groups; ++i) n_tiles += args.g[i].n_tiles;
  cfg.gridDim = dim3((args.M + BM - 1) / BM, n_tiles, split_k);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = split_k;
  cfg.attrs = attr;
  cfg.numAttrs = kSplit ? 1 : 0;
  cfg.numAttrs += pdl_attr(&attr[cfg.numAttrs]);
  return cudaLaunchKernelEx(&cfg, kern, args, stages, split_k, bias_off);
}

template <bool kBf16>
cudaError_t dispatch_bn(const GemmArgs& args, int BN, int split_k, cudaStream_t stream) {
  const bool sp = split_k > 1;
  switch (BN) {
    case 32: return sp ? launch_gemm_t<kBf16, 32, true>(args, split_k, stream) : launch_gemm_t<kBf16, 32, false>(args, 1, stream);
    case 64: return sp ? launch_gemm_t<kBf16, 64, true>(args, split_k, stream) : launch_gemm_t<kBf16, 64, false>(args, 1, stream);
    case 128: return sp ? launch_gemm_t<kBf16, 128, true>(args, split_k, stream) : launch_gemm_t<kBf16, 128, false>(args, 1, stream);
    case 256: return sp ? launch_gemm_t<kBf16, 256, true>(args, split_k, stream) : launch_gemm_t<kBf16, 256, false>(args, 1, stream);
    case 512: return sp ? cudaErrorInvalidValue : launch_gemm_t<kBf16, 512, false>(args, 1, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool kBf16>
__global__ void pair_combine_kernel(const float* __restrict__ hp, void* __restrict__ s, int N, int B, int r) {
  grid_dep_wait();  // hp comes from the preceding kernel
  grid_dep_launch();
  const int64_t total = static_cast<int64_t>(N) * (B - 1) * r;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % r);
    const int64_t np = i / r;  // n * (B-1) + p
    const int64_t n = np / (B - 1), p = np % (B - 1);
    const int64_t row = n * B + p;
    const float v = hp[row * 2 * r + c] + hp[(row + 1) * 2 * r + r + c];
    store_act1<kBf16>(s, i, v);
  }
}


// ---------------------------------------------------------------- fused z -> P / Q
// The candidate fusion z = SiLU(W_f [b; g]) and the candidate blocks of the first MLP layer
// (U z, V z, folded into the scorer's operands P and Q) for one 128-row tile, in one kernel:
//   phase 1  acc1 = b W_f[:, 0:r]^T in TMEM (b tile loaded once by TMA, W_f k-blocks through the
//            ring); the epilogue warps write z = SiLU(acc1 + gw[slot]) in bf16 over the b tile,
//            in the 128-byte swizzled operand layout, and hand it to the MMA warp in two column
//            halves, so that the first phase-2 k-blocks start while the second half is written;
//   phase 2  acc2 = z U^T (grid.y even) or z V^T (grid.y odd), one block of at most 256 output
//            columns after the other (or, when the grid is small, one block per CTA), their
//            weight k-blocks through the same ring; the epilogue of a column block (the logit
//            term, for P the bias and W s_p, the halving, f16 rows by tensor-map stores) runs
//            while the MMAs of the next block do.
// TMEM columns: acc1 at [0, r); the first phase-2 block at [256, 256 + NC), clear of acc1 while
// its second column half is still being read; a second block at [0, NC), issued only once all
// of acc1 has been read.
// The ring's four 32 KB stages take every W_f k-block before the kernel waits for its
// predecessors, and the first U or V k-blocks while phase 1 runs.
// z never leaves shared memory.  Warp roles as in gemm_kernel: 0 TMA producer, 1 MMA issuer,
// 2-9 epilogue (two per TMEM lane quarter, each with half of the columns).
constexpr int kZuvRing = 4;
constexpr int kZuvStage = 256 * 128;  // one k-block of up to 256 weight rows
constexpr int kZuvConst = 32 * 1024;  // per-tile constants of the epilogues

// tanh of two values in packed half precision (one SFU instruction for both).
__device__ __forceinline__ float2 tanh2_f16(float a, float b) {
  const __half2 x = __floats2half2_rn(a, b);
  uint32_t t;
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&x)));
  return __half22float2(*reinterpret_cast<const __half2*>(&t));
}

// Eight values in half precision, clamped to +-30000 so that a sum of two stays finite.
__device__ __forceinline__ uint4 pack8_f16_clamped(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2 t = __floats2half2_rn(fminf(fmaxf(v[2 * e], -30000.f), 30000.f),
                                        fminf(fmaxf(v[2 * e + 1], -30000.f), 30000.f));
    w[e] = *reinterpret_cast<const uint32_t*>(&t);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One 32-byte store to a 32-byte aligned global address.
__device__ __forceinline__ void st_global_32(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}


template <int R>
__global__ void __launch_bounds__(kThreads, 1) zuv_kernel(const __grid_constant__ ZuvArgs args) {
  constexpr int NK = R / 64;      // k-blocks of both products (their K is r)
  constexpr int A_KB = BM * 128;  // one k-block of the 128-row operand
  constexpr uint32_t IDESC1 = mma_idesc(1u, BM, R);
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* a_reg = smem;            // NK x 16 KB: the b tile, then z
  uint8_t* ring = smem + NK * A_KB;  // kZuvRing x kZuvStage
  __shared__ __align__(8) uint64_t full_bar[kZuvRing];
  __shared__ __align__(8) uint64_t empty_bar[kZuvRing];
  __shared__ __align__(8) uint64_t a_bar, acc1_bar;
  __shared__ __align__(8) uint64_t z_bar[2];  // the two column halves of z (k-blocks of phase 2)
  __shared__ __align__(8) uint64_t acc2_bar[2];  // one per phase-2 column block
  __shared__ uint32_t tmem_base_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x;
  const bool is_q = (blockIdx.y & 1) != 0;
  const int H = args.H;
  const int NC = H <= 256 ? H : 256;  // columns per phase-2 MMA (and per column block)
  // grid.y = 2: every column block of P (y = 0) or Q (y = 1) in this CTA; grid.y = 2 H / NC
  // (small grids): only column block y >> 1 of P or Q, so that the CTAs' chains are shorter
  const bool one_block = gridDim.y > 2;
  const int cb0 = one_block ? static_cast<int>(blockIdx.y >> 1) : 0;  // first column block
  const int NH2 = one_block ? 1 : H / NC;                                // column blocks here
  const uint32_t idesc2 = mma_idesc(1u, BM, static_cast<uint32_t>(NC));
  const CUtensorMap* w2_map = is_q ? &args.v_map : &args.u_map;
  // ring loads: NK k-blocks of W_f, then NK k-blocks of U or V per column block
  const int total = NK + NH2 * NK;
  // TMEM column of phase-2 column block cb (acc1 holds [0, R))
  auto acc2_col = [](int cb) { return cb == 0 ? 256u : 0u; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kZuvRing; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&a_bar), 1);
    mbar_init(smem_u32(&acc1_bar), 1);
    mbar_init(smem_u32(&z_bar[0]), 1);
    mbar_init(smem_u32(&z_bar[1]), 1);
    mbar_init(smem_u32(&acc2_bar[0]), 1);
    mbar_init(smem_u32(&acc2_bar[1]), 1);
    fence_mbar_init();
    prefetch_tmap(&args.b_map);
    prefetch_tmap(&args.wf_map);
    prefetch_tmap(w2_map);
    prefetch_tmap(is_q ? &args.q_map : &args.p_map);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t ring0 = smem_u32(ring), a0 = smem_u32(a_reg);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto issue = [&](int i) {
        const int s = i % kZuvRing;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t dst = ring0 + s * kZuvStage;
        if (i < NK) {
          mbar_expect_tx(fb, R * 128);
          tma_load_2d(dst, &args.wf_map, i * 64, 0, fb);
        } else {
          const int j = i - NK, cb = j / NK, kb = j - cb * NK;
          mbar_expect_tx(fb, NC * 128);
          tma_load_2d(dst, w2_map, kb * 64, (cb0 + cb) * NC, fb);
        }
      };
      // the weight tiles do not depend on the preceding kernels: request them first
      for (int i = 0; i < kZuvRing && i < total; ++i) issue(i);
      grid_dep_wait();  // the b rows come from the preceding kernel
      const uint32_t ab = smem_u32(&a_bar);
      mbar_expect_tx(ab, NK * A_KB);
      for (int kb = 0; kb < NK; ++kb) tma_load_2d(a0 + kb * A_KB, &args.b_map, kb * 64, m_tile * BM, ab);
      for (int i = kZuvRing; i < total; ++i) {
        const int s = i % kZuvRing;
        if (!mbar_wait(smem_u32(&empty_bar[s]), ((i / kZuvRing) & 1) ^ 1)) {
          atomicOr(args.status, DEV_TIMEOUT_MMA);
          break;
        }
        issue(i);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(smem_u32(&a_bar), 0);
      if (!ok) atomicOr(args.status, DEV_TIMEOUT_TMA);
      for (int i = 0; ok && i < total; ++i) {
        // phase 2 reads z, which the epilogue writes over b once it has read acc1: its first
        // k-blocks as soon as the first column half of z is written, the rest after the second
        if (i == NK) tc_commit(smem_u32(&acc1_bar));
        if (i == NK || i == NK + NK / 2) {
          const int first = i == NK ? 0 : 1, last = (i == NK && NK / 2 > 0) ? 0 : 1;
          for (int zh = first; ok && zh <= last; ++zh) {
            if (!mbar_wait(smem_u32(&z_bar[zh]), 0)) {
              atomicOr(args.status, DEV_TIMEOUT_ACC);
              ok = false;
            }
          }
          if (!ok) break;
          tc_fence_after();
        }
        const int s = i % kZuvRing;
        if (!mbar_wait(smem_u32(&full_bar[s]), (i / kZuvRing) & 1)) {
          atomicOr(args.status, DEV_TIMEOUT_TMA);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t b_s = ring0 + s * kZuvStage;
        const int cb = i < NK ? 0 : (i - NK) / NK;  // phase-2 column block
        const int kb = i < NK ? i : i - NK - cb * NK;
        const uint32_t a_s = a0 + kb * A_KB;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = sw128_desc(a_s + j * 32);
          const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
          if (i < NK)
            tc_mma<false>(tmem, ad, sw128_desc(b_s + j * 32), IDESC1, acc);
          else
            tc_mma<false>(tmem + acc2_col(cb), ad, sw128_desc(b_s + j * 32), idesc2, acc);
        }
        tc_commit(smem_u32(&empty_bar[s]));
        if (i >= NK && kb == NK - 1) tc_commit(smem_u32(&acc2_bar[cb]));  // this column block is done
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int q = warp & 3;            // TMEM lane quarter
    const int half = (warp - 2) >> 2;  // which half of the columns
    const int row = q * 32 + lane;
    const int m = m_tile * BM + row;
    const bool live = m < args.M;
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    grid_dep_wait();  // gw, W s and the logits come from earlier kernels
    // Per-tile constants, staged in shared memory while the MMAs run (when they fit): the gw rows
    // of the tile's slots; per slot (b1 + W s_p) / 2 for P (zero for Q); u / 2.  Rows past M (a
    // ragged last tile) take the tile's first slot, so that their lookups stay inside what is
    // staged.
    const int first_slot = (m_tile * BM) / args.cand;
    const int slot = live ? m / args.cand : first_slot;  // stream * slots + slot
    const int nslots = (min(args.M, m_tile * BM + BM) - 1) / args.cand - first_slot + 1;
    const bool staged = (nslots * (R + H) + H) * 4 <= kZuvConst;
    float* s_gw = reinterpret_cast<float*>(ring + kZuvRing * kZuvStage);  // [nslots][R]
    float* s_add = s_gw + nslots * R;                                       // [nslots][H]
    float* s_u = s_add + nslots * H;                                        // [H]
    const void* col_u = is_q ? args.u_b : args.u_a;
    if (staged) {
      const int et = threadIdx.x - 64;
      for (int i = et; i < nslots * (R / 4); i += kEpiThreads) {
        const int sl = i / (R / 4), c4 = i % (R / 4);
        *reinterpret_cast<float4*>(s_gw + sl * R + c4 * 4) =
            *reinterpret_cast<const float4*>(args.gw + static_cast<size_t>(first_slot + sl) * R + c4 * 4);
      }
      for (int i = et; i < nslots * (H / 4); i += kEpiThreads) {
        const int sl = i / (H / 4), col = (i % (H / 4)) * 4;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!is_q) {
          a4 = ldw4<true>(args.b1, col);
          const int qs = first_slot + sl, st = qs / args.slots;
          if (qs - st * args.slots < args.slots - 1) {
            const float4 r4 = *reinterpret_cast<const float4*>(args.wsp + static_cast<size_t>(qs - st) * H + col);
            a4.x += r4.x;
            a4.y += r4.y;
            a4.z += r4.z;
            a4.w += r4.w;
          }
        }
        *reinterpret_cast<float4*>(s_add + sl * H + col) = make_float4(0.5f * a4.x, 0.5f * a4.y, 0.5f * a4.z, 0.5f * a4.w);
      }
      for (int i = et; i < H / 4; i += kEpiThreads) {
        const float4 u4 = ldw4<true>(col_u, i * 4);
        *reinterpret_cast<float4*>(s_u + i * 4) = make_float4(0.5f * u4.x, 0.5f * u4.y, 0.5f * u4.z, 0.5f * u4.w);
      }
    }
    named_barrier_sync(1, kEpiThreads);
    // phase 1: z = SiLU(acc1 + gw[slot]) in bf16, over the b tile, swizzled as TMA would load it;
    // SiLU(x) = h + h tanh(h), h = x / 2, with the tanh in packed half precision (z is rounded to
    // bf16, whose step is eight times the half-precision tanh's)
    bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&acc1_bar), 0));
    if (!ok && lane == 0) atomicOr(args.status, DEV_TIMEOUT_ACC);
    tc_fence_after();
    const float* gwr = staged ? s_gw + (slot - first_slot) * R : args.gw + static_cast<size_t>(slot) * R;
    // z in two passes over the column halves [0, R/2) and [R/2, R), each handed to the MMA warp
    // as soon as it is written; within a pass the two warps of a lane quarter split the 32-column
    // chunks, whose TMEM loads are issued together before they are converted.
    constexpr int NCHK = R / 32;       // 32-column chunks of the row
    constexpr int PASS = NCHK / 2;     // chunks per pass
    constexpr int MINE = PASS >= 2 ? PASS / 2 : 1;  // chunks of one warp per pass
#pragma unroll
    for (int zh = 0; zh < 2; ++zh) {
      const bool work = PASS >= 2 || half == zh;  // one chunk per pass (r = 64): one warp of two
      const int c0 = zh * (R / 2) + (PASS >= 2 ? half * MINE * 32 : 0);
      if (work) {
        uint32_t rbuf[MINE][32];
#pragma unroll
        for (int k = 0; k < MINE; ++k) tmem_ld32_nowait(trow + c0 + 32 * k, rbuf[k]);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < MINE; ++k) {
          const int c = c0 + 32 * k;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rbuf[k][i]);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gwr + c + i);
            const float h0 = 0.5f * (v[i] + g4.x), h1 = 0.5f * (v[i + 1] + g4.y);
            const float h2 = 0.5f * (v[i + 2] + g4.z), h3 = 0.5f * (v[i + 3] + g4.w);
            const float2 t01 = tanh2_f16(h0, h1), t23 = tanh2_f16(h2, h3);
            v[i] = live ? fmaf(h0, t01.x, h0) : 0.f;
            v[i + 1] = live ? fmaf(h1, t01.y, h1) : 0.f;
            v[i + 2] = live ? fmaf(h2, t23.x, h2) : 0.f;
            v[i + 3] = live ? fmaf(h3, t23.y, h3) : 0.f;
          }
          uint8_t* kbase = a_reg + (c / 64) * A_KB + row * 128;
          const int ch0 = (c % 64) / 8;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            *reinterpret_cast<uint4*>(kbase + (((ch0 + t) ^ (row & 7)) << 4)) = pack8_bf16(v + 8 * t);
        }
      }
      fence_proxy_async();  // the tensor core reads this half of z next
      tc_fence_before();
      named_barrier_sync(1, kEpiThreads);
      if (threadIdx.x == 64) mbar_arrive(smem_u32(&z_bar[zh]));
    }
    // phase 2: P or Q, one column block at a time.  Each thread owns one row and stores its
    // f16 values straight to global memory, 32 bytes per store (16 when the output is only
    // 16-byte aligned): the ring still feeds the next block's MMAs, so nothing is staged.
    const float l = live ? args.vals[m] : 0.f;
    const int stream_i = slot / args.slots, p = slot - stream_i * args.slots;
    const float* rb = (!is_q && live && p < args.slots - 1) ? args.wsp + static_cast<size_t>(slot - stream_i) * H
                                                            : nullptr;
    const float* addr = s_add + (slot - first_slot) * H;
    const int nsub = NC / 64;  // 128-byte (64-column f16) sub-tiles of a column block
    const int halves = nsub >= 2 ? 2 : 1;
    __half* out_row = static_cast<__half*>(is_q ? args.q : args.p) + static_cast<size_t>(live ? m : 0) * H;
    uint8_t* stg = ring + (warp - 2) * 8192;  // staging of the last block (see below)
    const int y0 = m_tile * BM + q * 32;
    const CUtensorMap* out_map = is_q ? &args.q_map : &args.p_map;
    const bool wide = ((reinterpret_cast<uintptr_t>(is_q ? args.q : args.p) | static_cast<uintptr_t>(H) * 2) & 31) == 0;
    for (int cb = 0; cb < NH2; ++cb) {
      const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&acc2_bar[cb]), 0));
      if (!got && lane == 0) atomicOr(args.status, DEV_TIMEOUT_ACC);
      ok = ok && got;
      if (cb == 0) grid_dep_launch();  // the next kernel may start its prologue
      tc_fence_after();
      const int cbg = cb0 + cb;  // the column block in P or Q
      const int j0 = cbg * nsub + half * nsub / halves, j1 = cbg * nsub + (half + 1) * nsub / halves;
      for (int j = j0; half < halves && j < j1; ++j) {
        float v[64];
        {
          uint32_t r[2][32];
          const uint32_t tc = trow + acc2_col(cb) + (j - cbg * nsub) * 64;
          tmem_ld32_nowait(tc, r[0]);
          tmem_ld32_nowait(tc + 32, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = __uint_as_float(r[0][i]);
            v[32 + i] = __uint_as_float(r[1][i]);
          }
        }
        if (staged) {
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const int col = j * 64 + i;
            const float4 u4 = *reinterpret_cast<const float4*>(s_u + col);
            const float4 a4 = *reinterpret_cast<const float4*>(addr + col);
            v[i] = fmaf(0.5f, v[i], fmaf(u4.x, l, a4.x));
            v[i + 1] = fmaf(0.5f, v[i + 1], fmaf(u4.y, l, a4.y));
            v[i + 2] = fmaf(0.5f, v[i + 2], fmaf(u4.z, l, a4.z));
            v[i + 3] = fmaf(0.5f, v[i + 3], fmaf(u4.w, l, a4.w));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const int col = j * 64 + i;
            const float4 u4 = ldw4<true>(col_u, col);
            float4 add = (!is_q) ? ldw4<true>(args.b1, col) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (rb != nullptr) {
              const float4 r4 = *reinterpret_cast<const float4*>(rb + col);
              add.x += r4.x;
              add.y += r4.y;
              add.z += r4.z;
              add.w += r4.w;
            }
            v[i] = 0.5f * (v[i] + add.x + u4.x * l);
            v[i + 1] = 0.5f * (v[i + 1] + add.y + u4.y * l);
            v[i + 2] = 0.5f * (v[i + 2] + add.z + u4.z * l);
            v[i + 3] = 0.5f * (v[i + 3] + add.w + u4.w * l);
          }
        }
        if (cb == NH2 - 1) {
          // The last block: every MMA has completed, so the ring is free to stage the rows (two
          // 4 KB halves per warp) for tensor-map stores, which leave the warps at once.
          uint8_t* buf = stg + ((j - j0) & 1) * 4096;
          if (j - j0 >= 2) {
            if (lane == 0) bulk_wait_read<1>();  // the store that used this half has read it
            __syncwarp();
          }
          stage_row<2>(buf, lane, v);
          fence_proxy_async();
          __syncwarp();
          if (lane == 0 && y0 < args.M && ok) {
            tma_store_2d(out_map, j * 64, y0, smem_u32(buf));
            bulk_commit();
          }
        } else if (live && ok) {
          // Earlier blocks: the ring still feeds the next block's MMAs, so each thread stores its
          // row's 64 values straight from registers.
          uint4 h[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) h[c] = pack8_f16_clamped(v + 8 * c);
          __half* dst = out_row + j * 64;
          if (wide) {
#pragma unroll
            for (int c = 0; c < 8; c += 2) st_global_32(dst + 8 * c, h[c], h[c + 1]);
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + 8 * c) = h[c];
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int R>
cudaError_t launch_zuv_t(const ZuvArgs& a, cudaStream_t stream) {
  const int smem = (R / 64) * BM * 128 + kZuvRing * kZuvStage + kZuvConst + 1024;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(zuv_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  // one column block per CTA when that still fits one wave
  const int tiles = (a.M + BM - 1) / BM, nh = a.H > 256 ? a.H / 256 : 1;
  cfg.gridDim = dim3(tiles, (nh > 1 && tiles * 2 * nh <= sm_count()) ? 2 * nh : 2, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return cudaLaunchKernelEx(&cfg, zuv_kernel<R>, a);
}


}  // namespace

cudaError_t launch_gemm(const GemmArgs& args, bool is_bf16, int BN, int split_k, cudaStream_t stream) {
  if (split_k < 1 || split_k > 8 || (BM % split_k) != 0) return cudaErrorInvalidValue;
  return is_bf16 ? dispatch_bn<true>(args, BN, split_k, stream) : dispatch_bn<false>(args, BN, split_k, stream);
}

bool zuv_supported(bool is_bf16, int r, int H) {
  return is_bf16 && (r == 64 || r == 128 || r == 256) && H % 64 == 0 && H >= 64 && (H <= 256 || H == 512);
}

cudaError_t launch_zuv(const ZuvArgs& a, cudaStream_t stream) {
  if (!zuv_supported(true, a.r, a.H)) return cudaErrorInvalidValue;
  switch (a.r) {
    case 64: return launch_zuv_t<64>(a, stream);
    case 128: return launch_zuv_t<128>(a, stream);
    default: return launch_zuv_t<256>(a, stream);
  }
}

cudaError_t launch_pair_combine(const float* hp, void* s, bool is_bf16, int N, int B, int r, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(N) * (B - 1) * r;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((total + threads - 1) / threads, 152 * 8));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return is_bf16 ? cudaLaunchKernelEx(&cfg, pair_combine_kernel<true>, hp, s, N, B, r)
                 : cudaLaunchKernelEx(&cfg, pair_combine_kernel<false>, hp, s, N, B, r);
}

unsigned int* device_status_word(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_status_word);
  return static_cast<unsigned int*>(p);
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_tmap(CUtensorMap* map, const void* base, bool is_bf16, uint64_t rows, uint64_t cols, uint64_t pitch_elems,
               uint32_t box_rows, const char** err) {
  static EncodeTiled encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      *err = "cuTensorMapEncodeTiled is not available from the driver";
      return false;
    }
    encode = reinterpret_cast<EncodeTiled>(fn);
  }
  const uint32_t esize = is_bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * esize};
  cuuint32_t box[2] = {128u / esize, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled rejected a tensor map (alignment, pitch or box)";
    return false;
  }
  return true;
}

}  // namespace dcoco
