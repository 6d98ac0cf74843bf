// Fused drafter output projection and top-K on the 5th-generation tensor cores.
//
// [Blog] "Score neighboring candidates in parallel" and "Keep the leading candidates": the
// corrector starts from what the drafter's own pass produced, whose last step projects the
// final hidden state h of every slot onto the vocabulary (l[v] = h . W_lm[v]) and keeps the K
// largest logits.  Here both happen in one pass over W_lm: the [rows, V] logits exist only in
// tensor memory and never reach HBM.
//
// Kernel shape (persistent, one CTA per SM, 10 warps):
//   Each CTA covers one 128-row tile of h and walks one contiguous range of 256-token
//   vocabulary tiles.
//   warp 0     TMA producer: this CTA's h tile and the W_lm tile per k-block.
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and issues
//              tcgen05.mma; each stage is released back to the producer by a commit.
//   warps 2-5  epilogue (one per TMEM lane quarter; warps 6-9 idle): while the next tile
//              accumulates in the other buffer, each thread reads the 256 columns of its row
//              and keeps a running top-K of everything it has seen: a descending list of
//              KR >= K keys in registers.  Per 32 columns a lane compares their maximum with
//              its list's last key and, if it reaches it, marks the values that do and parks
//              the 32 values in shared memory; then every pass of a loop inserts each lane's
//              next marked value with one compare-exchange pass over the lists, the whole warp
//              together (lanes with nothing left pass a null key), until no lane has marks left.
// CTA-pair variant (bf16): the two CTAs of a cluster of 2 act as one MMA unit.  Each holds its
// own 128-row h tile and one half (128 tokens) of the W_lm tile; the even CTA issues
// 256 x 256 x 16 MMAs (cta_group::2) that read A and B from both CTAs' shared memory and leave
// each CTA's 128 rows in its own TMEM.  Per SM that halves the W_lm bytes the tensor core reads
// and TMA writes per flop; the smaller stages (32 KB) also leave room for 6 of them.
// Both CTAs' loads count on the even CTA's stage barrier; its commits release the stages and
// accumulators in both CTAs (one commit arriving on the same barrier offset in each CTA); both
// CTAs' epilogues release an accumulator to the even CTA.  Every TMA load writes only the
// issuing CTA's own shared memory.
// Each (row, cluster) leaves a sorted list of K keys; lm_merge_kernel merges the lists of a
// row.  Keys are ordered value bits << 32 | ~token, as in the top-K kernel, so the
// selection is exact on the fp32 logits and deterministic.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;  // vocabulary entries per tile: one accumulator of 256 fp32 columns
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = BN * 128;
constexpr int kMaxListsPerLane = 16;  // merge: up to 512 lists per row
// Epilogue warps that share one row's 256 columns of a tile (each keeps its own list of its
// 256 / kColSplit columns); 4 * kColSplit epilogue warps work, the others stay idle.  One warp
// per row needs about 30 % fewer insertion passes in all than two warps with a list each (a
// row's list fills once instead of twice), and the passes take tensor-pipe issue slots and
// power: the kernel is 1.5 % faster with 1 than with 2.
constexpr int kColSplit = 1;
constexpr int kEpiWorkWarps = 4 * kColSplit;
constexpr int kStageValsBytes = kEpiThreads * 32 * 4;  // one 32-column chunk per epilogue thread
// One-CTA MMAs: 4 stages of the h tile and the whole W_lm tile.  CTA pairs: 6 stages of the h
// tile and half the W_lm tile.
template <bool kPair>
struct Pipe {
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr int kBStage = kPair ? B_BYTES / 2 : B_BYTES;
  static constexpr int kStageBytes = A_BYTES + kBStage;
  static constexpr int kSmem = kStages * kStageBytes + kStageValsBytes + 1024;
};
constexpr int kMaxStages = 6;
static_assert(Pipe<true>::kSmem <= 227 * 1024 - 256, "pair pipeline exceeds shared memory");

struct LmArgs {
  CUtensorMap a_map;  // h [rows, d], box {128 bytes, 128 rows}
  CUtensorMap b_map;  // W_lm [V, d], box {128 bytes, BN / cm rows} (each CTA of a pair loads half)
  unsigned long long* partial;  // [rows, n_lists, K] keys, each list descending
  int rows, d, V, K;
  int n_vt;    // vocabulary tiles, ceil(V / BN)
  int nclus;   // clusters per row group (vocabulary ranges); n_lists = kColSplit * nclus
  int cm;      // CTAs per cluster: 2 for CTA pairs, else 1
  unsigned int* status;
};

// Inserts x into the descending list a[0..KR-1] and drops the smallest key: one
// compare-exchange pass (x = 0, below every real key, leaves the list unchanged).
template <int KR>
__device__ __forceinline__ void list_insert(unsigned long long (&a)[KR], unsigned long long x) {
#pragma unroll
  for (int j = 0; j < KR; ++j) {
    const unsigned long long hi = a[j] > x ? a[j] : x;
    x = a[j] > x ? x : a[j];
    a[j] = hi;
  }
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// KR: list length kept per thread (K rounded up to 4, 8, 16, 32 or 64).  kPair: CTA-pair MMAs
// (bf16 only; clusters of exactly 2).
template <bool kBf16, int KR, bool kPair>
__global__ void __launch_bounds__(kThreads, 1) lm_topk_kernel(const __grid_constant__ LmArgs args) {
  static_assert(!kPair || kBf16, "CTA-pair MMAs are built for bf16 inputs");
  constexpr int BK = kBf16 ? 64 : 32;  // elements per 128-byte row of a stage
  constexpr int UK = kBf16 ? 16 : 8;   // K of one MMA instruction
  constexpr uint32_t IDESC = mma_idesc(kBf16 ? 1u : 2u, kPair ? 2 * BM : BM, BN);
  constexpr int S = Pipe<kPair>::kStages;
  constexpr int STAGE_BYTES = Pipe<kPair>::kStageBytes;

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ uint32_t tmem_base_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int CW = KR >= 64 ? 16 : 32;  // columns per TMEM load (fewer registers beside a long list)
  constexpr int cm = kPair ? 2 : 1;
  const int K = args.K;
  const uint32_t rank = cm > 1 ? cluster_rank() : 0u;
  const bool leader = rank == 0;  // pairs: the CTA that issues the MMAs
  const int clus = blockIdx.x / cm;
  const int m_tile = blockIdx.y * cm + static_cast<int>(rank);
  const int t0 = static_cast<int>(static_cast<long long>(clus) * args.n_vt / args.nclus);
  const int t1 = static_cast<int>(static_cast<long long>(clus + 1) * args.n_vt / args.nclus);
  const int ntile = t1 - t0;
  const int nkb = (args.d + BK - 1) / BK;
  const uint16_t mask = static_cast<uint16_t>((1u << cm) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);  // pairs: the even CTA's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), (kPair ? 2 : 1) * kEpiWorkWarps);  // pairs: both CTAs' epilogue warps
    }
    fence_mbar_init();
    prefetch_tmap(&args.a_map);
    prefetch_tmap(&args.b_map);
  }
  if (warp == 1) {
    if constexpr (kPair)
      tmem_alloc_pair(smem_u32(&tmem_base_s), 2 * BN);
    else
      tmem_alloc(smem_u32(&tmem_base_s), 2 * BN);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (kPair) cluster_sync();  // both CTAs' barriers exist before the first remote arrival lands
  const uint32_t tmem = tmem_base_s;
  const uint32_t smem0 = smem_u32(smem);
  const int total = ntile * nkb;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int slice = BN / cm;
      for (int i = 0; i < total; ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1)) {
          atomicOr(args.status, DEV_TIMEOUT_MMA);
          break;
        }
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t a_s = smem0 + s * STAGE_BYTES;
        const uint32_t b_s = a_s + A_BYTES;
        const int tile = t0 + i / nkb;
        const int kx = (i % nkb) * BK;
        if constexpr (kPair) {
          // both CTAs' h tiles and W_lm halves count on the even CTA's barrier
          const uint32_t fb_lead = leader ? fb : map_to_rank(fb, 0);
          if (leader) mbar_expect_tx(fb, 2 * STAGE_BYTES);
          tma_load_2d_pair(a_s, &args.a_map, kx, m_tile * BM, fb_lead);
          tma_load_2d_pair(b_s, &args.b_map, kx, tile * BN + static_cast<int>(rank) * slice, fb_lead);
        } else {
          mbar_expect_tx(fb, STAGE_BYTES);  // the h tile and the whole W_lm tile
          tma_load_2d(a_s, &args.a_map, kx, m_tile * BM, fb);
          tma_load_2d(b_s, &args.b_map, kx, tile * BN, fb);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (!kPair || leader)) {
      int i = 0;
      bool ok = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const int buf = t & 1;
        const bool freed = kPair ? mbar_wait_cluster(smem_u32(&acc_empty[buf]), ((t >> 1) & 1) ^ 1)
                                 : mbar_wait(smem_u32(&acc_empty[buf]), ((t >> 1) & 1) ^ 1);
        if (!freed) {
          atomicOr(args.status, DEV_TIMEOUT_ACC);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int kb = 0; kb < nkb; ++kb, ++i) {
          const int s = i % S;
          const uint32_t ph = (i / S) & 1;
          const bool landed = kPair ? mbar_wait_cluster(smem_u32(&full_bar[s]), ph) : mbar_wait(smem_u32(&full_bar[s]), ph);
          if (!landed) {
            atomicOr(args.status, DEV_TIMEOUT_TMA);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_s = smem0 + s * STAGE_BYTES;
          const uint32_t b_s = a_s + A_BYTES;
#pragma unroll
          for (int j = 0; j < BK / UK; ++j) {
            const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
            if constexpr (kPair)
              tc_mma_pair_f16(d_tmem, sw128_desc(a_s + j * 32), sw128_desc(b_s + j * 32), IDESC, acc);
            else
              tc_mma<!kBf16>(d_tmem, sw128_desc(a_s + j * 32), sw128_desc(b_s + j * 32), IDESC, acc);
          }
          if constexpr (kPair)
            tc_commit_pair_multicast(smem_u32(&empty_bar[s]), mask);
          else
            tc_commit(smem_u32(&empty_bar[s]));
        }
        if (ok) {
          if constexpr (kPair)
            tc_commit_pair_multicast(smem_u32(&acc_full[buf]), mask);
          else
            tc_commit(smem_u32(&acc_full[buf]));
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWorkWarps) {
    // ------------------------------------------------------------ epilogue (warps 2..)
    constexpr int CPW = BN / kColSplit;  // columns of each tile per warp
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which CPW columns of each tile
    const int row = m_tile * BM + q * 32 + lane;
    const bool live = row < args.rows;
    // this warp's staging area: column i of the current chunk at sv[i * 32] (lanes interleaved)
    float* sv = reinterpret_cast<float*>(smem + S * STAGE_BYTES) + (warp - 2) * 32 * 32 + lane;
    unsigned long long a[KR];
#pragma unroll
    for (int j = 0; j < KR; ++j) a[j] = 0ull;  // below every real key
    // The last key's value: NaN while the list is not full (every value then reaches the key
    // test); rows past the end see only zero-filled inputs and +inf keeps them out.
    float thr = live ? __uint_as_float(0xFFFFFFFFu) : __int_as_float(0x7F800000);
    for (int t = 0; t < ntile; ++t) {
      const int buf = t & 1;
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&acc_full[buf]), (t >> 1) & 1));
      if (!ok) {
        if (lane == 0) atomicOr(args.status, DEV_TIMEOUT_ACC);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + half * CPW;
      const int col0 = (t0 + t) * BN + half * CPW;
      for (int c = 0; c < CPW; c += CW) {
        // Which of these CW columns reach this lane's threshold (columns past V hold products
        // with zero-filled W_lm rows and never count).
        uint32_t m = 0;
        {
          float v[CW];
          if constexpr (CW == 32)
            tmem_ld32(taddr + c, v);
          else
            tmem_ld16(taddr + c, v);
          // Most chunks hold nothing that reaches the list: one max, one compare.  (fmaxf skips
          // NaN, which ranks below every number; NaN thr, a list not yet full, takes every chunk.)
          float mx = v[0];
#pragma unroll
          for (int i = 1; i < CW; ++i) mx = fmaxf(mx, v[i]);
          if (!(mx < thr)) {
#pragma unroll
            for (int i = 0; i < CW; ++i) {
              m |= (v[i] < thr ? 0u : 1u) << i;
              sv[i * 32] = v[i];
            }
          }
        }
        const int valid = args.V - (col0 + c);
        if (valid < CW) m &= valid > 0 ? (1u << valid) - 1u : 0u;
        // Each pass inserts every lane's next marked value (the lowest marked column left), so
        // the warp runs as many passes as its busiest lane has marks, in a loop (not unrolled).
        while (__any_sync(0xFFFFFFFFu, m != 0u)) {
          const int i = m != 0u ? __ffs(m) - 1 : 0;
          const float x = sv[i * 32];
          const bool pass = m != 0u && !(x < thr);
          m &= m - 1u;
          list_insert<KR>(a, pass ? make_key(__float_as_uint(x), static_cast<uint32_t>(col0 + c + i)) : 0ull);
          thr = key_value(a[KR - 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair && !leader)
          mbar_arrive_cluster(map_to_rank(smem_u32(&acc_empty[buf]), 0));
        else
          mbar_arrive(smem_u32(&acc_empty[buf]));
      }
    }
    if (live) {
      unsigned long long* dst =
          args.partial + (static_cast<size_t>(row) * (kColSplit * args.nclus) + clus * kColSplit + half) *
                             static_cast<size_t>(K);
#pragma unroll
      for (int j = 0; j < KR; ++j)
        if (j < K) dst[j] = a[j];
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) {
    // the pair's TMEM is released together, once neither CTA reads it any more
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, 2 * BN);
    }
  } else if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
  if constexpr (kPair) cluster_sync();  // neither CTA leaves while a pair commit may still arrive in it
}

// One warp per row: K rounds of "largest head among the row's sorted lists".
__global__ void __launch_bounds__(256) lm_merge_kernel(const unsigned long long* __restrict__ partial, int rows,
                                                       int n_lists, int K, float* __restrict__ vals,
                                                       int32_t* __restrict__ ids) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const unsigned long long* base = partial + static_cast<size_t>(row) * n_lists * K;
  unsigned long long head[kMaxListsPerLane];
  int pos[kMaxListsPerLane];
#pragma unroll
  for (int j = 0; j < kMaxListsPerLane; ++j) {
    const int l = lane + 32 * j;
    pos[j] = 0;
    head[j] = l < n_lists ? base[static_cast<size_t>(l) * K] : 0ull;
  }
  for (int r = 0; r < K; ++r) {
    unsigned long long best = 0ull;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < kMaxListsPerLane; ++j)
      if (head[j] > best) {
        best = head[j];
        bj = j;
      }
    unsigned long long wmax = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, wmax, o);
      wmax = other > wmax ? other : wmax;
    }
    // keys of one row are distinct (each token sits in exactly one list), so one lane advances
    if (bj >= 0 && best == wmax) {
#pragma unroll
      for (int j = 0; j < kMaxListsPerLane; ++j)
        if (j == bj) {
          ++pos[j];
          head[j] = pos[j] < K ? base[static_cast<size_t>(lane + 32 * j) * K + pos[j]] : 0ull;
        }
    }
    if (lane == 0) {
      vals[static_cast<size_t>(row) * K + r] = key_value(wmax);
      ids[static_cast<size_t>(row) * K + r] = static_cast<int32_t>(key_index(wmax));
    }
  }
}

struct Plan {
  int cm, m_groups, nclus, n_vt;
  bool pair;
};

int list_len(int K) { return K <= 4 ? 4 : K <= 8 ? 8 : K <= 16 ? 16 : K <= 32 ? 32 : 64; }

using KernelFn = void (*)(LmArgs);

template <bool kBf16, bool kPair>
KernelFn kernel_for(int KR) {
  switch (KR) {
    case 4: return lm_topk_kernel<kBf16, 4, kPair>;
    case 8: return lm_topk_kernel<kBf16, 8, kPair>;
    case 16: return lm_topk_kernel<kBf16, 16, kPair>;
    case 32: return lm_topk_kernel<kBf16, 32, kPair>;
    default: return lm_topk_kernel<kBf16, 64, kPair>;
  }
}

// Kernel instances: f32, bf16 (one-CTA MMAs), bf16 CTA pairs; five list lengths each.
constexpr int kSlots = 15;
struct Instance {
  KernelFn fn;
  int slot, smem;
};
Instance instance(bool is_bf16, bool pair, int KR) {
  const int k = KR == 4 ? 0 : KR == 8 ? 1 : KR == 16 ? 2 : KR == 32 ? 3 : 4;
  if (pair) return {kernel_for<true, true>(KR), 10 + k, Pipe<true>::kSmem};
  if (is_bf16) return {kernel_for<true, false>(KR), 5 + k, Pipe<false>::kSmem};
  return {kernel_for<false, false>(KR), k, Pipe<false>::kSmem};
}

// Sets the dynamic shared-memory size once per kernel instance and device.
cudaError_t configure(const Instance& in) {
  static bool done[64][kSlots] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev][in.slot]) {
    e = cudaFuncSetAttribute(in.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, in.smem);
    if (e != cudaSuccess) return e;
    done[dev][in.slot] = true;
  }
  return cudaSuccess;
}

// Clusters of `cm` CTAs of this kernel that fit on the device at once (0 on failure).
int active_clusters(const Instance& in, int cm) {
  if (configure(in) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cm * 64, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = in.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cm;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(in.fn), &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// The launch plan.  CTA pairs (bf16) when pair_mode > 0, or when pair_mode == 0 and h has at
// least two row tiles; otherwise the one-CTA kernel (clusters of 1).  Then as many vocabulary
// ranges as fit in one wave.
cudaError_t plan_for(bool is_bf16, int rows, int V, int K, int pair_mode, Plan* p) {
  const int KR = list_len(K);
  const int m_tiles = (rows + BM - 1) / BM;
  p->n_vt = (V + BN - 1) / BN;
  p->pair = is_bf16 && (pair_mode > 0 || (pair_mode == 0 && m_tiles >= 2));
  static int cache[64][kSlots];  // active clusters + 1 per device and instance (0 = unknown)
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const Instance in = instance(is_bf16, p->pair, KR);
  p->cm = p->pair ? 2 : 1;
  int& c = cache[dev][in.slot];
  if (c == 0) c = active_clusters(in, p->cm) + 1;
  p->m_groups = (m_tiles + p->cm - 1) / p->cm;
  const int fit = std::max(1, c - 1);
  p->nclus = std::max(1, std::min(p->n_vt, fit / p->m_groups));
  return cudaSuccess;
}

// Guards the per-device plan and attribute caches against concurrent calls.
std::mutex g_plan_mu;

}  // namespace

size_t lm_topk_partial_bytes(bool is_bf16, int rows, int V, int K, int pair_mode) {
  Plan p;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (plan_for(is_bf16, rows, V, K, pair_mode, &p) != cudaSuccess) return 0;
  return static_cast<size_t>(rows) * (kColSplit * p.nclus) * K * 8;
}

cudaError_t launch_lm_topk(const void* h, const void* W_lm, bool is_bf16, int rows, int d, int V, int K, int pair_mode, float* vals, int32_t* ids, void* partial, size_t partial_bytes,
                           unsigned int* status, cudaStream_t stream) {
  Plan p;
  std::unique_lock<std::mutex> lock(g_plan_mu);
  cudaError_t e = plan_for(is_bf16, rows, V, K, pair_mode, &p);
  if (e != cudaSuccess) return e;
  const int n_lists = kColSplit * p.nclus;
  if (n_lists > 32 * kMaxListsPerLane) return cudaErrorInvalidValue;
  if (static_cast<size_t>(rows) * n_lists * K * 8 > partial_bytes) return cudaErrorInvalidValue;
  LmArgs a;
  const char* err = nullptr;
  if (!make_tmap(&a.a_map, h, is_bf16, static_cast<uint64_t>(rows), static_cast<uint64_t>(d), static_cast<uint64_t>(d),
                 BM, &err) ||
      !make_tmap(&a.b_map, W_lm, is_bf16, static_cast<uint64_t>(V), static_cast<uint64_t>(d), static_cast<uint64_t>(d),
                 static_cast<uint32_t>(BN / p.cm), &err))
    return cudaErrorInvalidValue;
  a.partial = static_cast<unsigned long long*>(partial);
  a.rows = rows;
  a.d = d;
  a.V = V;
  a.K = K;
  a.n_vt = p.n_vt;
  a.nclus = p.nclus;
  a.cm = p.cm;
  a.status = status;
  const Instance in = instance(is_bf16, p.pair, list_len(K));
  e = configure(in);
  lock.unlock();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.cm * p.nclus, p.m_groups, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = in.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cm;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, in.fn, a);
  if (e != cudaSuccess) return e;
  lm_merge_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(static_cast<const unsigned long long*>(partial), rows, n_lists, K,
                                                      vals, ids);
  return cudaGetLastError();
}

}  // namespace dcoco
