// Host-side launchers shared between the kernel translation units and the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dcoco {

// Kernels enqueued by this thread while set carry the programmatic-stream-serialization launch
// attribute, so that each may start (prologue, weight loads) while its predecessor finishes.
// It is set only where every predecessor is one of this library's kernels, none of which writes
// the weights (the cycle after its helper streams join, and the second and later kernels of the
// pair-state and slot chains), and every kernel waits (grid_dep_wait) before touching its data.
extern thread_local bool g_pdl;
struct PdlScope {
  PdlScope() { g_pdl = true; }
  ~PdlScope() { g_pdl = false; }
};
// Fills attr with the programmatic-serialization attribute when g_pdl is set; returns the count (0 or 1).
inline unsigned pdl_attr(cudaLaunchAttribute* attr) {
  if (!g_pdl) return 0;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

// Streaming multiprocessors of the current device (152 if the query fails); cached per device.
int sm_count();

// ------------------------------------------------------------------ top-K
// Rows of `logits` ([rows, V], bf16 bits if is_bf16 else f32); ctas_per_row in 1..8.
// after_unrelated: the kernel is launched programmatically behind a kernel that does not write
// the logits (and itself started only after the logits' producer finished), so it does not
// wait for that kernel to finish.
cudaError_t launch_topk(const void* logits, bool is_bf16, int rows, int V, int K, int ctas_per_row, float* vals,
                        int32_t* ids, cudaStream_t stream, bool after_unrelated = false);
// Thread blocks per row launch_topk uses (ctas_per_row 0: its automatic choice); at most four
// blocks of top-K are resident on one SM.
int topk_ctas_per_row(int rows, int V, bool is_bf16, int ctas_per_row);

// ------------------------------------------------------------------ fused LM head + top-K
// Bytes of the per-row partial lists launch_lm_topk needs (0 if no plan exists).  pair_mode 0
// uses CTA-pair MMAs for bf16 with at least two row tiles, 1 always for bf16, -1 never.
size_t lm_topk_partial_bytes(bool is_bf16, int rows, int V, int K, int pair_mode);
// h [rows, d], W_lm [V, d] (bf16 bits if is_bf16 else f32) -> vals, ids [rows, K].
cudaError_t launch_lm_topk(const void* h, const void* W_lm, bool is_bf16, int rows, int d, int V, int K, int pair_mode,
                           float* vals, int32_t* ids, void* partial, size_t partial_bytes, unsigned int* status,
                           cudaStream_t stream);

// ------------------------------------------------------------------ GEMM
// C[m, n] = sum_k A[m, k] * B[n, k] on tcgen05 tensor cores (bf16 -> kind::f16, f32 -> kind::tf32),
// fp32 accumulation in tensor memory, 128 x BN tiles, optional split-K across a thread-block
// cluster, and one fused epilogue per B group.
enum Epilogue : int {
  EPI_F32 = 0,        // out (f32) = acc
  EPI_ACT = 1,        // out (activation dtype) = acc
  EPI_LN = 2,         // out (activation dtype) = LayerNorm_noaffine(acc row)   (group covers the full row)
  EPI_SILU_BIAS = 3,  // out (activation dtype) = SiLU(acc + bias[m / bias_div, n])  (bias f32)
  // Scorer operand (no split-K): out = (acc + col_b[n] + col_u[n] * row_l[m] + row_bias[pair(m), n]) / 2,
  // written in half precision (clamped to +-30000) for bf16 inputs, f32 otherwise.  Row m is
  // candidate (stream, slot, k) with m / bias_div = stream * slots + slot; the pair row is
  // stream * (slots - 1) + slot and the last slot of a stream takes no row bias.  col_b and
  // row_bias may be null.
  EPI_PREP = 4,
};

struct GemmGroup {
  CUtensorMap b_map;    // B operand [Ng, K] (K contiguous), 128-byte swizzle, box {BK, min(BN,256)}
  CUtensorMap out_map;  // output [M, Ng] (pitch ldo), 128-byte swizzle, box {128 bytes, 32 rows}
  void* out;            // output base; row m, column n at out[m * ldo + n]
  int ldo;
  int epi;
  int n_tiles;        // Ng / BN
  const void* col_u;      // EPI_PREP: [Ng] weight dtype
  const void* col_b;      // EPI_PREP: [Ng] weight dtype, or null
  const float* row_bias;  // EPI_PREP: [pairs, Ng] f32 (pitch ld_bias), or null
};

struct GemmArgs {
  CUtensorMap a_map;        // A [M, K] tiled (box {BK, 128}); unused when the rows are gathered
  const int32_t* gather;    // non-null: A row m is table row gather[m]
  int gather_limit;         // rows of the gather table (ids outside [0, limit) are replaced by 0)
  const void* gather_base;  // the gather table (rows are loaded from here by the epilogue warps)
  int gather_pitch_bytes;
  int M, K;
  int n_groups;             // 1 to 3 (each group its own B operand, output and epilogue)
  GemmGroup g[3];
  const float* bias;        // EPI_SILU_BIAS
  int bias_div, ld_bias;
  const float* row_l;       // EPI_PREP: [M] per-row scale
  int slots;                // EPI_PREP: slots per stream
  float ln_eps;
  // Nonzero: the kernel lets the next kernel of its stream launch as soon as it starts (for a
  // next kernel that does not read this one's outputs; it must not wait on it either).
  int early_dependents;
  unsigned int* status;
};

// Encodes a 2-D tensor map over a row-major [rows, cols] matrix with the given row pitch (elements).
// box_rows is the box height (1 for a table that is only gathered from).
bool make_tmap(CUtensorMap* map, const void* base, bool is_bf16, uint64_t rows, uint64_t cols, uint64_t pitch_elems,
               uint32_t box_rows, const char** err);


// BN in {32, 64, 128, 256, 512}; split_k >= 1 (BN <= 256 when split_k > 1).
cudaError_t launch_gemm(const GemmArgs& args, bool is_bf16, int BN, int split_k, cudaStream_t stream);

// The candidate fusion and the candidate blocks of the first MLP layer in one kernel (bf16 only):
//   z = SiLU(b W_f[:, 0:r]^T + gw[slot])                      kept in shared memory, never stored
//   P = (z U^T + b1 + W s[pair] + u_a l) / 2,  Q = (z V^T + u_b l) / 2     f16, clamped to +-30000
// with the row and slot conventions of EPI_SILU_BIAS and EPI_PREP.  Grid (m_tiles, 2): y = 0
// writes P and y = 1 writes Q; both recompute z for their 128 rows.  When H spans two 256-column
// blocks and 4 m_tiles CTAs fit on the SMs, the grid is (m_tiles, 4): y & 1 picks P or Q and
// y >> 1 the column block.
struct ZuvArgs {
  CUtensorMap b_map;   // b [M, r], box {64, 128}
  CUtensorMap wf_map;  // W_f [r, 2r] (its first r columns act on b), box {64, r}
  CUtensorMap u_map;   // U [H, r], box {64, min(H, 256)}
  CUtensorMap v_map;   // V [H, r], same box
  void* p;             // P [M, H] f16 (16-byte aligned)
  void* q;             // Q [M, H] f16 (16-byte aligned)
  CUtensorMap p_map;   // P, box {64, 32} (stores of the last column block)
  CUtensorMap q_map;   // Q, same box
  const float* gw;     // [slots total, r] f32: W_f[:, r:2r] g of each slot
  const float* wsp;    // [pairs, H] f32: W s_p
  const float* vals;   // [M] f32: the candidate's logit l
  const void* b1;      // [H] bf16
  const void* u_a;     // [H] bf16
  const void* u_b;     // [H] bf16
  int M, r, H;
  int cand;            // candidates per slot (K): row m belongs to slot m / cand
  int slots;           // slots per stream (B)
  unsigned int* status;
};
// True when launch_zuv supports the shape (bf16, r in {64, 128, 256}, H a multiple of 64 up to 512).
bool zuv_supported(bool is_bf16, int r, int H);
cudaError_t launch_zuv(const ZuvArgs& a, cudaStream_t stream);

// s[n, p, :] = act(hp[n, p, 0:r] + hp[n, p+1, r:2r]), hp [N, B, 2r] f32, s [N, B-1, r] activation dtype.
cudaError_t launch_pair_combine(const float* hp, void* s, bool is_bf16, int N, int B, int r, cudaStream_t stream);

// ------------------------------------------------------------------ scores
struct ScoreArgs {
  const void* uz;       // [N, B, K, H] activation dtype
  const void* vz;
  const float* wsp;     // [N, B-1, H]
  const float* vals;    // [N, B, K]
  const void* u_a;      // [H] weight dtype
  const void* u_b;
  const void* b1;
  const void* w2;
  const void* b2;       // [1]
  float* S;             // [N, B-1, K, K]
  int N, B, K, H;
};
cudaError_t launch_scores(const ScoreArgs& a, bool is_bf16, cudaStream_t stream);
// Scores from operands already prepared by the EPI_PREP epilogue: uz holds the P rows
// (uz + b1 + W s + u_a l)/2 and vz the Q rows (vz + u_b l)/2, in half precision for bf16
// weights and f32 otherwise; wsp, u_a, u_b and b1 are not read.
cudaError_t launch_scores_prepped(const ScoreArgs& a, bool is_bf16, cudaStream_t stream);

// ------------------------------------------------------------------ walk + verify
struct SelectVerifyArgs {
  // walk (skipped when S == nullptr: `draft` is then read as the block to verify)
  const float* S;
  const float* vals;
  const int32_t* ids;
  int32_t* k_sel;
  int32_t* tokens;       // written by the walk, read by verification
  int rule;              // 0 prefix-first greedy walk, 1 discounted max-sum over whole paths
  float lam;             // rule 1: the discount (1 = Global-Sum)
  // verification (skipped when mode < 0)
  int mode;              // 0 greedy, 1 stochastic (point mass), 2 speculative (draft distribution p), -1 none
  const int32_t* draft;  // block to verify when there is no walk
  const int32_t* t;
  const float* q;
  const float* p;        // mode 2: [N, B, V] draft distribution
  const float* u;
  int32_t* accept_len;
  int32_t* committed;
  int32_t* n_commit;
  int32_t* near_tie;
  int N, B, K, V;
};
cudaError_t launch_select_verify(const SelectVerifyArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ status word
unsigned int* device_status_word(cudaError_t* err);

}  // namespace dcoco
