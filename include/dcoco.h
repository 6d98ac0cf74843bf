/*
 * dcoco.h -- C ABI of the DCOCO per-cycle correction hot path on one GB300 GPU.
 *
 * DCOCO (DFlash Contextual Corrector) re-selects a parallel drafter's B-slot block
 * from the drafter's own top-K candidates: it scores every candidate pair of
 * neighbouring slots with a small shared network and walks the block left to right,
 * then the verifier accepts the longest matching prefix.  Sources: Two Delta, "Two
 * Delta makes NVIDIA Nemotron 3.5 Super even faster with DCOCO" ("How DCOCO works");
 * jaehun.me review of arXiv 2610.12570, "Contextual Correction of Parallel Drafts for
 * Speculative Decoding", §3.1-§3.3 and App. D.
 *
 * Conventions (all entry points):
 *  - Return value: a dcoco_status.  Nothing aborts; no C++ exception crosses the ABI.
 *    On failure, dcoco_last_error() (per host thread) describes the first problem found.
 *  - Tensor pointers are caller-owned DEVICE memory on the current CUDA device, dense
 *    row-major, 16-byte aligned, and never alias one another.  The library allocates
 *    nothing: scratch comes from a caller-supplied workspace of at least the size the
 *    matching *_workspace_size() call returns (16-byte aligned, contents ignored).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *    asynchronously; no entry point synchronises.  Argument errors are reported before
 *    anything is enqueued; launch errors are reported as DCOCO_ERR_CUDA.
 *  - Kernel-side faults never trap: a bounded wait that gives up, or a token id outside
 *    [0, V) reaching the gather, sets a bit in the device status word
 *    (dcoco_device_status).
 *  - Shape limits: N >= 1, B >= 2, 1 <= K <= 64, K <= V, B <= 64.  Corrector width r in
 *    {32, 64, 128, 256, 512}; MLP width H a multiple of 64; d and E multiples of 8.
 *  - Index conventions: stream n in [0,N), slot i in [0,B), candidate k in [0,K),
 *    transition p in [0,B-1) scoring slot p -> slot p+1.
 */
#ifndef DCOCO_H_
#define DCOCO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DCOCO_OK = 0,
  DCOCO_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned pointer */
  DCOCO_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set */
  DCOCO_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  DCOCO_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  DCOCO_ERR_TIMEOUT = 5      /* device status word reports a bounded wait that gave up */
} dcoco_status;

typedef enum { DCOCO_F32 = 0, DCOCO_BF16 = 1 } dcoco_dtype;

typedef enum { DCOCO_VERIFY_GREEDY = 0, DCOCO_VERIFY_STOCHASTIC = 1 } dcoco_verify_mode;

/*
 * Corrector parameters, shared across slots and transitions (jaehun.me review of
 * arXiv 2610.12570, §3.2).  Every pointer has element type `dtype`; matrices are
 * [rows, cols] row-major ("out x in").
 *   W_e    [r, E]   projects the candidate's frozen token embedding
 *   W_h    [r, d]   projects the slot's drafter hidden state
 *   W_f    [r, 2r]  fuses [b; g]: columns 0..r-1 act on b, r..2r-1 on g
 *   W_pair [r, 2d]  pair state from [h_p; h_{p+1}]: columns 0..d-1 act on h_p
 *   U, V, W [H, r]  first MLP layer blocks on z_{p,a}, z_{p+1,b} and s_p
 *   u_a, u_b, b1, w2 [H]; b2 [1]   logit weights, first-layer bias, output layer
 */
typedef struct dcoco_weights {
  int dtype; /* dcoco_dtype */
  int d, E, r, H;
  const void* W_e;
  const void* W_h;
  const void* W_f;
  const void* W_pair;
  const void* U;
  const void* V;
  const void* W;
  const void* u_a;
  const void* u_b;
  const void* b1;
  const void* w2;
  const void* b2;
} dcoco_weights;

/* Library version (major*10000 + minor*100 + patch). */
int dcoco_version(void);

/* Description of the last failure on this host thread ("" if none). */
const char* dcoco_last_error(void);

/*
 * Reads and clears the device status word of the current device (DEV_* bits: 1 TMA
 * wait gave up, 2 MMA commit wait gave up, 4 accumulator wait gave up, 8 gathered id
 * out of range).  Synchronises `stream` first.  Returns DCOCO_ERR_TIMEOUT if any
 * timeout bit was set, DCOCO_OK otherwise; *bits receives the raw word (may be NULL).
 */
int dcoco_device_status(void* stream, uint32_t* bits);

/*
 * Self-test of the device-side failure path (the pages have no counterpart; it checks this
 * library's own error reporting).  Enqueues one warp that waits on an mbarrier nothing ever
 * arrives at, with the bounded wait every pipeline of the library uses but at most `polls`
 * polls (1..65536), and then sets bit 1 (a TMA wait gave up) in the status word, as a copy that
 * never lands would.  Nothing faults, no copy is in flight, and the context stays usable; the
 * next dcoco_device_status returns DCOCO_ERR_TIMEOUT.  Errors: DCOCO_ERR_INVALID_ARG for polls
 * outside [1, 65536].
 */
int dcoco_selftest_timeout(uint32_t polls, void* stream);

/*
 * Helper streams of dcoco_cycle, dcoco_cycle_table and dcoco_cycle_lm on the calling host thread:
 * two distinct caller-owned cudaStream_t of the device the cycles run on (the caller keeps them
 * alive while cycles use them), or NULL, NULL for the library's shared per-device streams (the
 * default).  Applies to later calls on this host thread only.  Errors: DCOCO_ERR_INVALID_ARG when
 * exactly one is NULL or both are the same stream.
 */
int dcoco_set_helper_streams(void* helper_a, void* helper_b);

/*
 * Tuning knob: thread blocks per logits row in dcoco_topk (1..8; 0 = automatic).
 * Process-wide; returns the previous value.
 */
int dcoco_set_topk_split(int ctas_per_row);

/*
 * a1. Top-K candidate retention (Two Delta blog, "Keep the leading candidates";
 * review §3.2): for every row (n,i) of `logits` [N, B, V] (dtype bf16 or f32), the K
 * largest values, sorted by value descending with equal values ordered by ascending
 * token id.  NaN ranks as -inf and is reported as -inf; -0 is reported as +0.
 *   vals [N, B, K] float32   the kept logits l_i(k) (exact widening of the input)
 *   ids  [N, B, K] int32     the token ids c_ik
 * Deterministic: the result does not depend on scheduling.  No workspace.
 * `logits` may be device memory or page-locked host memory mapped for the device (read once over
 * the host link; on GB300 that streams at about 100 GB/s, so a bulk copy into HBM first is faster);
 * pageable host memory gives DCOCO_ERR_INVALID_ARG.  The same holds for dcoco_cycle's logits.
 */
int dcoco_topk(const void* logits, int dtype, int N, int B, int V, int K, float* vals, int32_t* ids, void* stream);

/*
 * a2. Candidate representation (Two Delta blog, "Score neighboring candidates in
 * parallel"; review §3.2) with the first MLP layer's per-candidate blocks:
 *   b_ik = LN(W_e Emb[c_ik]),  g_i = LN(W_h h_i)   (non-affine LayerNorm, eps 1e-5)
 *   z_ik = SiLU(W_f [b_ik; g_i])
 *   uz = U z_ik,  vz = V z_ik
 *   ids [N, B, K] int32; emb [V, E] (w->dtype); h [N, B, d] (w->dtype)
 *   uz, vz [N, B, K, H], element type w->dtype (bf16 rounding of the fp32 result)
 */
size_t dcoco_candidate_repr_workspace_size(const dcoco_weights* w, int N, int B, int K);
int dcoco_candidate_repr(const int32_t* ids, const void* emb, int V, const void* h, const dcoco_weights* w, int N,
                         int B, int K, void* uz, void* vz, void* workspace, size_t workspace_bytes, void* stream);

/*
 * a3. Pair state (Two Delta blog, the pair context s_p; review §3.2):
 *   s_p = W_pair [h_p; h_{p+1}],  ws_pair[n, p] = W s_p      for p in [0, B-1)
 *   h [N, B, d] (w->dtype) -> ws_pair [N, B-1, H] float32
 */
size_t dcoco_pair_state_workspace_size(const dcoco_weights* w, int N, int B);
int dcoco_pair_state(const void* h, const dcoco_weights* w, int N, int B, float* ws_pair, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * dcoco_pair_state without a caller-supplied workspace.  The method's papers have no
 * counterpart: this exists for callers that cannot allocate device memory themselves --
 * for example a serving engine that hands nearly all HBM to its own pool up front (its
 * KV cache) and does not expose that pool, or host code that must not call cudaFree
 * because it can synchronise the whole device.  Same inputs, outputs and results as
 * dcoco_pair_state.
 *  - Scratch is a library-owned, statically sized 8 MiB device array
 *    (DCOCO_PAIR_STATE_NOALLOC_SCRATCH_BYTES).  Every GPU that loads the library holds it
 *    until the process exits.  A shape whose scratch (dcoco_pair_state_workspace_size)
 *    exceeds it is rejected with DCOCO_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call before any
 *    stream capture begins.
 *  - The call allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *  - All calls share the one array and it keeps the last call's contents.  Nothing in it
 *    needs to start at zero: every call writes each scratch byte before reading it.  Calls
 *    that can overlap on the GPU (other streams, other host threads) race on the array
 *    and corrupt each other's results: order them on one stream or with events.
 */
#define DCOCO_PAIR_STATE_NOALLOC_SCRATCH_BYTES (8u << 20)
int dcoco_pair_state_noalloc(const void* h, const dcoco_weights* w, int N, int B, float* ws_pair, void* stream);

/*
 * a4. Transition scores (Two Delta blog, "Score neighboring candidates in parallel";
 * review §3.2), all (B-1)K^2 at once, unnormalised:
 *   S[n,p,a,b] = l_{p+1}(b) + w2 . SiLU(uz[n,p,a] + vz[n,p+1,b] + ws_pair[n,p]
 *                                      + u_a l_p(a) + u_b l_{p+1}(b) + b1) + b2
 *   uz, vz [N, B, K, H] (w->dtype); ws_pair [N, B-1, H] f32; vals [N, B, K] f32
 *   S [N, B-1, K, K] float32, predecessor a major, successor b minor.
 */
int dcoco_score_transitions(const void* uz, const void* vz, const float* ws_pair, const float* vals,
                            const dcoco_weights* w, int N, int B, int K, float* S, void* stream);

/*
 * a5. Prefix-first greedy walk (Two Delta blog, "Select using the realized token
 * identities"; review §3.3): k_0 = argmax_k vals[n,0,k]; k_{p+1} = argmax_b S[n,p,k_p,b];
 * ties go to the lower candidate index, NaN ranks lowest.
 *   k_sel [N, B] int32, tokens [N, B] int32 (= ids[n, i, k_sel[n,i]])
 */
int dcoco_select(const float* S, const float* vals, const int32_t* ids, int N, int B, int K, int32_t* k_sel,
                 int32_t* tokens, void* stream);

/* Path rules for dcoco_select_path. */
enum { DCOCO_PATH_GREEDY = 0, DCOCO_PATH_DISCOUNTED = 1 };

/*
 * Whole-path selection rules on the same score grid, for comparison with the prefix-first walk
 * (review of arXiv 2610.12570, "path choice and ablation", Tab. 3: Global-Sum and a geometric
 * discount with lambda = 0.75).  Both formulas were lost from the page; the reading implemented
 * maximises, over all K^B paths,
 *   vals[n,0,k_0] + sum_{p=0}^{B-2} lambda^(p+1) S[n,p,k_p,k_{p+1}]        (lambda = 1: Global-Sum)
 * by the max-sum recursion in float32, each maximum taken by the lowest candidate index among
 * equal values (NaN ranks lowest).  rule DCOCO_PATH_GREEDY is dcoco_select (lambda unused);
 * DCOCO_PATH_DISCOUNTED needs 0 < lambda <= 1.  Outputs as for dcoco_select.  Errors:
 * DCOCO_ERR_INVALID_ARG for an unknown rule, lambda outside (0, 1] or a bad shape or pointer.
 */
int dcoco_select_path(const float* S, const float* vals, const int32_t* ids, int N, int B, int K, int rule,
                      float lambda, int32_t* k_sel, int32_t* tokens, void* stream);

/*
 * a6. Verification of the corrected draft (review §3.1 and App. D).
 *  GREEDY: t [N, B+1] int32 verifier greedy tokens; slot j is accepted while
 *    draft[j] == t[j]; A = accepted prefix length; commits draft[0..A-1] then t[A].
 *  STOCHASTIC (point-mass proposal): q [N, B+1, V] f32 verifier probabilities,
 *    u [N, B+1, 2] f32 uniforms in [0,1).  Slot j is accepted iff u[j,0] < q[j, draft[j]];
 *    at the first rejection j the committed token is the smallest v != draft[j] whose
 *    running residual mass (vocabulary order) exceeds u[j,1] * R with
 *    R = sum_{v != draft[j]} q[j, v]; if all B are accepted the bonus token is drawn the
 *    same way from q[B] (no exclusion) with u[B,1].  R <= 0 commits draft[j].  Masses are
 *    summed exactly in 62-bit fixed point (probabilities below 2^-38 round down by less than
 *    2^-62); rows of q must be probability vectors (summing to less than 3.5).
 *  Outputs: accept_len [N], committed [N, B+1] (-1 after the last committed token),
 *    n_commit [N] = accept_len + 1, all int32.  near_tie [N] int32 (may be NULL,
 *    stochastic only): 1 where u*R lay within 2^-30 R (about 1e-9 R) of a step of the running
 *    sum, where R < 2^-15 (truncation could matter), or where the row sums to 3.5 or more.
 *  Unused inputs of the other mode may be NULL.
 */
int dcoco_verify(int mode, const int32_t* draft, const int32_t* t, const float* q, const float* u, int N, int B, int V,
                 int32_t* accept_len, int32_t* committed, int32_t* n_commit, int32_t* near_tie, void* stream);

/*
 * Speculative sampling with a general draft distribution (review §3.1: the standard rule that
 * App. D specialises to the corrected draft's point mass).  draft [N, B] int32 are tokens drawn
 * from p [N, B, V] f32; q [N, B+1, V] f32 and u [N, B+1, 2] f32 as for STOCHASTIC.  Slot j is
 * accepted iff u[j,0] * p[j, draft[j]] < q[j, draft[j]] (float32 operands, product and
 * comparison in float64); at the first rejection j the committed token is the smallest v whose
 * running mass of max(0, q[j,v] - p[j,v]) (exact fixed point, vocabulary order) exceeds u[j,1] * R, R the
 * total (R <= 0 keeps draft[j]); if all B are accepted the bonus token is drawn from q[B] as for
 * STOCHASTIC.  A one-hot p at the draft token reproduces STOCHASTIC exactly.  Outputs and errors
 * as for dcoco_verify.
 */
int dcoco_verify_speculative(const int32_t* draft, const float* p, const float* q, const float* u, int N, int B, int V,
                             int32_t* accept_len, int32_t* committed, int32_t* n_commit, int32_t* near_tie,
                             void* stream);

/*
 * One whole correction cycle a1..a6: top-K, candidate representation, pair state,
 * transition scores, walk and verification, with intermediates in the workspace.  Inputs as
 * above; `t` (greedy) or `q`,`u` (stochastic) per `mode`.
 * Besides `stream`, the call uses two helper streams for the projections that need only h (g and
 * its fusion half; the pair states and W s): they fork from `stream` and join back into it through
 * events, so they overlap top-K.  By default these are two library-owned streams per device
 * (created on the first call, highest priority), shared by every host thread of the process; a
 * process-wide lock then serialises enqueueing, and cycles enqueued on different streams queue
 * behind one another on the helper streams.  dcoco_set_helper_streams gives a host thread its own
 * pair of helper streams (and its own events), with no lock.  The call can be captured into a CUDA
 * graph once the helper streams exist (after the first call, or with caller-owned streams).
 * Outputs (any may be NULL except tokens, accept_len, committed, n_commit):
 *   vals, ids [N,B,K]; S [N,B-1,K,K]; k_sel, tokens [N,B]; accept_len, n_commit [N];
 *   committed [N,B+1]; near_tie [N].
 */
size_t dcoco_cycle_workspace_size(const dcoco_weights* w, int N, int B, int K);
int dcoco_cycle(const void* logits, int V, const void* emb, const void* h, const dcoco_weights* w, int N, int B, int K,
                int mode, const int32_t* t, const float* q, const float* u, float* vals, int32_t* ids, float* S,
                int32_t* k_sel, int32_t* tokens, int32_t* accept_len, int32_t* committed, int32_t* n_commit,
                int32_t* near_tie, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Per-vocabulary candidate table (a builder-proposed variant; the pages have no counterpart):
 * Emb and W_e are frozen at inference, so b(v) = LN(W_e Emb[v]) can be computed once for every
 * token v.  table [V, r] in w->dtype (dcoco_embedding_table_bytes bytes), one tcgen05 GEMM with
 * the LayerNorm epilogue over Emb [V, E].  dcoco_cycle_table is dcoco_cycle with the rows
 * table[c] gathered in place of the per-cycle projection of Emb[c] (512 bytes instead of 2E per
 * candidate); same outputs, workspace and errors.
 */
size_t dcoco_embedding_table_bytes(const dcoco_weights* w, int V);
int dcoco_embedding_table(const void* emb, int V, const dcoco_weights* w, void* table, void* stream);
int dcoco_cycle_table(const void* logits, int V, const void* table, const void* h, const dcoco_weights* w, int N,
                      int B, int K, int mode, const int32_t* t, const float* q, const float* u, float* vals,
                      int32_t* ids, float* S, int32_t* k_sel, int32_t* tokens, int32_t* accept_len,
                      int32_t* committed, int32_t* n_commit, int32_t* near_tie, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Fused drafter output projection and top-K (Two Delta blog, "Score neighboring candidates in
 * parallel": the corrector reuses the drafter's own pass; its logits are that pass's projection
 * of the final hidden state onto the vocabulary).  For every row (n,i) of h [N, B, d] the
 * logits l[v] = sum_k h[n,i,k] W_lm[v,k], v in [0, V), are formed on the tensor cores (bf16
 * products or tf32 for f32 inputs, fp32 accumulation) and reduced to the K largest in the
 * same kernel; the [N, B, V] logits are never written.  W_lm [V, d] row-major (one row per
 * token), same dtype as h; d a multiple of 16 bytes' worth of elements; 1 <= K <= min(64, V).
 *   vals [N, B, K] float32  the kept fp32 logits, descending, equal values by ascending id
 *   ids  [N, B, K] int32
 * Workspace: dcoco_lm_head_topk_workspace_size bytes (per-row partial lists; the size depends
 * on the current device and dcoco_set_lm_pair), 16-byte aligned, caller-owned.
 * Selection is exact on the fp32 logits it computes and deterministic.  The fp32 logits differ
 * from exact dot products by accumulation rounding, so two tokens whose exact logits lie within
 * that rounding may rank in either order.
 */
size_t dcoco_lm_head_topk_workspace_size(int dtype, int N, int B, int V, int K);
int dcoco_lm_head_topk(const void* h, const void* W_lm, int dtype, int N, int B, int d, int V, int K, float* vals,
                       int32_t* ids, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Tuning knob: CTA-pair MMAs in dcoco_lm_head_topk for bf16 inputs (two CTAs of a cluster
 * issue one 256-row MMA together, each holding half of every W_lm tile).  0 = automatic
 * (pairs when h has at least two 128-row tiles), 1 = always, -1 = never (every CTA then loads
 * whole W_lm tiles and issues 128-row MMAs alone).  f32 inputs never use pairs.  Process-wide;
 * returns the previous value.  Query workspace sizes after setting it.
 */
int dcoco_set_lm_pair(int mode);

/*
 * dcoco_cycle starting from the drafter's hidden state instead of its logits: top-K is
 * dcoco_lm_head_topk of h with W_lm [V, d] (w->dtype), and the same h feeds the corrector.
 * Same outputs and errors as dcoco_cycle; workspace dcoco_cycle_lm_workspace_size bytes.
 */
size_t dcoco_cycle_lm_workspace_size(const dcoco_weights* w, int N, int B, int K, int V);
int dcoco_cycle_lm(const void* W_lm, int V, const void* emb, const void* h, const dcoco_weights* w, int N, int B,
                   int K, int mode, const int32_t* t, const float* q, const float* u, float* vals, int32_t* ids,
                   float* S, int32_t* k_sel, int32_t* tokens, int32_t* accept_len, int32_t* committed,
                   int32_t* n_commit, int32_t* near_tie, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DCOCO_H_ */
