// C ABI of the library: argument checking, workspace layout, tensor maps and launches.
// Every entry point validates all of its arguments before it enqueues anything.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/dcoco.h"
#include "internal.h"
#include "ptx.cuh"

namespace dcoco {
thread_local bool g_pdl = false;

int sm_count() {
  static std::atomic<int> sms[64];  // per device, 0 until first asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace dcoco

using namespace dcoco;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(DCOCO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}
void clear_err() { g_err[0] = '\0'; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Process-wide tuning knobs.  Each entry point reads a knob once and uses that one value for
// both its workspace check and its launch, so a concurrent change cannot split the two.
std::atomic<int> g_topk_split{0};  // 0 = automatic
std::atomic<int> g_lm_pair{0};     // 0 = automatic, 1 = always (bf16), -1 = never

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Bump allocator over the caller's workspace.
struct Carve {
  char* base;
  size_t used = 0;
  explicit Carve(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t bytes) {
    T* p = reinterpret_cast<T*>(base ? base + used : nullptr);
    used += round256(bytes);
    return p;
  }
};

int check_weights(const dcoco_weights* w) {
  if (w == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "weights is NULL");
  if (w->dtype != DCOCO_BF16 && w->dtype != DCOCO_F32) return fail(DCOCO_ERR_UNSUPPORTED, "weights dtype %d", w->dtype);
  if (w->d <= 0 || w->E <= 0 || w->r <= 0 || w->H <= 0)
    return fail(DCOCO_ERR_INVALID_ARG, "non-positive weight dims d=%d E=%d r=%d H=%d", w->d, w->E, w->r, w->H);
  const int r = w->r;
  if (r != 32 && r != 64 && r != 128 && r != 256 && r != 512)
    return fail(DCOCO_ERR_UNSUPPORTED, "corrector width r=%d (supported: 32, 64, 128, 256, 512)", r);
  if (w->H % 64 != 0) return fail(DCOCO_ERR_UNSUPPORTED, "MLP width H=%d is not a multiple of 64", w->H);
  if (w->d % 8 != 0 || w->E % 8 != 0)
    return fail(DCOCO_ERR_UNSUPPORTED, "d=%d and E=%d must be multiples of 8", w->d, w->E);
  const void* ptrs[] = {w->W_e, w->W_h, w->W_f, w->W_pair, w->U, w->V, w->W, w->u_a, w->u_b, w->b1, w->w2, w->b2};
  const char* names[] = {"W_e", "W_h", "W_f", "W_pair", "U", "V", "W", "u_a", "u_b", "b1", "w2", "b2"};
  for (int i = 0; i < 12; ++i) {
    if (ptrs[i] == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "weight %s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(DCOCO_ERR_INVALID_ARG, "weight %s is not 16-byte aligned", names[i]);
  }
  return DCOCO_OK;
}

int check_block(int N, int B, int K) {
  if (N < 1 || B < 2 || B > 64 || K < 1 || K > 64)
    return fail(DCOCO_ERR_INVALID_ARG, "shape N=%d B=%d K=%d outside N>=1, 2<=B<=64, 1<=K<=64", N, B, K);
  if (static_cast<int64_t>(N) * B > 65535 * 8 || static_cast<int64_t>(N) * (B - 1) > (1ll << 31) - 1)
    return fail(DCOCO_ERR_UNSUPPORTED, "too many streams N=%d", N);
  return DCOCO_OK;
}

int check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(DCOCO_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return DCOCO_OK;
}

// Logits may live in device memory or in page-locked host memory that is mapped into the
// device's address space (then top-K streams them once over the host link instead of after a
// bulk copy).  *dev receives the address kernels use; pageable host memory is rejected.
int resolve_readable(const void* p, const char* name, const void** dev) {
  cudaPointerAttributes at{};
  const cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return cuda_fail(e, name);
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *dev = p;
    return 0;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    *dev = at.devicePointer;
    return 0;
  }
  return fail(DCOCO_ERR_INVALID_ARG, "%s is neither device memory nor page-locked host memory mapped for the device", name);
}

#define DCOCO_TRY(x)             \
  do {                           \
    const int _rc = (x);         \
    if (_rc != DCOCO_OK) return _rc; \
  } while (0)

unsigned int* status_word(int* rc) {
  static unsigned int* words[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *rc = fail(DCOCO_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  if (words[dev] == nullptr) {
    cudaError_t e;
    unsigned int* p = device_status_word(&e);
    if (e != cudaSuccess) {
      *rc = cuda_fail(e, "cudaGetSymbolAddress(status word)");
      return nullptr;
    }
    words[dev] = p;
  }
  *rc = DCOCO_OK;
  return words[dev];
}

// N-tile width for an output group of width n (n a multiple of 64, or r in {32..512}).
int pick_bn(int n, bool allow512) {
  if (allow512 && n == 512) return 512;
  if (n % 256 == 0) return 256;
  if (n % 128 == 0) return 128;
  if (n % 64 == 0) return 64;
  return 32;
}


// Split-K factor for long reductions only (>= 16 K blocks): double it while the grid stays
// within max_ctas (the SM count by default) and every split keeps at least 8 K blocks.  Short
// reductions run whole.
int pick_split(int m_tiles, int n_tiles, int nkb, int BN, int max_ctas) {
  if (BN > 256 || nkb < 16) return 1;
  int s = 1;
  while (s < 8 && m_tiles * n_tiles * s * 2 <= max_ctas && nkb / (s * 2) >= 8) s *= 2;
  return s;
}

struct Dims {
  bool bf16;
  size_t esz;
  int N, B, K, d, E, r, H;
  int M() const { return N * B * K; }
  int NB() const { return N * B; }
  int NP() const { return N * (B - 1); }
};

Dims dims_of(const dcoco_weights* w, int N, int B, int K) {
  Dims D;
  D.bf16 = w->dtype == DCOCO_BF16;
  D.esz = D.bf16 ? 2 : 4;
  D.N = N;
  D.B = B;
  D.K = K;
  D.d = w->d;
  D.E = w->E;
  D.r = w->r;
  D.H = w->H;
  return D;
}

// ---------------------------------------------------------------- workspace layouts
struct ReprScratch {
  void* b;     // [M, r] act
  void* z;     // [M, r] act
  void* g;     // [NB, r] act
  float* gw;   // [NB, r]
};
size_t repr_scratch(const Dims& D, Carve& c, ReprScratch* s) {
  const size_t start = c.used;
  s->b = c.take<void>(static_cast<size_t>(D.M()) * D.r * D.esz);
  s->z = c.take<void>(static_cast<size_t>(D.M()) * D.r * D.esz);
  s->g = c.take<void>(static_cast<size_t>(D.NB()) * D.r * D.esz);
  s->gw = c.take<float>(static_cast<size_t>(D.NB()) * D.r * 4);
  return c.used - start;
}
struct PairScratch {
  float* hp;  // [NB, 2r]
  void* s;    // [NP, r] act
};
size_t pair_scratch(const Dims& D, Carve& c, PairScratch* s) {
  const size_t start = c.used;
  s->hp = c.take<float>(static_cast<size_t>(D.NB()) * 2 * D.r * 4);
  s->s = c.take<void>(static_cast<size_t>(D.NP()) * D.r * D.esz);
  return c.used - start;
}

// ---------------------------------------------------------------- GEMM helpers
// One output group: weight block [rows, cols] (pitch in elements) -> out [M, rows] (pitch ldo).
int gemm_group(GemmGroup* g, const void* w_base, const Dims& D, uint64_t rows, uint64_t cols, uint64_t pitch, int BN,
               void* out, int ldo, int epi, int M) {
  const char* err = nullptr;
  if (!make_tmap(&g->b_map, w_base, D.bf16, rows, cols, pitch, static_cast<uint32_t>(std::min(BN, 256)), &err))
    return fail(DCOCO_ERR_CUDA, "%s", err);
  const bool out_bf16 = D.bf16 && epi != EPI_F32;
  if (!make_tmap(&g->out_map, out, out_bf16, static_cast<uint64_t>(M), rows, static_cast<uint64_t>(ldo), 32, &err))
    return fail(DCOCO_ERR_CUDA, "%s", err);
  g->out = out;
  g->ldo = ldo;
  g->epi = epi;
  g->n_tiles = static_cast<int>(rows / BN);
  return DCOCO_OK;
}

// max_ctas bounds the split-K grid (0: the SM count), for GEMMs that share the GPU with another.
int run_gemm(GemmArgs& a, const Dims& D, int BN, cudaStream_t st, const char* what, int max_ctas = 0) {
  int rc;
  a.status = status_word(&rc);
  if (rc != DCOCO_OK) return rc;
  a.ln_eps = 1e-5f;
  const int m_tiles = (a.M + 127) / 128;
  int n_tiles = 0;
  bool prep = false;
  for (int i = 0; i < a.n_groups; ++i) {
    n_tiles += a.g[i].n_tiles;
    prep = prep || a.g[i].epi == EPI_PREP;
  }
  const int bk = D.bf16 ? 64 : 32;
  const int nkb = (a.K + bk - 1) / bk;
  const int split = prep ? 1 : pick_split(m_tiles, n_tiles, nkb, BN, max_ctas > 0 ? max_ctas : sm_count());
  const cudaError_t e = launch_gemm(a, D.bf16, BN, split, st);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DCOCO_OK;
}

int a_map_tiled(GemmArgs& a, const void* base, const Dims& D, uint64_t rows, uint64_t cols, uint64_t pitch) {
  const char* err = nullptr;
  if (!make_tmap(&a.a_map, base, D.bf16, rows, cols, pitch, 128, &err)) return fail(DCOCO_ERR_CUDA, "%s", err);
  a.gather = nullptr;
  return DCOCO_OK;
}

// Candidate representation, slot part (needs only h): g = LN(W_h h), gw = W_f[:, r:2r] g.
int enqueue_repr_slot(const Dims& D, const void* h, const dcoco_weights* w, const ReprScratch& s, cudaStream_t st,
                      int max_ctas = 0) {
  const int NB = D.NB(), r = D.r;
  // g = LN(W_h h)
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, h, D, NB, D.d, D.d));
    a.M = NB;
    a.K = D.d;
    a.n_groups = 1;
    const int BN = r;
    DCOCO_TRY(gemm_group(&a.g[0], w->W_h, D, r, D.d, D.d, BN, s.g, r, EPI_LN, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm g = LN(W_h h)", max_ctas));
  }
  // gw follows this library's own g GEMM: it may launch early
  PdlScope pdl_chain;
  // gw = W_f[:, r:2r] g   (the g half of the fusion, once per slot)
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, s.g, D, NB, r, r));
    a.M = NB;
    a.K = r;
    a.n_groups = 1;
    const int BN = pick_bn(r, false);
    DCOCO_TRY(gemm_group(&a.g[0], static_cast<const char*>(w->W_f) + r * D.esz, D, r, r, 2 * r, BN, s.gw, r, EPI_F32, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm gw = W_f,g g"));
  }
  return DCOCO_OK;
}

// Candidate representation, gather part: b = LN(W_e Emb[c]) (needs the ids).
int enqueue_repr_gather(const Dims& D, const int32_t* ids, const void* emb, int V, const dcoco_weights* w,
                        const ReprScratch& s, cudaStream_t st) {
  const int M = D.M(), r = D.r;
  // b = LN(W_e Emb[ids])   (gathered A operand)
  {
    GemmArgs a = {};
    const char* err = nullptr;
    if (!make_tmap(&a.a_map, emb, D.bf16, V, D.E, D.E, 1, &err)) return fail(DCOCO_ERR_CUDA, "%s", err);
    a.gather = ids;
    a.gather_limit = V;
    a.gather_base = emb;
    a.gather_pitch_bytes = static_cast<int>(D.E * D.esz);
    a.M = M;
    a.K = D.E;
    a.n_groups = 1;
    const int BN = pick_bn(r, true);
    if (BN != r) return fail(DCOCO_ERR_UNSUPPORTED, "r=%d", r);
    DCOCO_TRY(gemm_group(&a.g[0], w->W_e, D, r, D.E, D.E, BN, s.b, r, EPI_LN, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm b = LN(W_e Emb[c])"));
  }
  return DCOCO_OK;
}

// Candidate representation, fusion part: z = SiLU(W_f[:, 0:r] b + gw[slot]), uz = U z, vz = V z.
// With prep_vals set, the U z / V z epilogue writes the scorer's operands instead:
// uz <- (U z + b1 + W s + u_a l)/2 and vz <- (V z + u_b l)/2 (W s from prep_wsp).
// before_uv, when set, is an event the U z / V z GEMM waits for (the producer of prep_wsp).
// table, when set, replaces b: the A rows of the z GEMM are gathered as table[ids[m]] (V rows).
int enqueue_repr_fuse(const Dims& D, const dcoco_weights* w, void* uz, void* vz, const ReprScratch& s,
                      cudaStream_t st, const float* prep_vals = nullptr, const float* prep_wsp = nullptr,
                      cudaEvent_t before_uv = nullptr, const void* table = nullptr, const int32_t* ids = nullptr,
                      int V = 0) {
  const int M = D.M(), r = D.r, H = D.H;
  if (prep_vals != nullptr && table == nullptr && zuv_supported(D.bf16, r, H)) {
    // z and the scorer operands in one kernel: z stays on chip
    if (before_uv != nullptr) {
      const cudaError_t e = cudaStreamWaitEvent(st, before_uv, 0);
      if (e != cudaSuccess) return cuda_fail(e, "wait for W s");
    }
    ZuvArgs z = {};
    const char* err = nullptr;
    if (!make_tmap(&z.b_map, s.b, true, M, r, r, 128, &err) || !make_tmap(&z.wf_map, w->W_f, true, r, 2 * r, 2 * r, r, &err) ||
        !make_tmap(&z.u_map, w->U, true, H, r, r, std::min(H, 256), &err) ||
        !make_tmap(&z.v_map, w->V, true, H, r, r, std::min(H, 256), &err) ||
        !make_tmap(&z.p_map, uz, true, M, H, H, 32, &err) || !make_tmap(&z.q_map, vz, true, M, H, H, 32, &err))
      return fail(DCOCO_ERR_CUDA, "%s", err);
    z.p = uz;
    z.q = vz;
    z.gw = s.gw;
    z.wsp = prep_wsp;
    z.vals = prep_vals;
    z.b1 = w->b1;
    z.u_a = w->u_a;
    z.u_b = w->u_b;
    z.M = M;
    z.r = r;
    z.H = H;
    z.cand = D.K;
    z.slots = D.B;
    int rc;
    z.status = status_word(&rc);
    if (rc != DCOCO_OK) return rc;
    const cudaError_t e = launch_zuv(z, st);
    if (e != cudaSuccess) return cuda_fail(e, "fused z, U z / V z");
    return DCOCO_OK;
  }
  // z = SiLU(W_f[:, 0:r] b + gw[slot])
  {
    GemmArgs a = {};
    if (table != nullptr) {
      const char* err = nullptr;
      if (!make_tmap(&a.a_map, table, D.bf16, V, r, r, 1, &err)) return fail(DCOCO_ERR_CUDA, "%s", err);
      a.gather = ids;
      a.gather_limit = V;
      a.gather_base = table;
      a.gather_pitch_bytes = static_cast<int>(r * D.esz);
    } else {
      DCOCO_TRY(a_map_tiled(a, s.b, D, M, r, r));
    }
    a.M = M;
    a.K = r;
    a.n_groups = 1;
    a.bias = s.gw;
    a.bias_div = D.K;
    a.ld_bias = r;
    // narrower tiles while the grid would cover less than half of the SMs
    int BN = pick_bn(r, false);
    const int m_tiles = (M + 127) / 128;
    while (BN > 64 && m_tiles * (r / BN) * 2 <= sm_count()) BN /= 2;
    DCOCO_TRY(gemm_group(&a.g[0], w->W_f, D, r, r, 2 * r, BN, s.z, r, EPI_SILU_BIAS, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm z = SiLU(W_f [b; g])"));
  }
  if (before_uv != nullptr) {
    const cudaError_t e = cudaStreamWaitEvent(st, before_uv, 0);
    if (e != cudaSuccess) return cuda_fail(e, "wait for W s");
  }
  // uz = U z, vz = V z
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, s.z, D, M, r, r));
    a.M = M;
    a.K = r;
    a.n_groups = 2;
    // 512-wide tiles when 256-wide ones would need more than one wave of CTAs
    const int m_tiles = (M + 127) / 128;
    const int BN = (H % 512 == 0 && m_tiles * (2 * H / 256) > sm_count()) ? 512 : pick_bn(H, false);
    const int epi = prep_vals != nullptr ? EPI_PREP : EPI_ACT;
    DCOCO_TRY(gemm_group(&a.g[0], w->U, D, H, r, r, BN, uz, H, epi, a.M));
    DCOCO_TRY(gemm_group(&a.g[1], w->V, D, H, r, r, BN, vz, H, epi, a.M));
    if (prep_vals != nullptr) {
      a.row_l = prep_vals;
      a.bias_div = D.K;
      a.slots = D.B;
      a.ld_bias = H;
      a.g[0].col_u = w->u_a;
      a.g[0].col_b = w->b1;
      a.g[0].row_bias = prep_wsp;
      a.g[1].col_u = w->u_b;
    }
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm uz, vz"));
  }
  return DCOCO_OK;
}

int enqueue_repr(const Dims& D, const int32_t* ids, const void* emb, int V, const void* h, const dcoco_weights* w,
                 void* uz, void* vz, const ReprScratch& s, cudaStream_t st) {
  DCOCO_TRY(enqueue_repr_gather(D, ids, emb, V, w, s, st));
  DCOCO_TRY(enqueue_repr_slot(D, h, w, s, st));
  return enqueue_repr_fuse(D, w, uz, vz, s, st);
}

// CTAs of the embedding-row GEMM b = LN(W_e Emb[c]) (the same choices enqueue_repr_gather makes).
int gather_gemm_ctas(const Dims& D) {
  const int m_tiles = (D.M() + 127) / 128;
  const int BN = pick_bn(D.r, true);
  const int n_tiles = D.r / BN;
  const int nkb = (D.E + (D.bf16 ? 64 : 32) - 1) / (D.bf16 ? 64 : 32);
  return m_tiles * n_tiles * pick_split(m_tiles, n_tiles, nkb, BN, sm_count());
}

// Per-device helper streams (highest priority) and fork/join events for dcoco_cycle; the
// mutex keeps one enqueue sequence at a time per process.
struct SideStream {
  cudaStream_t stream = nullptr, stream2 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
};
int make_events(SideStream& s) {
  cudaError_t e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join2, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "helper event set-up");
  return DCOCO_OK;
}
// Library-owned helper streams (highest priority) and events, one set per device, shared by
// every host thread: g_side_mu keeps one enqueue sequence at a time on them.
std::mutex g_side_mu;
int side_stream(SideStream** out) {
  static SideStream per_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(DCOCO_ERR_CUDA, "no current CUDA device");
  SideStream& s = per_dev[dev];
  if (s.stream == nullptr) {
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&s.stream2, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return cuda_fail(e, "helper stream set-up");
    DCOCO_TRY(make_events(s));
  }
  *out = &s;
  return DCOCO_OK;
}
// Caller-owned helper streams of this host thread (dcoco_set_helper_streams) and this thread's
// own fork/join events, one set per device.
thread_local cudaStream_t t_helper[2] = {nullptr, nullptr};
struct ThreadEvents {
  SideStream dev[64];
  ~ThreadEvents() {
    for (SideStream& s : dev)
      for (cudaEvent_t ev : {s.fork, s.join, s.join2})
        if (ev != nullptr) (void)cudaEventDestroy(ev);
  }
};
thread_local ThreadEvents t_events;
int caller_side_stream(SideStream** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(DCOCO_ERR_CUDA, "no current CUDA device");
  SideStream& s = t_events.dev[dev];
  if (s.fork == nullptr) DCOCO_TRY(make_events(s));
  s.stream = t_helper[0];
  s.stream2 = t_helper[1];
  *out = &s;
  return DCOCO_OK;
}

int enqueue_pair(const Dims& D, const void* h, const dcoco_weights* w, float* wsp, const PairScratch& s,
                 cudaStream_t st, int max_ctas = 0) {
  const int NB = D.NB(), r = D.r, H = D.H, d = D.d;
  // hp[:, 0:r] = W_pair[:, 0:d] h,  hp[:, r:2r] = W_pair[:, d:2d] h   (every slot once)
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, h, D, NB, d, d));
    a.M = NB;
    a.K = d;
    a.n_groups = 2;
    const int BN = pick_bn(r, false);
    DCOCO_TRY(gemm_group(&a.g[0], w->W_pair, D, r, d, 2 * d, BN, s.hp, 2 * r, EPI_F32, a.M));
    DCOCO_TRY(gemm_group(&a.g[1], static_cast<const char*>(w->W_pair) + d * D.esz, D, r, d, 2 * d, BN, s.hp + r,
                         2 * r, EPI_F32, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm W_pair h", max_ctas));
  }
  // the rest of the chain follows this library's own kernels: each may launch early
  PdlScope pdl_chain;
  // s_p = hp[p, 0:r] + hp[p+1, r:2r]
  {
    const cudaError_t e = launch_pair_combine(s.hp, s.s, D.bf16, D.N, D.B, r, st);
    if (e != cudaSuccess) return cuda_fail(e, "pair combine");
  }
  // wsp = W s_p
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, s.s, D, D.NP(), r, r));
    a.M = D.NP();
    a.K = r;
    a.n_groups = 1;
    const int BN = pick_bn(H, false);
    DCOCO_TRY(gemm_group(&a.g[0], w->W, D, H, r, r, BN, wsp, H, EPI_F32, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st, "gemm W s"));
  }
  return DCOCO_OK;
}

// The cycle's projections that need only h, as one GEMM over h with three output groups:
// g = LN(W_h h) and the two halves of W_pair applied to every slot (hp).  It lets the next
// kernel of the stream (top-K, which does not read its outputs) launch as soon as it starts.
int enqueue_hproj(const Dims& D, const void* h, const dcoco_weights* w, const ReprScratch& rs, const PairScratch& ps,
                  cudaStream_t st, int max_ctas) {
  const int NB = D.NB(), r = D.r, d = D.d;
  GemmArgs a = {};
  DCOCO_TRY(a_map_tiled(a, h, D, NB, d, d));
  a.M = NB;
  a.K = d;
  a.n_groups = 3;
  a.early_dependents = 1;
  const int BN = pick_bn(r, true);  // the LayerNorm group needs its whole row in one tile
  if (BN != r) return fail(DCOCO_ERR_UNSUPPORTED, "r=%d", r);
  DCOCO_TRY(gemm_group(&a.g[0], w->W_h, D, r, d, d, BN, rs.g, r, EPI_LN, a.M));
  DCOCO_TRY(gemm_group(&a.g[1], w->W_pair, D, r, d, 2 * d, BN, ps.hp, 2 * r, EPI_F32, a.M));
  DCOCO_TRY(gemm_group(&a.g[2], static_cast<const char*>(w->W_pair) + d * D.esz, D, r, d, 2 * d, BN, ps.hp + r, 2 * r,
                       EPI_F32, a.M));
  return run_gemm(a, D, BN, st, "gemm g = LN(W_h h), W_pair h", max_ctas);
}

// The rest of the h-only work after enqueue_hproj, on two streams: s_p = hp[p, 0:r] +
// hp[p+1, r:2r] and W s_p on st_pair; the g half of the fusion gw = W_f[:, r:2r] g on st_slot.
int enqueue_h_tail(const Dims& D, const dcoco_weights* w, float* wsp, const ReprScratch& rs, const PairScratch& ps,
                   cudaStream_t st_pair, cudaStream_t st_slot) {
  const int r = D.r, H = D.H;
  {
    const cudaError_t e = launch_pair_combine(ps.hp, ps.s, D.bf16, D.N, D.B, r, st_pair);
    if (e != cudaSuccess) return cuda_fail(e, "pair combine");
  }
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, rs.g, D, D.NB(), r, r));
    a.M = D.NB();
    a.K = r;
    a.n_groups = 1;
    const int BN = pick_bn(r, false);
    DCOCO_TRY(gemm_group(&a.g[0], static_cast<const char*>(w->W_f) + r * D.esz, D, r, r, 2 * r, BN, rs.gw, r, EPI_F32,
                         a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st_slot, "gemm gw = W_f,g g"));
  }
  PdlScope pdl_chain;  // W s follows this library's own pair-combine kernel
  {
    GemmArgs a = {};
    DCOCO_TRY(a_map_tiled(a, ps.s, D, D.NP(), r, r));
    a.M = D.NP();
    a.K = r;
    a.n_groups = 1;
    const int BN = pick_bn(H, false);
    DCOCO_TRY(gemm_group(&a.g[0], w->W, D, H, r, r, BN, wsp, H, EPI_F32, a.M));
    DCOCO_TRY(run_gemm(a, D, BN, st_pair, "gemm W s"));
  }
  return DCOCO_OK;
}

int enqueue_scores(const Dims& D, const void* uz, const void* vz, const float* wsp, const float* vals,
                   const dcoco_weights* w, float* S, cudaStream_t st) {
  ScoreArgs a;
  a.uz = uz;
  a.vz = vz;
  a.wsp = wsp;
  a.vals = vals;
  a.u_a = w->u_a;
  a.u_b = w->u_b;
  a.b1 = w->b1;
  a.w2 = w->w2;
  a.b2 = w->b2;
  a.S = S;
  a.N = D.N;
  a.B = D.B;
  a.K = D.K;
  a.H = D.H;
  const cudaError_t e = launch_scores(a, D.bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "transition scores");
  return DCOCO_OK;
}

int enqueue_scores_prepped(const Dims& D, const void* P, const void* Q, const float* vals, const dcoco_weights* w,
                           float* S, cudaStream_t st) {
  ScoreArgs a = {};
  a.uz = P;
  a.vz = Q;
  a.vals = vals;
  a.w2 = w->w2;
  a.b2 = w->b2;
  a.S = S;
  a.N = D.N;
  a.B = D.B;
  a.K = D.K;
  a.H = D.H;
  const cudaError_t e = launch_scores_prepped(a, D.bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "transition scores");
  return DCOCO_OK;
}

// 0 lets the top-K launcher choose the split from the device's occupancy.
int topk_split(int, int, bool) { return g_topk_split.load(); }

}  // namespace

extern "C" {

int dcoco_version(void) { return 100; }

const char* dcoco_last_error(void) { return g_err; }

int dcoco_set_helper_streams(void* helper_a, void* helper_b) {
  clear_err();
  if ((helper_a == nullptr) != (helper_b == nullptr))
    return fail(DCOCO_ERR_INVALID_ARG, "helper streams: pass two streams or two NULLs");
  if (helper_a != nullptr && helper_a == helper_b)
    return fail(DCOCO_ERR_INVALID_ARG, "helper streams: the two streams must differ");
  t_helper[0] = as_stream(helper_a);
  t_helper[1] = as_stream(helper_b);
  return DCOCO_OK;
}

int dcoco_set_topk_split(int ctas_per_row) {
  return g_topk_split.exchange(std::max(0, std::min(8, ctas_per_row)));
}

int dcoco_set_lm_pair(int mode) { return g_lm_pair.exchange(mode > 0 ? 1 : mode < 0 ? -1 : 0); }

}  // extern "C"

namespace {
// One warp: lane 0 waits on an mbarrier that nothing arrives at, with the same bounded wait the
// library's pipelines use but at most `polls` polls, records the TMA-wait timeout bit the way a
// producer whose copy never lands would, and invalidates the barrier.  No copy is in flight.
__global__ void wait_timeout_kernel(uint32_t polls, unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait_n(smem_u32(&bar), 0, polls)) atomicOr(status, DEV_TIMEOUT_TMA);
    mbar_inval(smem_u32(&bar));
  }
  __syncwarp();
}
}  // namespace

extern "C" {

int dcoco_selftest_timeout(uint32_t polls, void* stream) {
  clear_err();
  if (polls < 1 || polls > 65536) return fail(DCOCO_ERR_INVALID_ARG, "polls=%u outside [1, 65536]", polls);
  int rc;
  unsigned int* w = status_word(&rc);
  if (rc != DCOCO_OK) return rc;
  wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>(polls, w);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return DCOCO_OK;
}

int dcoco_device_status(void* stream, uint32_t* bits) {
  clear_err();
  int rc;
  unsigned int* w = status_word(&rc);
  if (rc != DCOCO_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  e = cudaMemset(w, 0, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "clear status word");
  if (bits) *bits = v;
  if (v & 7u) return fail(DCOCO_ERR_TIMEOUT, "device status 0x%x: a bounded wait gave up", v);
  return DCOCO_OK;
}

int dcoco_topk(const void* logits, int dtype, int N, int B, int V, int K, float* vals, int32_t* ids, void* stream) {
  clear_err();
  if (dtype != DCOCO_BF16 && dtype != DCOCO_F32) return fail(DCOCO_ERR_UNSUPPORTED, "logits dtype %d", dtype);
  if (N < 1 || B < 1 || V < 1 || K < 1 || K > 64 || K > V)
    return fail(DCOCO_ERR_INVALID_ARG, "shape N=%d B=%d V=%d K=%d (need 1<=K<=min(64,V))", N, B, V, K);
  if (static_cast<int64_t>(N) * B > 65535) return fail(DCOCO_ERR_UNSUPPORTED, "N*B=%lld rows > 65535", (long long)N * B);
  DCOCO_TRY(check_ptr(logits, "logits"));
  DCOCO_TRY(check_ptr(vals, "vals"));
  DCOCO_TRY(check_ptr(ids, "ids"));
  DCOCO_TRY(resolve_readable(logits, "logits", &logits));
  const bool bf16 = dtype == DCOCO_BF16;
  const int rows = N * B;
  const cudaError_t e = launch_topk(logits, bf16, rows, V, K, topk_split(rows, V, bf16), vals, ids, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-K launch");
  return DCOCO_OK;
}

size_t dcoco_lm_head_topk_workspace_size(int dtype, int N, int B, int V, int K) {
  if ((dtype != DCOCO_BF16 && dtype != DCOCO_F32) || N < 1 || B < 1 || V < 1 || K < 1 || K > 64 || K > V ||
      static_cast<int64_t>(N) * B > 65535)
    return 0;
  return lm_topk_partial_bytes(dtype == DCOCO_BF16, N * B, V, K, g_lm_pair.load());
}

int dcoco_lm_head_topk(const void* h, const void* W_lm, int dtype, int N, int B, int d, int V, int K, float* vals,
                       int32_t* ids, void* workspace, size_t workspace_bytes, void* stream) {
  clear_err();
  if (dtype != DCOCO_BF16 && dtype != DCOCO_F32) return fail(DCOCO_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (N < 1 || B < 1 || V < 1 || K < 1 || K > 64 || K > V || d < 1)
    return fail(DCOCO_ERR_INVALID_ARG, "shape N=%d B=%d d=%d V=%d K=%d (need 1<=K<=min(64,V))", N, B, d, V, K);
  if (static_cast<int64_t>(N) * B > 65535) return fail(DCOCO_ERR_UNSUPPORTED, "N*B=%lld rows > 65535", (long long)N * B);
  const bool bf16 = dtype == DCOCO_BF16;
  if ((static_cast<size_t>(d) * (bf16 ? 2 : 4)) % 16 != 0)
    return fail(DCOCO_ERR_INVALID_ARG, "d=%d: rows of h and W_lm must be a multiple of 16 bytes", d);
  DCOCO_TRY(check_ptr(h, "h"));
  DCOCO_TRY(check_ptr(W_lm, "W_lm"));
  DCOCO_TRY(check_ptr(vals, "vals"));
  DCOCO_TRY(check_ptr(ids, "ids"));
  const int pair_mode = g_lm_pair.load();
  const size_t need = lm_topk_partial_bytes(bf16, N * B, V, K, pair_mode);
  if (need == 0) return fail(DCOCO_ERR_CUDA, "no launch plan for the fused LM-head top-K on this device");
  if (workspace == nullptr || workspace_bytes < need)
    return fail(DCOCO_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(DCOCO_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  int rc;
  unsigned int* status = status_word(&rc);
  if (rc != DCOCO_OK) return rc;
  const cudaError_t e = launch_lm_topk(h, W_lm, bf16, N * B, d, V, K, pair_mode, vals, ids, workspace,
                                       workspace_bytes, status, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "LM-head top-K launch");
  return DCOCO_OK;
}

size_t dcoco_candidate_repr_workspace_size(const dcoco_weights* w, int N, int B, int K) {
  if (w == nullptr || N < 1 || B < 1 || K < 1) return 0;
  Carve c(nullptr);
  ReprScratch s;
  repr_scratch(dims_of(w, N, B, K), c, &s);
  return c.used;
}

int dcoco_candidate_repr(const int32_t* ids, const void* emb, int V, const void* h, const dcoco_weights* w, int N,
                         int B, int K, void* uz, void* vz, void* workspace, size_t workspace_bytes, void* stream) {
  clear_err();
  DCOCO_TRY(check_weights(w));
  DCOCO_TRY(check_block(N, B, K));
  if (V < K) return fail(DCOCO_ERR_INVALID_ARG, "V=%d < K=%d", V, K);
  DCOCO_TRY(check_ptr(ids, "ids"));
  DCOCO_TRY(check_ptr(emb, "emb"));
  DCOCO_TRY(check_ptr(h, "h"));
  DCOCO_TRY(check_ptr(uz, "uz"));
  DCOCO_TRY(check_ptr(vz, "vz"));
  const Dims D = dims_of(w, N, B, K);
  const size_t need = dcoco_candidate_repr_workspace_size(w, N, B, K);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(DCOCO_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(DCOCO_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  Carve c(workspace);
  ReprScratch s;
  repr_scratch(D, c, &s);
  return enqueue_repr(D, ids, emb, V, h, w, uz, vz, s, as_stream(stream));
}

size_t dcoco_pair_state_workspace_size(const dcoco_weights* w, int N, int B) {
  if (w == nullptr || N < 1 || B < 2) return 0;
  Carve c(nullptr);
  PairScratch s;
  pair_scratch(dims_of(w, N, B, 1), c, &s);
  return c.used;
}

int dcoco_pair_state(const void* h, const dcoco_weights* w, int N, int B, float* ws_pair, void* workspace,
                     size_t workspace_bytes, void* stream) {
  clear_err();
  DCOCO_TRY(check_weights(w));
  DCOCO_TRY(check_block(N, B, 1));
  DCOCO_TRY(check_ptr(h, "h"));
  DCOCO_TRY(check_ptr(ws_pair, "ws_pair"));
  const Dims D = dims_of(w, N, B, 1);
  const size_t need = dcoco_pair_state_workspace_size(w, N, B);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(DCOCO_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(DCOCO_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  Carve c(workspace);
  PairScratch s;
  pair_scratch(D, c, &s);
  return enqueue_pair(D, h, w, ws_pair, s, as_stream(stream));
}

int dcoco_score_transitions(const void* uz, const void* vz, const float* ws_pair, const float* vals,
                            const dcoco_weights* w, int N, int B, int K, float* S, void* stream) {
  clear_err();
  DCOCO_TRY(check_weights(w));
  DCOCO_TRY(check_block(N, B, K));
  DCOCO_TRY(check_ptr(uz, "uz"));
  DCOCO_TRY(check_ptr(vz, "vz"));
  DCOCO_TRY(check_ptr(ws_pair, "ws_pair"));
  DCOCO_TRY(check_ptr(vals, "vals"));
  DCOCO_TRY(check_ptr(S, "S"));
  return enqueue_scores(dims_of(w, N, B, K), uz, vz, ws_pair, vals, w, S, as_stream(stream));
}

int dcoco_select(const float* S, const float* vals, const int32_t* ids, int N, int B, int K, int32_t* k_sel,
                 int32_t* tokens, void* stream) {
  clear_err();
  DCOCO_TRY(check_block(N, B, K));
  DCOCO_TRY(check_ptr(S, "S"));
  DCOCO_TRY(check_ptr(vals, "vals"));
  DCOCO_TRY(check_ptr(ids, "ids"));
  DCOCO_TRY(check_ptr(k_sel, "k_sel"));
  DCOCO_TRY(check_ptr(tokens, "tokens"));
  SelectVerifyArgs a = {};
  a.S = S;
  a.vals = vals;
  a.ids = ids;
  a.k_sel = k_sel;
  a.tokens = tokens;
  a.mode = -1;
  a.N = N;
  a.B = B;
  a.K = K;
  a.V = 0;
  const cudaError_t e = launch_select_verify(a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return DCOCO_OK;
}

int dcoco_select_path(const float* S, const float* vals, const int32_t* ids, int N, int B, int K, int rule,
                      float lambda, int32_t* k_sel, int32_t* tokens, void* stream) {
  clear_err();
  if (rule != DCOCO_PATH_GREEDY && rule != DCOCO_PATH_DISCOUNTED) return fail(DCOCO_ERR_INVALID_ARG, "path rule %d", rule);
  if (rule == DCOCO_PATH_DISCOUNTED && !(lambda > 0.f && lambda <= 1.f))
    return fail(DCOCO_ERR_INVALID_ARG, "discount lambda=%g outside (0, 1]", static_cast<double>(lambda));
  DCOCO_TRY(check_block(N, B, K));
  DCOCO_TRY(check_ptr(S, "S"));
  DCOCO_TRY(check_ptr(vals, "vals"));
  DCOCO_TRY(check_ptr(ids, "ids"));
  DCOCO_TRY(check_ptr(k_sel, "k_sel"));
  DCOCO_TRY(check_ptr(tokens, "tokens"));
  SelectVerifyArgs a = {};
  a.S = S;
  a.vals = vals;
  a.ids = ids;
  a.k_sel = k_sel;
  a.tokens = tokens;
  a.rule = rule;
  a.lam = lambda;
  a.mode = -1;
  a.N = N;
  a.B = B;
  a.K = K;
  a.V = 0;
  const cudaError_t e = launch_select_verify(a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return DCOCO_OK;
}

static int check_verify(int mode, const int32_t* draft, const int32_t* t, const float* q, const float* u, int N, int B,
                        int V, int32_t* accept_len, int32_t* committed, int32_t* n_commit, bool need_draft) {
  if (mode != DCOCO_VERIFY_GREEDY && mode != DCOCO_VERIFY_STOCHASTIC)
    return fail(DCOCO_ERR_INVALID_ARG, "verify mode %d", mode);
  if (N < 1 || B < 1 || B > 64) return fail(DCOCO_ERR_INVALID_ARG, "shape N=%d B=%d (need 1<=B<=64)", N, B);
  if (need_draft) DCOCO_TRY(check_ptr(draft, "draft"));
  if (mode == DCOCO_VERIFY_GREEDY) {
    DCOCO_TRY(check_ptr(t, "t"));
  } else {
    if (V < 1) return fail(DCOCO_ERR_INVALID_ARG, "V=%d", V);
    DCOCO_TRY(check_ptr(q, "q"));
    DCOCO_TRY(check_ptr(u, "u"));
  }
  DCOCO_TRY(check_ptr(accept_len, "accept_len"));
  DCOCO_TRY(check_ptr(committed, "committed"));
  DCOCO_TRY(check_ptr(n_commit, "n_commit"));
  return DCOCO_OK;
}

int dcoco_verify(int mode, const int32_t* draft, const int32_t* t, const float* q, const float* u, int N, int B, int V,
                 int32_t* accept_len, int32_t* committed, int32_t* n_commit, int32_t* near_tie, void* stream) {
  clear_err();
  DCOCO_TRY(check_verify(mode, draft, t, q, u, N, B, V, accept_len, committed, n_commit, true));
  SelectVerifyArgs a = {};
  a.mode = mode;
  a.draft = draft;
  a.t = t;
  a.q = q;
  a.u = u;
  a.accept_len = accept_len;
  a.committed = committed;
  a.n_commit = n_commit;
  a.near_tie = near_tie;
  a.N = N;
  a.B = B;
  a.K = 1;
  a.V = V;
  const cudaError_t e = launch_select_verify(a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return DCOCO_OK;
}

int dcoco_verify_speculative(const int32_t* draft, const float* p, const float* q, const float* u, int N, int B, int V,
                             int32_t* accept_len, int32_t* committed, int32_t* n_commit, int32_t* near_tie,
                             void* stream) {
  clear_err();
  DCOCO_TRY(check_verify(DCOCO_VERIFY_STOCHASTIC, draft, nullptr, q, u, N, B, V, accept_len, committed, n_commit, true));
  DCOCO_TRY(check_ptr(p, "p"));
  SelectVerifyArgs a = {};
  a.mode = 2;
  a.draft = draft;
  a.p = p;
  a.q = q;
  a.u = u;
  a.accept_len = accept_len;
  a.committed = committed;
  a.n_commit = n_commit;
  a.near_tie = near_tie;
  a.N = N;
  a.B = B;
  a.K = 1;
  a.V = V;
  const cudaError_t e = launch_select_verify(a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return DCOCO_OK;
}

namespace {
struct CycleScratch {
  float* vals;
  int32_t* ids;
  float* S;
  int32_t* k_sel;
  void* uz;
  void* vz;
  float* wsp;
  ReprScratch repr;
  PairScratch pair;
};
size_t cycle_scratch(const Dims& D, Carve& c, CycleScratch* s) {
  const size_t start = c.used;
  const size_t M = static_cast<size_t>(D.M());
  s->vals = c.take<float>(M * 4);
  s->ids = c.take<int32_t>(M * 4);
  s->S = c.take<float>(static_cast<size_t>(D.NP()) * D.K * D.K * 4);
  s->k_sel = c.take<int32_t>(static_cast<size_t>(D.NB()) * 4);
  s->uz = c.take<void>(M * D.H * D.esz);
  s->vz = c.take<void>(M * D.H * D.esz);
  s->wsp = c.take<float>(static_cast<size_t>(D.NP()) * D.H * 4);
  repr_scratch(D, c, &s->repr);
  pair_scratch(D, c, &s->pair);
  return c.used - start;
}
}  // namespace

size_t dcoco_cycle_workspace_size(const dcoco_weights* w, int N, int B, int K) {
  if (w == nullptr || N < 1 || B < 2 || K < 1) return 0;
  Carve c(nullptr);
  CycleScratch s;
  cycle_scratch(dims_of(w, N, B, K), c, &s);
  return c.used;
}

}  // extern "C"

namespace {
// One cycle; exactly one of emb (gathered and projected every cycle) and table (rows of
// LN(W_e Emb) precomputed by dcoco_embedding_table) is set.
int cycle_impl(const void* logits, const void* W_lm, int V, const void* emb, const void* table, const void* h,
               const dcoco_weights* w, int N, int B, int K, int mode, const int32_t* t, const float* q, const float* u, float* vals,
               int32_t* ids, float* S, int32_t* k_sel, int32_t* tokens, int32_t* accept_len, int32_t* committed,
               int32_t* n_commit, int32_t* near_tie, void* workspace, size_t workspace_bytes, void* stream) {
  DCOCO_TRY(check_weights(w));
  DCOCO_TRY(check_block(N, B, K));
  if (V < K) return fail(DCOCO_ERR_INVALID_ARG, "V=%d < K=%d", V, K);
  if (static_cast<int64_t>(N) * B > 65535) return fail(DCOCO_ERR_UNSUPPORTED, "N*B > 65535");
  DCOCO_TRY(check_ptr(W_lm != nullptr ? W_lm : logits, W_lm != nullptr ? "W_lm" : "logits"));
  DCOCO_TRY(check_ptr(emb != nullptr ? emb : table, emb != nullptr ? "emb" : "table"));
  DCOCO_TRY(check_ptr(h, "h"));
  DCOCO_TRY(check_ptr(tokens, "tokens"));
  DCOCO_TRY(check_verify(mode, nullptr, t, q, u, N, B, V, accept_len, committed, n_commit, false));
  const float* opt[] = {vals, S};
  for (const float* p : opt)
    if (p && !aligned16(p)) return fail(DCOCO_ERR_INVALID_ARG, "an optional output is not 16-byte aligned");
  if ((ids && !aligned16(ids)) || (k_sel && !aligned16(k_sel)))
    return fail(DCOCO_ERR_INVALID_ARG, "an optional output is not 16-byte aligned");
  const Dims D = dims_of(w, N, B, K);
  const size_t base_need = dcoco_cycle_workspace_size(w, N, B, K);
  size_t lm_bytes = 0;
  const int pair_mode = g_lm_pair.load();
  if (W_lm != nullptr) {
    if ((static_cast<size_t>(D.d) * D.esz) % 16 != 0)
      return fail(DCOCO_ERR_INVALID_ARG, "d=%d: rows of h and W_lm must be a multiple of 16 bytes", D.d);
    lm_bytes = lm_topk_partial_bytes(D.bf16, N * B, V, K, pair_mode);
    if (lm_bytes == 0) return fail(DCOCO_ERR_CUDA, "no launch plan for the fused LM-head top-K on this device");
  }
  const size_t need = base_need + round256(lm_bytes);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(DCOCO_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(DCOCO_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  Carve c(workspace);
  CycleScratch s;
  cycle_scratch(D, c, &s);
  void* lm_partial = W_lm != nullptr ? c.take<void>(lm_bytes) : nullptr;
  float* o_vals = vals ? vals : s.vals;
  int32_t* o_ids = ids ? ids : s.ids;
  float* o_S = S ? S : s.S;
  int32_t* o_k = k_sel ? k_sel : s.k_sel;
  cudaStream_t st = as_stream(stream);

  const int rows = N * B;
  if (W_lm == nullptr) DCOCO_TRY(resolve_readable(logits, "logits", &logits));
  // the library's shared helper streams are used by one enqueue sequence at a time; a thread's
  // own helper streams need no lock
  std::unique_lock<std::mutex> lock(g_side_mu, std::defer_lock);
  SideStream* side = nullptr;
  if (t_helper[0] != nullptr) {
    DCOCO_TRY(caller_side_stream(&side));
  } else {
    lock.lock();
    DCOCO_TRY(side_stream(&side));
  }
  cudaError_t e;
  if (W_lm != nullptr) {
    // The fused LM-head kernel is persistent over every SM: the h-only work forks after it and
    // runs beside the embedding-row GEMM, on the SMs that GEMM leaves free.
    int rc;
    unsigned int* status = status_word(&rc);
    if (rc != DCOCO_OK) return rc;
    e = launch_lm_topk(h, W_lm, D.bf16, rows, D.d, V, K, pair_mode, o_vals, o_ids, lm_partial, lm_bytes, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-K launch");
    const int spare = std::max(12, sm_count() - gather_gemm_ctas(D));
    const int pair_ctas = spare * 2 / 3, slot_ctas = spare - pair_ctas;
    e = cudaEventRecord(side->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream2, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "fork to helper streams");
    DCOCO_TRY(enqueue_pair(D, h, w, s.wsp, s.pair, side->stream, pair_ctas));
    DCOCO_TRY(enqueue_repr_slot(D, h, w, s.repr, side->stream2, slot_ctas));
    e = cudaEventRecord(side->join, side->stream);
    if (e == cudaSuccess) e = cudaEventRecord(side->join2, side->stream2);
    if (e != cudaSuccess) return cuda_fail(e, "join from helper streams");
  } else {
    // The projections that need only h run first, as one GEMM on the SMs top-K leaves free
    // (top-K holds at most four blocks per SM); top-K launches programmatically behind it, as
    // soon as its CTAs have started, without waiting for it.  The tail of the h-only chain (pair
    // sums, W s, the g half of the fusion) runs on a helper stream once that GEMM is done, on
    // the SMs it frees, while top-K still streams the logits.
    const int topk_sms = (rows * topk_ctas_per_row(rows, V, D.bf16, topk_split(rows, V, D.bf16)) + 3) / 4;
    const int spare = std::max(12, sm_count() - topk_sms);
    DCOCO_TRY(enqueue_hproj(D, h, w, s.repr, s.pair, st, spare));
    e = cudaEventRecord(side->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream2, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "fork to helper streams");
    e = launch_topk(logits, D.bf16, rows, V, K, topk_split(rows, V, D.bf16), o_vals, o_ids, st, true);
    if (e != cudaSuccess) return cuda_fail(e, "top-K launch");
    DCOCO_TRY(enqueue_h_tail(D, w, s.wsp, s.repr, s.pair, side->stream, side->stream2));
    e = cudaEventRecord(side->join, side->stream);
    if (e == cudaSuccess) e = cudaEventRecord(side->join2, side->stream2);
    if (e != cudaSuccess) return cuda_fail(e, "join from helper streams");
  }
  if (table == nullptr) {
    PdlScope pdl_gather;  // behind top-K, whose ids it waits for after its prologue
    DCOCO_TRY(enqueue_repr_gather(D, o_ids, emb, V, w, s.repr, st));
  }
  e = cudaStreamWaitEvent(st, side->join2, 0);
  if (e != cudaSuccess) return cuda_fail(e, "join from helper streams");
  // From here on each kernel may launch while its predecessor finishes (programmatic
  // dependent launch); each waits for it before touching its data.
  PdlScope pdl;
  // uz/vz scratch holds the scorer's prepared operands P and Q here.
  DCOCO_TRY(enqueue_repr_fuse(D, w, s.uz, s.vz, s.repr, st, o_vals, s.wsp, side->join, table, o_ids, V));
  DCOCO_TRY(enqueue_scores_prepped(D, s.uz, s.vz, o_vals, w, o_S, st));
  SelectVerifyArgs a = {};
  a.S = o_S;
  a.vals = o_vals;
  a.ids = o_ids;
  a.k_sel = o_k;
  a.tokens = tokens;
  a.mode = mode;
  a.t = t;
  a.q = q;
  a.u = u;
  a.accept_len = accept_len;
  a.committed = committed;
  a.n_commit = n_commit;
  a.near_tie = near_tie;
  a.N = N;
  a.B = B;
  a.K = K;
  a.V = V;
  e = launch_select_verify(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "walk/verify launch");
  return DCOCO_OK;
}
}  // namespace

extern "C" {

int dcoco_cycle(const void* logits, int V, const void* emb, const void* h, const dcoco_weights* w, int N, int B, int K,
                int mode, const int32_t* t, const float* q, const float* u, float* vals, int32_t* ids, float* S,
                int32_t* k_sel, int32_t* tokens, int32_t* accept_len, int32_t* committed, int32_t* n_commit,
                int32_t* near_tie, void* workspace, size_t workspace_bytes, void* stream) {
  clear_err();
  if (emb == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "emb is NULL");
  return cycle_impl(logits, nullptr, V, emb, nullptr, h, w, N, B, K, mode, t, q, u, vals, ids, S, k_sel, tokens, accept_len,
                    committed, n_commit, near_tie, workspace, workspace_bytes, stream);
}

int dcoco_cycle_table(const void* logits, int V, const void* table, const void* h, const dcoco_weights* w, int N,
                      int B, int K, int mode, const int32_t* t, const float* q, const float* u, float* vals,
                      int32_t* ids, float* S, int32_t* k_sel, int32_t* tokens, int32_t* accept_len,
                      int32_t* committed, int32_t* n_commit, int32_t* near_tie, void* workspace,
                      size_t workspace_bytes, void* stream) {
  clear_err();
  if (table == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "table is NULL");
  return cycle_impl(logits, nullptr, V, nullptr, table, h, w, N, B, K, mode, t, q, u, vals, ids, S, k_sel, tokens, accept_len,
                    committed, n_commit, near_tie, workspace, workspace_bytes, stream);
}

size_t dcoco_cycle_lm_workspace_size(const dcoco_weights* w, int N, int B, int K, int V) {
  const size_t base = dcoco_cycle_workspace_size(w, N, B, K);
  if (base == 0 || (w->dtype != DCOCO_BF16 && w->dtype != DCOCO_F32)) return 0;
  const size_t lm = dcoco_lm_head_topk_workspace_size(w->dtype, N, B, V, K);
  return lm == 0 ? 0 : base + round256(lm);
}

int dcoco_cycle_lm(const void* W_lm, int V, const void* emb, const void* h, const dcoco_weights* w, int N, int B,
                   int K, int mode, const int32_t* t, const float* q, const float* u, float* vals, int32_t* ids,
                   float* S, int32_t* k_sel, int32_t* tokens, int32_t* accept_len, int32_t* committed,
                   int32_t* n_commit, int32_t* near_tie, void* workspace, size_t workspace_bytes, void* stream) {
  clear_err();
  if (W_lm == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "W_lm is NULL");
  if (emb == nullptr) return fail(DCOCO_ERR_INVALID_ARG, "emb is NULL");
  return cycle_impl(nullptr, W_lm, V, emb, nullptr, h, w, N, B, K, mode, t, q, u, vals, ids, S, k_sel, tokens,
                    accept_len, committed, n_commit, near_tie, workspace, workspace_bytes, stream);
}

size_t dcoco_embedding_table_bytes(const dcoco_weights* w, int V) {
  if (w == nullptr || V < 1) return 0;
  return static_cast<size_t>(V) * w->r * (w->dtype == DCOCO_BF16 ? 2 : 4);
}

int dcoco_embedding_table(const void* emb, int V, const dcoco_weights* w, void* table, void* stream) {
  clear_err();
  DCOCO_TRY(check_weights(w));
  if (V < 1) return fail(DCOCO_ERR_INVALID_ARG, "V=%d", V);
  DCOCO_TRY(check_ptr(emb, "emb"));
  DCOCO_TRY(check_ptr(table, "table"));
  const Dims D = dims_of(w, 1, 1, 1);
  GemmArgs a = {};
  DCOCO_TRY(a_map_tiled(a, emb, D, V, D.E, D.E));
  a.M = V;
  a.K = D.E;
  a.n_groups = 1;
  const int BN = pick_bn(D.r, true);
  if (BN != D.r) return fail(DCOCO_ERR_UNSUPPORTED, "r=%d", D.r);
  DCOCO_TRY(gemm_group(&a.g[0], w->W_e, D, D.r, D.E, D.E, BN, table, D.r, EPI_LN, a.M));
  return run_gemm(a, D, BN, as_stream(stream), "gemm LN(W_e Emb) table");
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free pair state
// Scratch of dcoco_pair_state_noalloc: one statically sized array per device, shared by
// every call.  In host code the name below is only a stand-in for the device object; the
// device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_pair_state_scratch[DCOCO_PAIR_STATE_NOALLOC_SCRATCH_BYTES];

namespace {
void* pair_state_scratch(int* rc) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *rc = fail(DCOCO_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_pair_state_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *rc = cuda_fail(e, "cudaGetSymbolAddress(pair-state scratch)");
      return nullptr;
    }
    addr[dev] = p;
  }
  *rc = DCOCO_OK;
  return addr[dev];
}
}  // namespace

extern "C" int dcoco_pair_state_noalloc(const void* h, const dcoco_weights* w, int N, int B, float* ws_pair,
                                        void* stream) {
  clear_err();
  DCOCO_TRY(check_weights(w));
  DCOCO_TRY(check_block(N, B, 1));
  DCOCO_TRY(check_ptr(h, "h"));
  DCOCO_TRY(check_ptr(ws_pair, "ws_pair"));
  const size_t need = dcoco_pair_state_workspace_size(w, N, B);
  if (need > DCOCO_PAIR_STATE_NOALLOC_SCRATCH_BYTES)
    return fail(DCOCO_ERR_WORKSPACE,
                "pair state of N=%d B=%d r=%d needs %zu bytes of scratch; the built-in array holds %u "
                "(call dcoco_pair_state with a workspace instead)",
                N, B, w->r, need, DCOCO_PAIR_STATE_NOALLOC_SCRATCH_BYTES);
  int rc;
  void* scratch = pair_state_scratch(&rc);
  if (rc != DCOCO_OK) return rc;
  Carve c(scratch);
  PairScratch s;
  pair_scratch(dims_of(w, N, B, 1), c, &s);
  return enqueue_pair(dims_of(w, N, B, 1), h, w, ws_pair, s, as_stream(stream));
}
