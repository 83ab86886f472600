// qmv_chain.cu -- a chain of M = 1 matvecs run by one persistent launch.
//
// What it computes: exactly what the same sequence of qmv_gemv /
// qmv_fused_rmsnorm_gemv calls computes, op by op, bit for bit (the same
// per-stage arithmetic, qmv_pipe.cuh).  Why: the pages' decode loop pays a
// per-dispatch tax between its matvecs and names a whole-layer or multi-stage
// single dispatch as the lever against it ("Gemma4 raw-Metal loop on A19",
// "What moved the needle", dispatch-count fusion; "The parked levers",
// mega-kernel restructure).
//
// How:
//   * One CTA per SM (cooperative launch, so all CTAs are resident), warp-
//     specialised like the single-matvec pipeline: a producer warp, a fold
//     warp and 16 compute warps.  The stage ring runs across op boundaries:
//     the producer streams the next matvec's weights while the compute warps
//     still finish the current one or wait at a dependency, so HBM keeps
//     streaming through the gaps a sequence of launches leaves.
//   * Every op's row groups are spread over the CTAs from a rotating start,
//     so the leftover groups of successive ops land on different CTAs.
//   * Dependencies: the host records each op's activation reads (x,
//     residual, gamma) and writes (y, h_out) as byte ranges.  Before an op
//     that reads what an earlier op (since the last barrier) writes, or
//     writes what one reads or writes, the chain inserts a grid-wide barrier;
//     ops without such a conflict overlap.  Packed weights are never written
//     by a chain.
//   * The barrier: the compute warps of a CTA meet on a named barrier, one
//     thread waits (bounded) until the fold warp has stored every output of
//     the earlier ops, then arrives on a global counter in the caller's
//     workspace and spins (bounded) on its generation word.
//   * Every wait is bounded.  A wait that runs out records an error code in
//     the chain's device error word and marks the CTA aborted; its warps then
//     skip the remaining work but still reach every named barrier, the
//     producer lets its copies land, and the kernel returns.
#include <mutex>
#include <new>
#include <vector>

#include "qmv_pipe.cuh"

namespace qmv {

__device__ int g_chain_error = 0;

using namespace pipe;

namespace {

constexpr int CH_TC = 512;                 // compute threads per CTA
constexpr int CH_THREADS = 64 + CH_TC;     // + producer warp + fold warp
constexpr int CH_U = 2;                    // rows per compute thread
constexpr int CH_SLOT = 24576;             // bytes per ring stage
constexpr int CH_RMAX = 32;                // rows per group at most
constexpr int CH_GS = 2048 / 32 + 4;       // fold-buffer row stride (segments of <= 2048 codes; 16-byte rows)
constexpr int CH_TBUF = CH_RMAX * CH_GS;   // floats per fold buffer
constexpr int CH_WS_HEAD = 256;            // workspace bytes before the op table
constexpr int ERR_GRID_BARRIER = 6, ERR_FOLD_WAIT = 7;

// Shared-memory layout of the chain kernel (bytes; the first 128 hold the
// mbarriers and flags).
struct ChainLayout {
  int y_off, ysum_off, bsum_off, stage_off, tbuf_off, smem;
};

}  // namespace

// One op of a chain as the kernel reads it (in the caller's workspace).
struct ChainOp {
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  GemvArgs a;
  TmaPlan P;
  int bits, exact, barrier, g_off, h_cta;
};
static_assert(alignof(ChainOp) >= 64 && sizeof(ChainOp) % 64 == 0, "tensor maps stay 64-byte aligned");

// The library's own chain scratch (barrier words + op table), for chains made
// by qmv_chain_create_no_alloc: a file-scope device array, so nothing is
// allocated at run time by anyone.  One per device (a module global); chains
// that use it must not run at the same time.
constexpr int CH_STATIC_OPS = 1024;
static __device__ __align__(256) unsigned char g_chain_scratch[256 + CH_STATIC_OPS * sizeof(ChainOp)];

namespace {

struct ChainParams {
  const ChainOp* ops;
  int n_ops;
  unsigned* bar;        // [0] arrivals, [1] generation
  ChainLayout L;
};

__device__ __forceinline__ int first_group(int g_off, int cta, int grid) {
  return (cta - g_off % grid + grid) % grid;
}

__device__ __forceinline__ int stages_of(const TmaPlan& P, int g0, int grid) {
  return (g0 < P.ngroups) ? ((P.ngroups - g0 + grid - 1) / grid) * P.NSEG : 0;
}

// Grid-wide barrier, called by one thread per CTA.
__device__ bool grid_barrier(unsigned* bar, volatile int* abort_f, int* err) {
  __threadfence();
  volatile unsigned* vgen = bar + 1;
  const unsigned gen = *vgen;
  if (atomicAdd(bar, 1u) == gridDim.x - 1) {
    atomicExch(bar, 0u);
    __threadfence();
    atomicAdd(bar + 1, 1u);
    return true;
  }
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (*vgen != gen) {
      __threadfence();
      return true;
    }
    if (*abort_f) return false;
    __nanosleep(64);
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  *abort_f = 1;
  atomicCAS(err, 0, ERR_GRID_BARRIER);
  return false;
}

// The fold warp has stored every output of ops < op.
__device__ bool wait_folds(volatile int* fold_done, int op, volatile int* abort_f, int* err) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (*fold_done >= op) return true;
    if (*abort_f) return false;
    __nanosleep(64);
    if (global_ns() - t0 > WAIT_LIMIT_NS) break;
  }
  *abort_f = 1;
  atomicCAS(err, 0, ERR_FOLD_WAIT);
  return false;
}

// The table build of one op variant, as a call of its own (its registers are
// then allocated apart from the kernel's stage loop).
template <int B, bool FU, bool EX>
__device__ __noinline__ void table_call(const ChainOp& o, float* y2f, float* ysum, float* bsum,
                                        float* inv_sh, __half* h_out, int tc) {
  build_table<B, FU, EX>(o.a, y2f, ysum, bsum, inv_sh, h_out, tc, CH_TC, 3);
}

__device__ __forceinline__ void table_any(const ChainOp& o, float* y2f, float* ysum, float* bsum,
                                          float* inv_sh, __half* h_out, int tc) {
  const bool fu = o.a.fused != 0, ex = o.exact != 0;
#define QMV_TABLE(B)                                                              \
  if (fu) {                                                                       \
    if (ex) table_call<B, true, true>(o, y2f, ysum, bsum, inv_sh, h_out, tc);     \
    else table_call<B, true, false>(o, y2f, ysum, bsum, inv_sh, h_out, tc);       \
  } else {                                                                        \
    if (ex) table_call<B, false, true>(o, y2f, ysum, bsum, inv_sh, h_out, tc);    \
    else table_call<B, false, false>(o, y2f, ysum, bsum, inv_sh, h_out, tc);      \
  }
  switch (o.bits) {
    case 2: QMV_TABLE(2) break;
    case 4: QMV_TABLE(4) break;
    default: QMV_TABLE(8) break;
  }
#undef QMV_TABLE
}

__device__ __forceinline__ void stage_any(const ChainOp& o, const TmaPlan& P, const unsigned char* st,
                                          int c, int rp, int seg, int rows, const u64* y2s,
                                          const float* ysum, float* tbr) {
  const bool pr = o.a.perrow != 0, ex = o.exact != 0;
#define QMV_STAGE(B)                                                                                 \
  if (pr) {                                                                                          \
    if (ex) compute_stage<B, true, true, CH_U>(st, P, c, rp, seg, rows, y2s, ysum, tbr, CH_GS);      \
    else compute_stage<B, true, false, CH_U>(st, P, c, rp, seg, rows, y2s, ysum, tbr, CH_GS);        \
  } else {                                                                                           \
    if (ex) compute_stage<B, false, true, CH_U>(st, P, c, rp, seg, rows, y2s, ysum, tbr, CH_GS);     \
    else compute_stage<B, false, false, CH_U>(st, P, c, rp, seg, rows, y2s, ysum, tbr, CH_GS);       \
  }
  switch (o.bits) {
    case 2: QMV_STAGE(2) break;
    case 4: QMV_STAGE(4) break;
    default: QMV_STAGE(8) break;
  }
#undef QMV_STAGE
}

__global__ void __launch_bounds__(CH_THREADS, 1) gemv_chain_kernel(ChainParams cp) {
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + NS;
  uint64_t* tfull = empty + NS;
  uint64_t* tempty = tfull + 2;
  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + 96);
  float* inv_sh = reinterpret_cast<float*>(sm + 100);
  volatile int* fold_done = reinterpret_cast<volatile int*>(sm + 104);
  float* y2f = reinterpret_cast<float*>(sm + cp.L.y_off);
  float* ysum = reinterpret_cast<float*>(sm + cp.L.ysum_off);
  float* bsum = reinterpret_cast<float*>(sm + cp.L.bsum_off);
  unsigned char* stages = sm + cp.L.stage_off;
  float* tbuf = reinterpret_cast<float*>(sm + cp.L.tbuf_off);
  int* err = &g_chain_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, grid = gridDim.x;

  if ((sa(sm) & 127u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(err, 0, ERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CH_TC / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], CH_TC / 32);
      mbar_init(&tempty[b], 1);
    }
    *abort_f = 0;
    *fold_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  if (warp == 0) {
    int i = 0;
    bool dead = false;
    for (int op = 0; op < cp.n_ops && !dead; ++op) {
      const ChainOp* o = cp.ops + op;
      const TmaPlan P = o->P;
      const int perrow = o->a.perrow;
      const int g0 = first_group(o->g_off, cta, grid);
      for (int g = g0; g < P.ngroups && !dead; g += grid) {
        for (int seg = 0; seg < P.NSEG; ++seg, ++i) {
          const int s = i & (NS - 1);
          if (i >= NS && !mbar_wait_fast(&empty[s], ((i / NS) - 1) & 1, abort_f, ERR_TIMEOUT_EMPTY, err)) {
            dead = true;
            break;
          }
          if (*abort_f) {
            dead = true;
            break;
          }
          unsigned char* st = stages + (size_t)s * CH_SLOT;
          if (lane == 0) {
            const uint32_t tx = (uint32_t)P.R * P.seg_bytes + (perrow ? 0u : (uint32_t)P.R * P.seg_sc);
            mbar_arrive_tx(&full[s], tx);
            tma_2d(st, &o->tm_codes, seg * (P.seg_bytes / 8), g * P.R, &full[s]);
            if (!perrow) tma_2d(st + P.sc_off, &o->tm_scales, seg * (P.KS / 32), g * P.R, &full[s]);
          }
        }
      }
    }
    // let every copy this warp issued land before the CTA can exit
    if (lane == 0)
      for (int j = (i > NS ? i - NS : 0); j < i; ++j) mbar_drain(&full[j % NS], (j / NS) & 1, err);
    return;
  }

  // ---------------------------------------------------------- fold warp --
  if (warp == 1) {
    int i = 0;
    bool dead = false;
    for (int op = 0; op < cp.n_ops; ++op) {
      const ChainOp* o = cp.ops + op;
      const TmaPlan P = o->P;
      const GemvArgs a = o->a;
      const int g0 = first_group(o->g_off, cta, grid);
      for (int g = g0; g < P.ngroups; g += grid) {
        float acc = 0.0f;
        const int64_t r0 = (int64_t)g * P.R;
        const int rows = (int)min((int64_t)P.R, (int64_t)a.N - r0);
        for (int seg = 0; seg < P.NSEG; ++seg, ++i) {
          const int tb = i & 1;
          if (!dead && !mbar_wait_fast(&tfull[tb], (i >> 1) & 1, abort_f, ERR_TIMEOUT_TFULL, err)) dead = true;
          if (!dead) fold_stage(a, P, tbuf + (size_t)tb * CH_TBUF, CH_GS, lane, GroupRows{r0, r0, rows, true},
                                seg, acc);
          __syncwarp();
          if (lane == 0 && !dead) mbar_arrive(&tempty[tb]);
        }
      }
      // publish: every output of ops <= op is stored
      __threadfence();
      __syncwarp();
      if (lane == 0) *fold_done = op + 1;
    }
    return;
  }

  // ------------------------------------------------------- compute warps --
  const int tc = threadIdx.x - 64;
  const u64* y2s = reinterpret_cast<const u64*>(y2f);
  int i = 0;
  bool dead = false;
  for (int op = 0; op < cp.n_ops; ++op) {
    const ChainOp* o = cp.ops + op;
    const TmaPlan P = o->P;
    // every compute warp is done with the previous op (its table and its
    // h_out stores)
    named_bar(3, CH_TC);
    if (o->barrier) {
      if (tc == 0 && !*abort_f && wait_folds(fold_done, op, abort_f, err))
        grid_barrier(cp.bar, abort_f, err);
      named_bar(3, CH_TC);
    }
    dead = dead || (*abort_f != 0);
    const int g0 = first_group(o->g_off, cta, grid);
    const int my_stages = stages_of(P, g0, grid);
    const bool writes_h = (cta == o->h_cta) && o->a.h_out != nullptr;
    // (built even by aborted warps: it holds named barriers of all compute warps)
    if (my_stages > 0 || writes_h) {
      table_any(*o, y2f, ysum, bsum, inv_sh, writes_h ? o->a.h_out : nullptr, tc);
      named_bar(3, CH_TC);
    }
    const bool active = tc < P.Cs * P.RP;
    const int c = active ? tc % P.Cs : 0;
    const int rp = active ? tc / P.Cs : 0;
    for (int g = g0; g < P.ngroups; g += grid) {
      const int64_t r0 = (int64_t)g * P.R;
      const int rows = (int)min((int64_t)P.R, (int64_t)o->a.N - r0);
      for (int seg = 0; seg < P.NSEG; ++seg, ++i) {
        const int s = i & (NS - 1);
        const int tb = i & 1;
        if (!dead && !mbar_wait_fast(&full[s], (i / NS) & 1, abort_f, ERR_TIMEOUT_FULL, err)) dead = true;
        if (!dead && i >= 2 &&
            !mbar_wait_fast(&tempty[tb], ((i >> 1) - 1) & 1, abort_f, ERR_TIMEOUT_TEMPTY, err))
          dead = true;
        if (!dead && active)
          stage_any(*o, P, stages + (size_t)s * CH_SLOT, c, rp, seg, rows, y2s, ysum,
                    tbuf + (size_t)tb * CH_TBUF);
        __syncwarp();
        if (lane == 0 && !dead) {
          mbar_arrive(&empty[s]);
          mbar_arrive(&tfull[tb]);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ host --

struct Range {
  uintptr_t lo, hi;   // [lo, hi)
};

bool overlaps(const std::vector<Range>& a, const Range& r) {
  for (const Range& q : a)
    if (q.lo < r.hi && r.lo < q.hi) return true;
  return false;
}

// The chain's plan for one op: U = 2 rows per compute thread and an even
// number of rows per group R <= 32 whose stage fits a ring slot, chosen so
// that the busiest CTA's share of the op -- its stages times the time of a
// stage, modelled as a fixed cost (a compute thread's own work does not
// shrink with R) plus R * segment codes -- is smallest (the op ends with its
// busiest CTA); on a tie the larger R.
constexpr int64_t CH_STAGE_FIXED = 65536;   // code-equivalents of a stage's fixed cost
bool chain_plan(int N, int K, int bits, bool perrow, int ctas, TmaPlan* P) {
  if (K % 256 != 0 || ctas < 1) return false;
  const int KS = tma_segment(K);
  const int Cs = KS / 64;
  const int seg_bytes = KS * bits / 8;
  const int seg_sc = perrow ? 0 : (KS / 32) * 2;
  int best_R = 0;
  int64_t best_cost = 0;
  for (int R = CH_RMAX; R >= 2; R -= 2) {
    const int RP = R / CH_U;
    if (Cs * RP > CH_TC) continue;
    const int sc_off = (R * seg_bytes + 127) & ~127;
    const int stage = (sc_off + R * seg_sc + 127) & ~127;
    if (stage > CH_SLOT) continue;
    const int64_t groups = ((int64_t)N + R - 1) / R;
    const int64_t t_stage = CH_STAGE_FIXED + (int64_t)R * KS;
    const int64_t cost = ((groups + ctas - 1) / ctas) * (K / KS) * t_stage;
    if (best_R == 0 || cost < best_cost) {
      best_R = R;
      best_cost = cost;
    }
  }
  if (best_R == 0) return false;
  const int R = best_R;
  memset(P, 0, sizeof(*P));
  P->C = K / 64;
  P->Cs = Cs;
  P->KS = KS;
  P->NSEG = K / KS;
  P->RP = R / CH_U;
  P->R = R;
  P->Tc = CH_TC;
  P->row_bytes = K * bits / 8;
  P->seg_bytes = seg_bytes;
  P->seg_sc = seg_sc;
  P->sc_off = (R * seg_bytes + 127) & ~127;
  P->stage_bytes = (P->sc_off + R * seg_sc + 127) & ~127;
  P->ngroups = (int)(((int64_t)N + R - 1) / R);
  return true;
}

ChainLayout chain_layout(int max_K) {
  ChainLayout L;
  L.y_off = 128;
  L.ysum_off = L.y_off + (max_K / 64) * YS * 8;
  L.bsum_off = L.ysum_off + (max_K / 32) * 4;
  L.stage_off = (L.bsum_off + (max_K / 32) * 4 + 127) & ~127;
  L.tbuf_off = L.stage_off + NS * CH_SLOT;
  L.smem = L.tbuf_off + 2 * CH_TBUF * 4;
  return L;
}

}  // namespace
}  // namespace qmv

#define QMV_CHAIN_MAGIC 0x51434841u

struct qmv_chain {
  uint32_t magic;
  int max_ops;
  unsigned char* d_ws;
  size_t ws_bytes;
  std::vector<qmv::ChainOp> ops;
  std::vector<qmv::Range> reads, writes;   // since the last barrier
  int n_barriers;
  int max_K;
  int groups_so_far;
  bool dirty;
  int static_dev;     // >= 0: the workspace is the library's scratch array on this device
};

static bool chain_ok(const qmv_chain* c) { return c && c->magic == QMV_CHAIN_MAGIC; }

extern "C" {

size_t qmv_chain_workspace_bytes(int max_ops) {
  if (max_ops < 1) return 0;
  return (size_t)qmv::CH_WS_HEAD + (size_t)max_ops * sizeof(qmv::ChainOp);
}

int qmv_chain_create(qmv_chain** out, int max_ops, void* d_workspace, size_t workspace_bytes) {
  if (!out || max_ops < 1 || !d_workspace) return QMV_ERR_INVALID_ARG;
  if (((uintptr_t)d_workspace % 256) != 0) return QMV_ERR_ALIGNMENT;
  if (workspace_bytes < qmv_chain_workspace_bytes(max_ops)) return QMV_ERR_INVALID_ARG;
  qmv_chain* c = new (std::nothrow) qmv_chain();
  if (!c) return QMV_ERR_INVALID_ARG;
  c->magic = QMV_CHAIN_MAGIC;
  c->max_ops = max_ops;
  c->d_ws = (unsigned char*)d_workspace;
  c->ws_bytes = workspace_bytes;
  c->n_barriers = 0;
  c->max_K = 0;
  c->groups_so_far = 0;
  c->dirty = true;
  c->static_dev = -1;
  *out = c;
  return QMV_OK;
}

// Host bookkeeping of the library's scratch array, one entry per device: its
// device address (looked up once) and the chain whose op table it holds.
// Chains on several host threads read and update both, so every access takes
// g_static_mu.
static std::mutex g_static_mu;
static void* g_static_addr[64];
static const qmv_chain* g_static_owner[64];

int qmv_chain_create_no_alloc(qmv_chain** out, int max_ops) {
  if (!out || max_ops < 1) return QMV_ERR_INVALID_ARG;
  if (max_ops > qmv::CH_STATIC_OPS) return QMV_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qmv::record_cuda_error(e);
  if (dev < 0 || dev >= 64) return QMV_ERR_UNSUPPORTED;
  void* addr = nullptr;
  {
    // the scratch array's address on this device (set-up, once per device)
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      e = cudaGetSymbolAddress(&g_static_addr[dev], qmv::g_chain_scratch);
      if (e != cudaSuccess) {
        g_static_addr[dev] = nullptr;
        return qmv::record_cuda_error(e);
      }
    }
    addr = g_static_addr[dev];
  }
  const int rc = qmv_chain_create(out, max_ops, addr, sizeof(qmv::g_chain_scratch));
  if (rc == QMV_OK) (*out)->static_dev = dev;
  return rc;
}

static int chain_add(qmv_chain* c, const qmv_pack* p, const void* x, const void* r, const void* g,
                     float eps, void* h_out, void* y, int y_dtype, int mode) {
  using namespace qmv;
  if (!chain_ok(c) || !p || p->magic != QMV_PACK_MAGIC || !p->bound || !x || !y) return QMV_ERR_INVALID_ARG;
  if ((int)c->ops.size() >= c->max_ops) return QMV_ERR_INVALID_ARG;
  if (y_dtype != QMV_F32 && y_dtype != QMV_F16) return QMV_ERR_INVALID_ARG;
  if (mode != QMV_FAST && mode != QMV_EXACT) return QMV_ERR_INVALID_ARG;
  const bool fused = r != nullptr;
  if (fused && (!g || !(eps >= 0.0f))) return QMV_ERR_INVALID_ARG;
  if (((uintptr_t)x % 16) || ((uintptr_t)y % 4) || (fused && ((uintptr_t)r % 16 || (uintptr_t)g % 16)) ||
      (h_out && (uintptr_t)h_out % 16))
    return QMV_ERR_ALIGNMENT;
  ChainOp o;
  memset(&o, 0, sizeof(o));
  GemvArgs& a = o.a;
  a.codes = (const uint4*)p->d_codes;
  a.scales = (const __half*)p->d_scales;
  a.N = p->N;
  a.K = p->K;
  a.G = p->G;
  a.row_u4 = (int)((int64_t)p->K * p->bits / 128);
  a.perrow = (p->group == p->K && p->K != 32) ? 1 : 0;
  a.x = (const __half*)x;
  a.y = y;
  a.y_f16 = (y_dtype == QMV_F16);
  a.M = 1;
  a.fused = fused ? 1 : 0;
  a.r = (const __half*)r;
  a.gamma = (const __half*)g;
  a.eps = eps;
  a.h_out = fused ? (__half*)h_out : nullptr;
  a.folded = (mode == QMV_FAST) ? 1 : 0;
  if (!chain_plan(a.N, a.K, p->bits, a.perrow != 0, dev_info().sms, &o.P)) return QMV_ERR_UNSUPPORTED;
  const int max_K = c->max_K > a.K ? c->max_K : a.K;
  if (chain_layout(max_K).smem > dev_info().max_smem_optin) return QMV_ERR_UNSUPPORTED;
  if (!encode_pack_maps(a, o.P, &o.tm_codes, &o.tm_scales)) return QMV_ERR_UNSUPPORTED;
  o.bits = p->bits;
  o.exact = (mode == QMV_EXACT) ? 1 : 0;
  // dependencies on the ops since the last barrier
  const uintptr_t K2 = (uintptr_t)a.K * 2;
  std::vector<Range> rd = {{(uintptr_t)x, (uintptr_t)x + K2}};
  if (fused) {
    rd.push_back({(uintptr_t)r, (uintptr_t)r + K2});
    rd.push_back({(uintptr_t)g, (uintptr_t)g + K2});
  }
  std::vector<Range> wr = {{(uintptr_t)y, (uintptr_t)y + (uintptr_t)a.N * (a.y_f16 ? 2 : 4)}};
  if (a.h_out) wr.push_back({(uintptr_t)h_out, (uintptr_t)h_out + K2});
  bool conflict = false;
  for (const Range& q : rd) conflict = conflict || overlaps(c->writes, q);
  for (const Range& q : wr) conflict = conflict || overlaps(c->writes, q) || overlaps(c->reads, q);
  if (conflict) {
    o.barrier = 1;
    c->n_barriers++;
    c->reads.clear();
    c->writes.clear();
  }
  c->reads.insert(c->reads.end(), rd.begin(), rd.end());
  c->writes.insert(c->writes.end(), wr.begin(), wr.end());
  // rotate the CTAs that get the leftover groups; h_out from the CTA that
  // owns the op's first group
  const int sms = dev_info().sms;
  o.g_off = c->groups_so_far % sms;
  o.h_cta = o.g_off;
  c->groups_so_far = (int)(((int64_t)c->groups_so_far + o.P.ngroups) % sms);
  c->max_K = max_K;
  c->ops.push_back(o);
  c->dirty = true;
  return QMV_OK;
}

int qmv_chain_add_gemv(qmv_chain* c, const qmv_pack* p, const void* x, void* y, int y_dtype, int mode) {
  return chain_add(c, p, x, nullptr, nullptr, 0.0f, nullptr, y, y_dtype, mode);
}

int qmv_chain_add_fused_rmsnorm_gemv(qmv_chain* c, const qmv_pack* p, const void* x, const void* residual,
                                     const void* gamma, float eps, void* h_out, void* y, int y_dtype,
                                     int mode) {
  if (!residual) return QMV_ERR_INVALID_ARG;
  return chain_add(c, p, x, residual, gamma, eps, h_out, y, y_dtype, mode);
}

int qmv_chain_run(qmv_chain* c, void* stream) {
  using namespace qmv;
  if (!chain_ok(c)) return QMV_ERR_INVALID_ARG;
  if (c->ops.empty()) return QMV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  // the scratch array's owner is read and set under the lock, together with
  // the upload it decides on, so two host threads agree on whose table is there
  std::unique_lock<std::mutex> lock(g_static_mu, std::defer_lock);
  if (c->static_dev >= 0) {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev != c->static_dev) return QMV_ERR_INVALID_ARG;
    lock.lock();
    if (g_static_owner[dev] != c) c->dirty = true;   // another chain's table is there
  }
  if (c->dirty) {
    // The op table goes up on the run's own stream, so it lands after the
    // work queued there before (an earlier run that still reads the table)
    // and before this run's kernel.  The source is pageable host memory:
    // the copy stages it before returning, so later edits of the chain
    // cannot reach the device copy.  A capture would record a copy from
    // pageable memory, which is not allowed: refuse it.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (cap != cudaStreamCaptureStatusNone) return QMV_ERR_UNSUPPORTED;
    e = cudaMemcpyAsync(c->d_ws + CH_WS_HEAD, c->ops.data(), c->ops.size() * sizeof(ChainOp),
                        cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return record_cuda_error(e);
    c->dirty = false;
    if (c->static_dev >= 0) g_static_owner[c->static_dev] = c;
  }
  if (lock.owns_lock()) lock.unlock();
  const ChainLayout L = chain_layout(c->max_K);
  static thread_local int set_dev = -1;
  static thread_local int set_smem = 0;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (dev != set_dev || L.smem > set_smem) {
    e = cudaFuncSetAttribute(gemv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (e != cudaSuccess) return record_cuda_error(e);
    set_dev = dev;
    set_smem = L.smem;
  }
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_chain_kernel, CH_THREADS, L.smem);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (occ < 1) return QMV_ERR_UNSUPPORTED;
  // the barrier words start at zero every run
  e = cudaMemsetAsync(c->d_ws, 0, 64, s);
  if (e != cudaSuccess) return record_cuda_error(e);
  ChainParams cp;
  cp.ops = reinterpret_cast<const ChainOp*>(c->d_ws + CH_WS_HEAD);
  cp.n_ops = (int)c->ops.size();
  cp.bar = reinterpret_cast<unsigned*>(c->d_ws);
  cp.L = L;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(dev_info().sms);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel, cp);
  if (e != cudaSuccess) return record_cuda_error(e);
  return QMV_OK;
}

int qmv_chain_info(const qmv_chain* c, int* n_ops, int* n_barriers, int* smem_bytes) {
  if (!chain_ok(c)) return QMV_ERR_INVALID_ARG;
  if (n_ops) *n_ops = (int)c->ops.size();
  if (n_barriers) *n_barriers = c->n_barriers;
  if (smem_bytes) *smem_bytes = c->ops.empty() ? 0 : qmv::chain_layout(c->max_K).smem;
  return QMV_OK;
}

int qmv_chain_destroy(qmv_chain* c) {
  if (!chain_ok(c)) return QMV_ERR_INVALID_ARG;
  if (c->static_dev >= 0) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_owner[c->static_dev] == c) g_static_owner[c->static_dev] = nullptr;
  }
  c->magic = 0;
  delete c;
  return QMV_OK;
}

}  // extern "C"

namespace qmv {

int read_chain_error(int clear, int* out) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_chain_error, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_chain_error, &z, sizeof(int));
    if (e != cudaSuccess) return (int)e;
  }
  *out = v;
  return 0;
}

}  // namespace qmv
