// Host layer of libdmuon: argument validation, status codes, the per-device workspace, the plan
// (workspace layout + grouped job/tile lists of every phase) and the C entry points of dmuon.h.
//
// Phase order of the Gram form ("Newton-Schulz 变体", sections "Gram 空间 NS（Dao-AILab）" and
// "重启机制"), per step k with coefficients (a, b, c), on every matrix at once:
//   start:            R = X X^T                                   (symmetric, K = n)
//   restart before k: X' = Q X ; R = X' X'^T ; Q = I              (K = m, then K = n)
//   step k:           Z = b R + c R^2  [Q = Z + a I after a (re)start]   (symmetric, K = m)
//                     Q' = Z Q + a Q   (otherwise)                        (K = m)
//                     S = Z R + a R ; R = S Z + a S   when step k+1 exists and is not a restart,
//                                                     i.e. R <- (aI+Z) R (aI+Z)   (both symmetric)
//   output:           W <- W - lr * (Q X), written in the caller's orientation.
// Direct form ("直接空间 NS（经典）"), per step: A = X X^T ; B = b A + c A^2 ; X' = B X + a X, the
// last step writing W <- W - lr * X' instead of X'.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
namespace {

__device__ unsigned g_status_word;  // device status word (kDevTimeout | kDevNonfinite)

thread_local std::string t_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DMUON_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define DM_CUDA(call, what)                   \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

constexpr size_t kNone = ~size_t(0);
constexpr int64_t kMaxDim = int64_t(1) << 24;
constexpr int kMaxGroups = 64;  // pipeline groups of one dmuon_muon_step_host call
// dmuon_muon_step_host gathers with one launch instead of a copy per matrix from this many matrices on,
// when they average less than this many gradient bytes.
constexpr int kGatherMinCount = 64;
constexpr int64_t kGatherMaxAvgBytes = int64_t(4) << 20;

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

enum PlanKind { kPlanNs = 0, kPlanMuon = 1, kPlanMomNorm = 2, kPlanNsTp = 3 };

// Host-only flag on a phase's single JobSpec: the phase is the fixed-order sum of a matrix's per-shard
// fp32 Gram partials into R (not a GEMM).
constexpr int kJobTpReduce = 1 << 10;

struct PlanKey {
  int kind = -1, backend = 0, steps = 0, gdtype = 0;
  int shards = 0;  // kPlanNsTp: column shards along the long side
  int groups = 1;  // kPlanMuon: consecutive matrix groups run one after another (host-gradient pipeline)
  std::vector<int> restarts;
  std::vector<int64_t> rows, cols;
  std::vector<uintptr_t> ptrs;  // W, G, M, X_out per matrix
  bool operator==(const PlanKey& o) const {
    return kind == o.kind && backend == o.backend && steps == o.steps && gdtype == o.gdtype && shards == o.shards &&
           groups == o.groups && restarts == o.restarts && rows == o.rows && cols == o.cols && ptrs == o.ptrs;
  }
};

struct MatInfo {
  int64_t rows, cols, m, n, ldx, ldm;
  bool trans;
  bool direct;  // this matrix runs the direct iteration (backend direct, or auto where it is cheaper)
  const void* G;
  float* M;
  float* W;
  void* xout;  // caller's fp16 X (momentum_normalize only)
  size_t X = kNone, Xb = kNone, R = kNone, Z = kNone, Q = kNone, Qb = kNone, S = kNone;
  size_t P = kNone;  // kPlanNsTp: `shards` fp32 planes of m x ldp (per-shard Gram partials)
  int64_t ldp = 0;
};

// One product in a phase; operands are arena offsets (kNone = unused), resolved when bound.
struct JobSpec {
  int mat;
  int M, N, K;
  int recipe, flags;
  size_t a, b, e, d, d2;
  int64_t lda, ldb, lde, ldd;
  float* W;
  int64_t ldw;
  size_t w_off = kNone;  // W inside the workspace (per-shard Gram partials) instead of a caller pointer
};

struct LaunchRec {
  int first_job, njobs, first_tile, ntiles, tile, coef;
  int group = 0;  // the matrix group whose phases this launch runs
  int tp_reduce = 0;  // 1: not a GEMM but the reduction of per-shard Gram partials (tp_mat's)
  int tp_mat = 0;
};

struct Plan {
  PlanKey key;
  bool bound = false;
  std::vector<MatInfo> mats;
  std::vector<std::vector<JobSpec>> phases;  // one grouped launch each
  std::vector<int> phase_coef;
  std::vector<int> phase_group;
  // Matrix groups [group_begin[g], group_begin[g + 1]): each runs its row-wise passes and then all its
  // Newton-Schulz phases before the next group starts. One group unless a host-gradient call pipelines
  // its copies against the computation.
  std::vector<int> group_begin;
  int64_t nchunks = 0, ncast = 0, npartials = 0;
  size_t off_rowmats = 0, off_chunk = 0, off_tilep = 0, off_partials = 0, off_norms = 0, off_inv = 0;
  size_t off_jobs = 0, off_tiles = 0, bytes = 0;
  // host images uploaded to the arena
  std::vector<RowMat> rowmats;
  std::vector<int64_t> chunk_prefix, tile_prefix;
  std::vector<GemmJob> jobs;
  std::vector<GemmTile> tiles;
  std::vector<LaunchRec> launches;
  // Fused small-matrix path (every matrix m <= 128, n <= 512): one ns_small launch instead of phases.
  bool small_fused = false;
  unsigned restart_mask = 0;
  size_t off_small = 0;
  std::vector<SmallJob> small_jobs;
  // Tensor-parallel emulation (kPlanNsTp): shard boundaries along the long side.
  std::vector<int64_t> shard_bounds;
  int tp_slabs = 0;
  // MMA work one run of the plan issues: every tile of every GEMM launch, K rounded up to the 64-wide
  // ring slice (dmuon_plan_info). -1 for the fused small-matrix plan, which is not tile-based.
  double exec_flops = 0.0;
  int64_t exec_tiles = 0;
};

struct Layout {
  size_t off = 0;
  size_t take(size_t bytes, size_t align = 256) {
    off = (off + align - 1) / align * align;
    const size_t r = off;
    off += bytes;
    return r;
  }
};

// Cached AdamW table: the tensors and chunk prefix of the last dmuon_adamw_step call on this device.
struct AdamPlan {
  std::vector<uintptr_t> key;  // pointers and sizes
  int gdtype = 0;
  std::vector<AdamTensor> tensors;
  std::vector<int64_t> chunk_prefix;
  char* buf = nullptr;
  size_t buf_bytes = 0;
  size_t off_prefix = 0;
  bool bound = false;
};

// What a captured run of the cached plan baked in besides the plan itself.
struct GraphKey {
  bool valid = false;
  uint64_t plan_serial = 0;
  std::vector<float> coeffs;
  float lr = 0.f, beta = 0.f, eps = 0.f;
  float* norms_out = nullptr;
  bool operator==(const GraphKey& o) const {
    return valid && o.valid && plan_serial == o.plan_serial && coeffs == o.coeffs && lr == o.lr &&
           beta == o.beta && eps == o.eps && norms_out == o.norms_out;
  }
};

struct DeviceState {
  bool init = false;
  int sms = 0;
  unsigned* status = nullptr;
  char* arena = nullptr;
  size_t arena_bytes = 0;
  Plan plan;
  uint64_t plan_serial = 0;  // bumped whenever the cached plan or its workspace changes
  // Graph replay of the cached plan: `graph` runs the launches run_plan issues for `graph_key`; `last_key`
  // is the previous call's, so that a run is captured the second time the same arguments come.
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t graph = nullptr;
  GraphKey graph_key, last_key;
  AdamPlan adam;
  // Host-gradient pipeline (dmuon_muon_step_host): the copy stream, an event marking the caller's stream
  // at entry, and per group the "gradients arrived" and "gradients read by the momentum pass" events.
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t entry = nullptr;
  std::vector<cudaEvent_t> copied, read;
  // Gather table of the last host-gradient call that took the one-launch gather (many small matrices):
  // built for gather_key (host pointers, device pointers, sizes), kept on the device.
  std::vector<uintptr_t> gather_key;
  bool gather_ok = false;  // every host pointer of gather_key is device-accessible
  char* gather_buf = nullptr;
  size_t gather_bytes = 0;
  int64_t gather_chunks = 0;
};

std::mutex g_mu;
constexpr int kMaxDevices = 64;
bool g_graphs = true;  // dmuon_set_graph_replay

// Opt-in event timing (dmuon_timing_enable / dmuon_timing_read).
struct TimedLaunch {
  int cls;
  cudaEvent_t start, stop;
};
bool g_timing = false;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Names of the timing classes (dmuon.h), also the NVTX range names of their launches.
const char* const kClassNames[DMUON_TIMING_CLASSES] = {"dmuon momentum_sumsq", "dmuon finalize_norms",
                                                        "dmuon normalize_cast", "dmuon gemm_tc",
                                                        "dmuon adamw",          "dmuon tp_reduce"};

// Records events around one launch when timing is on (and an NVTX range around its host-side enqueue, for
// a profiler's timeline); otherwise just launches.
template <typename F>
cudaError_t timed(int cls, cudaStream_t stream, F&& launch) {
  if (!g_timing) return launch();
  cudaEvent_t a = take_event(), b = take_event();
  if (a) cudaEventRecord(a, stream);
  nvtxRangePushA(kClassNames[cls]);
  const cudaError_t e = launch();
  nvtxRangePop();
  if (b) cudaEventRecord(b, stream);
  if (a && b) {
    g_timed.push_back({cls, a, b});
  } else {
    if (a) g_event_pool.push_back(a);
    if (b) g_event_pool.push_back(b);
  }
  return e;
}
DeviceState g_dev[kMaxDevices];
size_t g_ws_limit = 0;

int current_device(DeviceState** out) {
  int dev = 0;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DMUON_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  DeviceState& ds = g_dev[dev];
  if (!ds.init) {
    int major = 0, minor = 0;
    DM_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
    DM_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(DMUON_ERR_UNSUPPORTED, "libdmuon is built for sm_103a (GB300); device %d is sm_%d%d", dev,
                  major, minor);
    DM_CUDA(cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
    void* addr = nullptr;
    DM_CUDA(cudaGetSymbolAddress(&addr, g_status_word), "cudaGetSymbolAddress(status word)");
    ds.status = static_cast<unsigned*>(addr);
    DM_CUDA(cudaMemset(ds.status, 0, sizeof(unsigned)), "cudaMemset(status word)");
    ds.init = true;
  }
  *out = &ds;
  return DMUON_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_ns_args(const float* coeffs, int steps, const int* restarts, int n_restarts, int backend, float eps) {
  if (backend != DMUON_NS_DIRECT && backend != DMUON_NS_GRAM && backend != DMUON_NS_AUTO)
    return fail(DMUON_ERR_INVALID_ARG, "backend must be DMUON_NS_DIRECT (0), DMUON_NS_GRAM (1) or DMUON_NS_AUTO (2), got %d",
                backend);
  if (steps < 1 || steps > DMUON_MAX_STEPS)
    return fail(DMUON_ERR_INVALID_ARG, "steps must be in [1, %d], got %d", DMUON_MAX_STEPS, steps);
  if (!coeffs) return fail(DMUON_ERR_INVALID_ARG, "coeffs is NULL");
  for (int i = 0; i < 3 * steps; ++i)
    if (!std::isfinite(coeffs[i])) return fail(DMUON_ERR_INVALID_ARG, "coeffs[%d] is not finite", i);
  if (n_restarts < 0) return fail(DMUON_ERR_INVALID_ARG, "n_restarts must be >= 0");
  if (n_restarts > 0 && !restarts) return fail(DMUON_ERR_INVALID_ARG, "restarts is NULL with n_restarts > 0");
  for (int i = 0; i < n_restarts; ++i) {
    if (restarts[i] < 0 || restarts[i] >= steps)
      return fail(DMUON_ERR_INVALID_ARG, "restart index %d outside [0, steps-1]", restarts[i]);
    if (i > 0 && restarts[i] <= restarts[i - 1])
      return fail(DMUON_ERR_INVALID_ARG, "restart indices must be strictly increasing");
  }
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(DMUON_ERR_INVALID_ARG, "eps must be finite and >= 0");
  return DMUON_OK;
}

// ---------------------------------------------------------------------------- plan building

JobSpec make_job(int mat, int M, int N, int K, int recipe, int flags, size_t a, int64_t lda, size_t b, int64_t ldb,
                 size_t e, int64_t lde, size_t d, int64_t ldd, size_t d2 = kNone) {
  JobSpec j;
  j.mat = mat;
  j.M = M, j.N = N, j.K = K;
  j.recipe = recipe, j.flags = flags;
  j.a = a, j.b = b, j.e = e, j.d = d, j.d2 = d2;
  j.lda = lda, j.ldb = ldb, j.lde = lde, j.ldd = ldd;
  j.W = nullptr;
  j.ldw = 0;
  return j;
}

// Q and S = (aI + Z) R are polynomials in the Gram matrix, hence symmetric in exact arithmetic like R
// and Z. S is computed as a symmetric product (upper triangle + mirror): on every tested spectrum this
// changes the fp16 result by under 2% of its error while saving a third of the R update. Q is left a full
// product: it carries the accumulated iteration into the output, and mirroring its upper triangle drops
// the (fp16-rounding-sized) commutator of the stored Z and Q, which measurably raised the error on the
// hardest closed-form spectrum (2048 x 8192 with 205 singular values at 1 and the rest at 1e-4) close to
// the fp16 iteration's tolerance.
constexpr bool kMirrorS = true;
constexpr bool kMirrorQ = false;

// A matrix with m <= kFullSymMaxM computes its symmetric products (X X^T, R^2, the R update) in full
// instead of as upper triangle + mirror: at most 2 x 2 output tiles, so the extra tile runs beside the
// others, while a mirrored chunk costs its warp about three times a plain one (the transposed staging
// and the second store) on the phase's critical path. The choice depends on the matrix alone, so a
// matrix gets the same arithmetic whatever else is in the call.
constexpr int64_t kFullSymMaxM = 256;
int sym_flag(const MatInfo& mi) { return mi.m <= kFullSymMaxM ? 0 : kJobSymmetric; }

// Flags of a product whose operands are symmetric in exact arithmetic (R R, Z R, S Z; A A in the direct
// form). Mirrored, the stored operands are exactly symmetric and B read K-major (as B^T) is the same
// product. In full, the stored R and S are symmetric only up to fp16 rounding, so B is read MN-major and
// the product is the one the step defines: reading it as R R^T, Z R^T and S Z^T instead doubled the error
// of a 256 x 1024 Gram iteration over what fp16 storage alone causes.
int sym_product_flags(const MatInfo& mi) { return mi.m <= kFullSymMaxM ? kJobBMnMajor : kJobSymmetric; }

void build_gram_phases(Plan& pl, const std::vector<int>& restarts, int steps, const std::vector<int>& idx,
                       std::vector<std::vector<JobSpec>>& out, std::vector<int>& out_coef) {
  const int nm = static_cast<int>(pl.mats.size());
  const int q_mirror = kMirrorQ ? kJobSymmetric : 0;
  std::vector<char> is_restart(steps + 1, 0);
  for (int r : restarts)
    if (r > 0 && r < steps) is_restart[r] = 1;
  std::vector<size_t> X(nm), Xb(nm), Q(nm), Qb(nm);
  for (int i = 0; i < nm; ++i) X[i] = pl.mats[i].X, Xb[i] = pl.mats[i].Xb, Q[i] = pl.mats[i].Q, Qb[i] = pl.mats[i].Qb;

  auto push = [&](std::vector<JobSpec>&& ph, int coef) {
    if (!ph.empty()) {
      out.push_back(std::move(ph));
      out_coef.push_back(coef);
    }
  };
  auto gram_of_x = [&](int coef) {
    if (pl.key.shards > 0) {
      // Tensor-parallel form: each shard's X_t X_t^T as a full fp32 product into its own plane (what one
      // rank computes locally), then their fixed-order sum into R (the one all-reduce of the m x m Gram).
      std::vector<JobSpec> ph, red;
      for (int i : idx) {
        const MatInfo& mi = pl.mats[i];
        for (int t = 0; t < pl.key.shards; ++t) {
          const int64_t c0 = pl.shard_bounds[t], c1 = pl.shard_bounds[t + 1];
          const size_t xo = X[i] + static_cast<size_t>(c0) * sizeof(__half);
          JobSpec j = make_job(i, mi.m, mi.m, static_cast<int>(c1 - c0), kRecPlain, kJobFinal, xo, mi.ldx, xo, mi.ldx,
                               kNone, 0, kNone, 0);
          j.W = nullptr;
          j.w_off = mi.P + static_cast<size_t>(t) * mi.m * mi.ldp * sizeof(float);
          j.ldw = mi.ldp;
          ph.push_back(j);
        }
        JobSpec r = make_job(i, mi.m, mi.m, pl.key.shards, kRecPlain, kJobTpReduce, kNone, 0, kNone, 0, mi.P, mi.ldp,
                             mi.R, mi.ldm);
        red.push_back(r);
      }
      push(std::move(ph), coef);
      push(std::move(red), coef);
      return;
    }
    std::vector<JobSpec> ph;
    for (int i : idx) {
      const MatInfo& mi = pl.mats[i];
      ph.push_back(make_job(i, mi.m, mi.m, mi.n, kRecPlain, sym_flag(mi), X[i], mi.ldx, X[i], mi.ldx, kNone, 0,
                            mi.R, mi.ldm));
    }
    push(std::move(ph), coef);
  };

  gram_of_x(0);
  bool fresh = true;
  for (int k = 0; k < steps; ++k) {
    if (is_restart[k]) {
      std::vector<JobSpec> ph;
      for (int i : idx) {
        const MatInfo& mi = pl.mats[i];
        ph.push_back(make_job(i, mi.m, mi.n, mi.m, kRecPlain, kJobBMnMajor, Q[i], mi.ldm, X[i], mi.ldx, kNone, 0,
                              Xb[i], mi.ldx));
        std::swap(X[i], Xb[i]);
      }
      push(std::move(ph), k);
      gram_of_x(k);
      fresh = true;
    }
    {  // Z = b R + c R^2 (and the first Q after a (re)start)
      std::vector<JobSpec> ph;
      for (int i : idx) {
        const MatInfo& mi = pl.mats[i];
        ph.push_back(make_job(i, mi.m, mi.m, mi.m, kRecZ, sym_product_flags(mi) | (fresh ? kJobD2 : 0), mi.R,
                              mi.ldm, mi.R, mi.ldm, mi.R, mi.ldm, mi.Z, mi.ldm, fresh ? Q[i] : kNone));
      }
      push(std::move(ph), k);
    }
    const bool update_r = (k + 1 < steps) && !is_restart[k + 1];
    {
      std::vector<JobSpec> ph;
      for (int i : idx) {
        const MatInfo& mi = pl.mats[i];
        if (!fresh) {  // Q' = Z Q + a Q
          ph.push_back(make_job(i, mi.m, mi.m, mi.m, kRecAxpy, kJobBMnMajor | (q_mirror & sym_flag(mi)), mi.Z, mi.ldm,
                                Q[i], mi.ldm, Q[i], mi.ldm, Qb[i], mi.ldm));
        }
        if (update_r) {  // S = Z R + a R
          const int sf = kMirrorS ? sym_product_flags(mi) : kJobBMnMajor;
          ph.push_back(make_job(i, mi.m, mi.m, mi.m, kRecAxpy, sf, mi.Z, mi.ldm, mi.R, mi.ldm, mi.R, mi.ldm, mi.S,
                                mi.ldm));
        }
      }
      push(std::move(ph), k);
      if (!fresh)
        for (int i : idx) std::swap(Q[i], Qb[i]);
    }
    if (update_r) {  // R = S Z + a S (symmetric)
      std::vector<JobSpec> ph;
      for (int i : idx) {
        const MatInfo& mi = pl.mats[i];
        ph.push_back(make_job(i, mi.m, mi.m, mi.m, kRecAxpy, sym_product_flags(mi), mi.S, mi.ldm, mi.Z, mi.ldm, mi.S,
                              mi.ldm, mi.R, mi.ldm));
      }
      push(std::move(ph), k);
    }
    fresh = false;
  }
  {  // output: W <- w_alpha W + w_beta (Q X)
    std::vector<JobSpec> ph;
    for (int i : idx) {
      const MatInfo& mi = pl.mats[i];
      JobSpec j = make_job(i, mi.m, mi.n, mi.m, kRecPlain, kJobBMnMajor | kJobFinal | (mi.trans ? kJobFinalTrans : 0),
                           Q[i], mi.ldm, X[i], mi.ldx, kNone, 0, kNone, 0);
      j.W = mi.W;
      j.ldw = mi.cols;
      ph.push_back(j);
    }
    push(std::move(ph), steps - 1);
  }
}

void build_direct_phases(Plan& pl, int steps, const std::vector<int>& idx, std::vector<std::vector<JobSpec>>& out,
                         std::vector<int>& out_coef) {
  const int nm = static_cast<int>(pl.mats.size());
  std::vector<size_t> X(nm), Xb(nm);
  for (int i = 0; i < nm; ++i) X[i] = pl.mats[i].X, Xb[i] = pl.mats[i].Xb;
  for (int k = 0; k < steps; ++k) {
    std::vector<JobSpec> p1, p2, p3;
    for (int i : idx) {
      const MatInfo& mi = pl.mats[i];
      // A = X X^T (in R), B = b A + c A^2 (in Z)
      p1.push_back(make_job(i, mi.m, mi.m, mi.n, kRecPlain, sym_flag(mi), X[i], mi.ldx, X[i], mi.ldx, kNone, 0, mi.R,
                            mi.ldm));
      p2.push_back(make_job(i, mi.m, mi.m, mi.m, kRecZ, sym_product_flags(mi), mi.R, mi.ldm, mi.R, mi.ldm, mi.R,
                            mi.ldm, mi.Z, mi.ldm));
      if (k + 1 < steps) {  // X' = B X + a X
        p3.push_back(make_job(i, mi.m, mi.n, mi.m, kRecAxpy, kJobBMnMajor, mi.Z, mi.ldm, X[i], mi.ldx, X[i], mi.ldx,
                              Xb[i], mi.ldx));
      } else {
        JobSpec j = make_job(i, mi.m, mi.n, mi.m, kRecAxpy, kJobBMnMajor | kJobFinal | (mi.trans ? kJobFinalTrans : 0),
                             mi.Z, mi.ldm, X[i], mi.ldx, X[i], mi.ldx, kNone, 0);
        j.W = mi.W;
        j.ldw = mi.cols;
        p3.push_back(j);
      }
    }
    for (auto* ph : {&p1, &p2, &p3}) {
      if (ph->empty()) continue;
      out.push_back(std::move(*ph));
      out_coef.push_back(k);
    }
    if (k + 1 < steps)
      for (int i : idx) std::swap(X[i], Xb[i]);
  }
}

// Tile configuration of a launch: 128 x 128 single-CTA tiles when every product is at most 128 wide;
// 128 x 256 single-CTA tiles when every product has at most 128 rows (a 256-row pair tile would be half
// empty); otherwise 256 x 256 tiles on CTA pairs.
int pick_tile(int max_m, int max_n) {
  if (max_n <= 128) return kTileSingle128;
  if (max_m <= 128) return kTileSingle256;
  return kTilePair256;
}

// Output tiles of a launch under a tile configuration (symmetric products: upper-triangle tiles only).
int64_t count_tiles(const std::vector<JobSpec>& ph, int tile) {
  const int th = tile_rows(tile), tw = tile_cols(tile);
  int64_t n = 0;
  for (const JobSpec& js : ph) {
    const int tm_n = (js.M + th - 1) / th, tn_n = (js.N + tw - 1) / tw;
    for (int tm = 0; tm < tm_n; ++tm)
      for (int tn = 0; tn < tn_n; ++tn)
        if (!((js.flags & kJobSymmetric) && tn * tw + tw - 1 < tm * th)) ++n;
  }
  return n;
}

// A launch whose 256 x 256 pair tiles cannot fill the CTA pairs (a phase of a single matrix, or of a
// few, of moderate size) runs on 128 x 128 single-CTA tiles instead: about four times the work units,
// and half of a pair tile's epilogue per warp, for phases that would otherwise leave most SMs idle. When
// even those would occupy fewer than half of the SMs (`pair_units` is half the SM count), the tiles are
// halved again to 128 x 64: twice the work units, each with half the MMAs and one epilogue chunk per warp.
int launch_tile(const std::vector<JobSpec>& ph, int pair_units) {
  int max_m = 0, max_n = 0;
  for (const JobSpec& j : ph) max_m = std::max(max_m, j.M), max_n = std::max(max_n, j.N);
  int max_k = 0;
  for (const JobSpec& j : ph) max_k = std::max(max_k, j.K);
  int tile = pick_tile(max_m, max_n);
  // Short contractions (K <= 2048: the m x m products of matrices up to 2048 wide) keep the pair tiles down
  // to half the pairs (measured on one GB300: the full 2048 x 2048 products of a 2048 x 8192 matrix, 64
  // pair tiles, 31.7 -> 27.6 us per launch on pairs; the symmetric ones, 36 pair tiles, were slower on
  // pairs, 20.4 -> 26.5 us, so the floor stays above them).
  const int64_t pair_floor = max_k <= 2048 ? pair_units / 2 : pair_units;
  if (tile == kTilePair256 && count_tiles(ph, kTilePair256) < pair_floor) tile = kTileSingle128;
  if (tile == kTileSingle128 && count_tiles(ph, kTileSingle128) < pair_units) tile = kTileSingle64;
  return tile;
}

// Host-side plan: matrix layout, workspace offsets, phases, tiles. No device calls.
int build_plan_host(Plan& pl, const PlanKey& key, const std::vector<const void*>& G, const std::vector<float*>& Mom,
                    const std::vector<float*>& W, const std::vector<void*>& xout, int pair_units) {
  pl = Plan();
  pl.key = key;
  const int nm = static_cast<int>(key.rows.size());
  Layout lay;
  pl.off_rowmats = lay.take(sizeof(RowMat) * nm);
  pl.off_chunk = lay.take(sizeof(int64_t) * (nm + 1));
  pl.off_tilep = lay.take(sizeof(int64_t) * (nm + 1));
  pl.chunk_prefix.assign(nm + 1, 0);
  pl.tile_prefix.assign(nm + 1, 0);
  pl.mats.resize(nm);
  for (int i = 0; i < nm; ++i) {
    MatInfo& mi = pl.mats[i];
    mi.rows = key.rows[i];
    mi.cols = key.cols[i];
    mi.trans = mi.rows > mi.cols;
    mi.m = std::min(mi.rows, mi.cols);
    mi.n = std::max(mi.rows, mi.cols);
    mi.ldx = key.kind == kPlanMomNorm ? mi.n : round_up(mi.n, 8);
    mi.ldm = round_up(mi.m, 8);
    mi.G = G[i];
    mi.M = Mom[i];
    mi.W = W[i];
    mi.xout = xout[i];
    const int64_t numel = mi.rows * mi.cols;
    const int64_t chunk = momentum_chunk(numel);
    pl.chunk_prefix[i + 1] = pl.chunk_prefix[i] + (numel + chunk - 1) / chunk;
    pl.tile_prefix[i + 1] =
        pl.tile_prefix[i] + ((mi.rows + kCastTile - 1) / kCastTile) * ((mi.cols + kCastTile - 1) / kCastTile);
  }
  pl.nchunks = pl.chunk_prefix[nm];
  pl.ncast = pl.tile_prefix[nm];
  if (pl.nchunks >= (int64_t(1) << 31) || pl.ncast >= (int64_t(1) << 31))
    return fail(DMUON_ERR_UNSUPPORTED, "too many elements in one call");
  int64_t npartials = pl.nchunks;
  if (key.kind == kPlanNsTp) {
    // Shards along the long side, boundaries on multiples of 8 columns (16-byte aligned for TMA).
    const int64_t N = pl.mats[0].n;
    pl.shard_bounds.assign(key.shards + 1, N);
    for (int t = 0; t < key.shards; ++t) pl.shard_bounds[t] = (static_cast<int64_t>(t) * N / key.shards) / 8 * 8;
    pl.tp_slabs = static_cast<int>((pl.mats[0].m + kShardSlab - 1) / kShardSlab);
    npartials = std::max<int64_t>(npartials, static_cast<int64_t>(key.shards) * pl.tp_slabs);
  }
  pl.npartials = npartials;
  pl.off_partials = lay.take(sizeof(float) * npartials);
  pl.off_norms = lay.take(sizeof(float) * nm);
  pl.off_inv = lay.take(sizeof(float) * nm);
  // Every matrix small enough for the fused kernel: one launch runs the whole iteration.
  {
    bool all_small = key.kind != kPlanMomNorm && key.kind != kPlanNsTp;
    for (int i = 0; i < nm && all_small; ++i)
      all_small = pl.mats[i].m <= kSmallMaxM && pl.mats[i].n <= kSmallMaxN;
    pl.small_fused = all_small;
    for (int r : key.restarts)
      if (r > 0 && r < key.steps) pl.restart_mask |= 1u << r;
  }
  for (int i = 0; i < nm; ++i) {
    MatInfo& mi = pl.mats[i];
    // auto: direct where its flops (15 m^2 n + 5 m^3) are below Gram's (6 m^2 n + 17 m^3), i.e. n < 4m/3.
    mi.direct = key.backend == DMUON_NS_DIRECT || (key.backend == DMUON_NS_AUTO && 3 * mi.n < 4 * mi.m);
    const bool gram = !mi.direct;
    if (key.kind == kPlanMomNorm) continue;
    const size_t xbytes = sizeof(__half) * mi.m * mi.ldx;
    const size_t mbytes = sizeof(__half) * mi.m * mi.ldm;
    if (pl.small_fused) continue;  // the fused kernel reads M itself and keeps every operand on chip
    mi.X = lay.take(xbytes);
    mi.Xb = lay.take(xbytes);
    mi.R = lay.take(mbytes);
    mi.Z = lay.take(mbytes);
    if (gram) {
      mi.Q = lay.take(mbytes);
      mi.Qb = lay.take(mbytes);
      mi.S = lay.take(mbytes);
    }
    if (key.kind == kPlanNsTp) {
      mi.ldp = round_up(mi.m, 4);
      mi.P = lay.take(sizeof(float) * key.shards * mi.m * mi.ldp);
    }
  }
  pl.rowmats.resize(nm);
  int part = 0;
  for (int i = 0; i < nm; ++i) {
    const MatInfo& mi = pl.mats[i];
    RowMat& r = pl.rowmats[i];
    std::memset(&r, 0, sizeof(r));
    r.G = mi.G;
    r.M = mi.M;
    r.rows = mi.rows;
    r.cols = mi.cols;
    r.ldx = mi.ldx;
    r.gdtype = key.gdtype;
    r.trans = mi.trans ? 1 : 0;
    r.vec_ok = 1;  // pointers are validated 16-byte aligned
    r.chunk = momentum_chunk(mi.rows * mi.cols);
    r.part_begin = part;
    r.part_count = key.kind == kPlanNsTp ? key.shards * pl.tp_slabs
                                         : static_cast<int>(pl.chunk_prefix[i + 1] - pl.chunk_prefix[i]);
    part += r.part_count;
  }
  // Matrix groups: consecutive runs of gradient bytes. When the computation outruns the host link, the
  // first group's copy is what stays exposed, so the weights rise 1 : 2 : 3 from the start. When the link is
  // the slower side, the copies run back to back and what stays exposed is the computation still queued
  // after the last copy: the weights fall towards the end by a factor 0.85 per group (to 1.13 for the
  // last), so that each group's computation fits under the next group's copy down to a link at ~0.85 of
  // the computation's rate, and the last group is small. Weight of group g = min(ramp, fall) in hundredths;
  // boundary g sits at the cumulative weight of groups 0 .. g-1. One group for every other plan.
  {
    const int ng = (key.kind == kPlanMuon && !pl.small_fused) ? std::max(1, std::min(key.groups, nm)) : 1;
    auto weight = [ng](int g) -> int64_t {
      const int64_t ramp = std::min<int64_t>(100 * (g + 1), 300);
      const int64_t fall = static_cast<int64_t>(std::min(300.0, 113.0 * std::pow(1.0 / 0.85, ng - 1 - g)));
      return std::min(ramp, fall);
    };
    int64_t wsum = 0;
    for (int g = 0; g < ng; ++g) wsum += weight(g);
    pl.group_begin.assign(1, 0);
    int64_t total = 0;
    for (int i = 0; i < nm; ++i) total += pl.mats[i].rows * pl.mats[i].cols;
    int64_t run = 0, wcum = weight(0);  // cumulative weight up to the boundary being placed
    for (int i = 0; i < nm && static_cast<int>(pl.group_begin.size()) < ng; ++i) {
      run += pl.mats[i].rows * pl.mats[i].cols;
      const int g = static_cast<int>(pl.group_begin.size());  // boundary being placed
      // Close group g - 1 after matrix i once it holds its share, leaving a matrix for each later group.
      if (run * wsum >= total * wcum && nm - (i + 1) >= ng - g) {
        pl.group_begin.push_back(i + 1);
        wcum += weight(g);
      }
    }
    pl.group_begin.push_back(nm);
  }
  if (pl.small_fused) {
    pl.off_small = lay.take(sizeof(SmallJob) * nm, 256);
    pl.exec_flops = -1.0;
  } else if (key.kind != kPlanMomNorm) {
    for (size_t g = 0; g + 1 < pl.group_begin.size(); ++g) {
      std::vector<int> idx_gram, idx_direct;
      for (int i = pl.group_begin[g]; i < pl.group_begin[g + 1]; ++i)
        (pl.mats[i].direct ? idx_direct : idx_gram).push_back(i);
      std::vector<std::vector<JobSpec>> gp, dp;
      std::vector<int> gc, dc;
      if (!idx_gram.empty()) build_gram_phases(pl, key.restarts, key.steps, idx_gram, gp, gc);
      if (!idx_direct.empty()) build_direct_phases(pl, key.steps, idx_direct, dp, dc);
      // Both sequences advance step by step; the t-th launch of step k carries the t-th phase of step k
      // of each (their matrices are disjoint, and each sequence keeps its own order).
      size_t gi = 0, di = 0;
      for (int k = 0; k < key.steps; ++k) {
        std::vector<std::vector<JobSpec>> ga, da;
        while (gi < gp.size() && gc[gi] == k) ga.push_back(std::move(gp[gi++]));
        while (di < dp.size() && dc[di] == k) da.push_back(std::move(dp[di++]));
        for (size_t t = 0; t < std::max(ga.size(), da.size()); ++t) {
          std::vector<JobSpec> ph;
          if (t < ga.size()) ph.insert(ph.end(), ga[t].begin(), ga[t].end());
          if (t < da.size()) ph.insert(ph.end(), da[t].begin(), da[t].end());
          pl.phases.push_back(std::move(ph));
          pl.phase_coef.push_back(k);
          pl.phase_group.push_back(static_cast<int>(g));
        }
      }
    }
  }
  // Tiles: per launch, jobs in decreasing K (longest first), tiles row-major within a job.
  size_t njobs = 0;
  for (auto& ph : pl.phases) {
    std::stable_sort(ph.begin(), ph.end(), [](const JobSpec& x, const JobSpec& y) { return x.K > y.K; });
    njobs += ph.size();
  }
  for (size_t p = 0; p < pl.phases.size(); ++p) {
    const auto& ph = pl.phases[p];
    LaunchRec L;
    L.first_job = 0;  // filled below
    L.njobs = static_cast<int>(ph.size());
    L.tile = launch_tile(ph, pair_units);
    L.coef = pl.phase_coef[p];
    L.group = pl.phase_group[p];
    L.first_tile = static_cast<int>(pl.tiles.size());
    if (!ph.empty() && (ph[0].flags & kJobTpReduce)) {
      L.tp_reduce = 1;
      L.tp_mat = ph[0].mat;
      L.njobs = 0;
      L.ntiles = 0;
      pl.launches.push_back(L);
      continue;
    }
    const int th = tile_rows(L.tile), tw = tile_cols(L.tile);
    for (int j = 0; j < L.njobs; ++j) {
      const JobSpec& js = ph[j];
      const int tm_n = (js.M + th - 1) / th;
      const int tn_n = (js.N + tw - 1) / tw;
      // Tile order = the order the persistent workers pick tiles up, so it decides which tiles run at the
      // same time and share operands in L2. Walk the output column-wise within bands of `band` tile rows:
      // when the whole A operand fits comfortably in L2 (Q, Z, S, R and the small X of these products)
      // the band is every row, so each column block of B is read from DRAM once while A stays resident;
      // otherwise bands of 8 rows make the ~76 concurrent tiles a near-square block that shares both
      // operands.
      const int64_t a_bytes = static_cast<int64_t>(js.M) * js.K * 2;
      const int band = a_bytes <= (int64_t(40) << 20) ? tm_n : std::min(tm_n, 8);
      const size_t before = pl.tiles.size();
      for (int g0 = 0; g0 < tm_n; g0 += band)
        for (int tn = 0; tn < tn_n; ++tn)
          for (int tm = g0; tm < std::min(g0 + band, tm_n); ++tm) {
            if ((js.flags & kJobSymmetric) && tn * tw + tw - 1 < tm * th) continue;
            pl.tiles.push_back(GemmTile{j, tm, tn, 0});
          }
      const int64_t jt = static_cast<int64_t>(pl.tiles.size() - before);
      pl.exec_tiles += jt;
      pl.exec_flops += 2.0 * static_cast<double>(jt) * th * tw * static_cast<double>(round_up(js.K, kBK));
    }
    L.ntiles = static_cast<int>(pl.tiles.size()) - L.first_tile;
    pl.launches.push_back(L);
  }
  int acc = 0;
  for (auto& L : pl.launches) L.first_job = acc, acc += L.njobs;
  if (pl.tiles.size() >= (size_t(1) << 31)) return fail(DMUON_ERR_UNSUPPORTED, "too many tiles in one call");
  pl.off_jobs = lay.take(sizeof(GemmJob) * std::max<size_t>(njobs, 1), 256);
  pl.off_tiles = lay.take(sizeof(GemmTile) * std::max<size_t>(pl.tiles.size(), 1));
  pl.bytes = lay.off;
  return DMUON_OK;
}

// Place the plan in the device arena, resolve operand addresses, encode tensor maps and upload.
int bind_plan(DeviceState& ds, Plan& pl, cudaStream_t stream) {
  if (g_ws_limit && pl.bytes > g_ws_limit)
    return fail(DMUON_ERR_OOM, "workspace of %zu bytes exceeds the limit of %zu bytes", pl.bytes, g_ws_limit);
  DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize before re-planning");
  if (pl.bytes > ds.arena_bytes) {
    if (ds.arena) {
      cudaFree(ds.arena);
      ds.arena = nullptr;
      ds.arena_bytes = 0;
    }
    const size_t want = pl.bytes + (pl.bytes >> 4);
    if (cudaMalloc(&ds.arena, want) != cudaSuccess) {
      cudaGetLastError();
      ds.arena = nullptr;
      return fail(DMUON_ERR_OOM, "cudaMalloc of %zu workspace bytes failed", want);
    }
    ds.arena_bytes = want;
  }
  char* base = ds.arena;
  auto at = [&](size_t off) -> void* { return off == kNone ? nullptr : base + off; };
  for (size_t i = 0; i < pl.mats.size(); ++i) {
    pl.rowmats[i].X = static_cast<__half*>(pl.key.kind == kPlanMomNorm ? pl.mats[i].xout : at(pl.mats[i].X));
  }
  pl.jobs.clear();
  for (size_t p = 0; p < pl.phases.size(); ++p) {
    const int tile = pl.launches[p].tile;
    if (pl.launches[p].tp_reduce) continue;  // not a GEMM: no job records
    for (const JobSpec& js : pl.phases[p]) {
      GemmJob j;
      std::memset(&j, 0, sizeof(j));
      j.M = js.M, j.N = js.N, j.K = js.K;
      j.recipe = js.recipe, j.flags = js.flags;
      j.D = static_cast<__half*>(at(js.d));
      j.D2 = static_cast<__half*>(at(js.d2));
      j.E = static_cast<const __half*>(at(js.e));
      j.W = js.W ? js.W : static_cast<float*>(at(js.w_off));
      j.ldd = js.ldd, j.lde = js.lde, j.ldw = js.ldw;
      j.tiles_n = (js.N + tile_cols(tile) - 1) / tile_cols(tile);
      const char* err = nullptr;
      if (!encode_job_maps(j, at(js.a), js.lda, at(js.b), js.ldb, (js.flags & kJobBMnMajor) != 0, tile, &err) ||
          !encode_out_maps(j, &err))
        return fail(DMUON_ERR_CUDA, "%s", err);
      pl.jobs.push_back(j);
    }
  }
  if (pl.small_fused) {
    pl.small_jobs.assign(pl.mats.size(), SmallJob{});
    for (size_t i = 0; i < pl.mats.size(); ++i) {
      const MatInfo& mi = pl.mats[i];
      std::memset(&pl.small_jobs[i], 0, sizeof(SmallJob));
      const char* err = nullptr;
      const float* inv = reinterpret_cast<const float*>(base + pl.off_inv) + i;
      if (!encode_small_job(pl.small_jobs[i], mi.M, mi.cols, inv, mi.W, mi.cols, static_cast<int>(mi.m),
                            static_cast<int>(mi.n), mi.trans, mi.direct, &err))
        return fail(DMUON_ERR_CUDA, "%s", err);
    }
    DM_CUDA(cudaMemcpyAsync(base + pl.off_small, pl.small_jobs.data(), sizeof(SmallJob) * pl.small_jobs.size(),
                            cudaMemcpyHostToDevice, stream), "upload small-matrix jobs");
  }
  DM_CUDA(cudaMemcpyAsync(base + pl.off_rowmats, pl.rowmats.data(), sizeof(RowMat) * pl.rowmats.size(),
                          cudaMemcpyHostToDevice, stream), "upload matrix table");
  DM_CUDA(cudaMemcpyAsync(base + pl.off_chunk, pl.chunk_prefix.data(), sizeof(int64_t) * pl.chunk_prefix.size(),
                          cudaMemcpyHostToDevice, stream), "upload chunk table");
  DM_CUDA(cudaMemcpyAsync(base + pl.off_tilep, pl.tile_prefix.data(), sizeof(int64_t) * pl.tile_prefix.size(),
                          cudaMemcpyHostToDevice, stream), "upload tile table");
  if (!pl.jobs.empty())
    DM_CUDA(cudaMemcpyAsync(base + pl.off_jobs, pl.jobs.data(), sizeof(GemmJob) * pl.jobs.size(),
                            cudaMemcpyHostToDevice, stream), "upload job table");
  if (!pl.tiles.empty())
    DM_CUDA(cudaMemcpyAsync(base + pl.off_tiles, pl.tiles.data(), sizeof(GemmTile) * pl.tiles.size(),
                            cudaMemcpyHostToDevice, stream), "upload tile list");
  pl.bound = true;
  return DMUON_OK;
}

// Enqueue one run of a bound plan on `stream`. Groups run one after another, each its row-wise passes and
// then its Newton-Schulz launches. With `group_ready` the stream first waits for event g before group g
// (its gradients have arrived); with `group_read` event g is recorded once group g's momentum pass has
// read its gradients.
int run_plan(DeviceState& ds, const Plan& pl, const float* coeffs, float lr, float beta, float eps, float* norms_out,
             cudaStream_t stream, const cudaEvent_t* group_ready = nullptr, const cudaEvent_t* group_read = nullptr) {
  char* base = ds.arena;
  RowLaunch rl;
  rl.mats = reinterpret_cast<const RowMat*>(base + pl.off_rowmats);
  rl.nmats = static_cast<int>(pl.mats.size());
  rl.chunk_prefix = reinterpret_cast<const int64_t*>(base + pl.off_chunk);
  rl.tile_prefix = reinterpret_cast<const int64_t*>(base + pl.off_tilep);
  rl.partials = reinterpret_cast<float*>(base + pl.off_partials);
  rl.norms = reinterpret_cast<float*>(base + pl.off_norms);
  rl.inv = reinterpret_cast<float*>(base + pl.off_inv);
  rl.norms_out = norms_out;
  rl.beta = beta;
  rl.eps = eps;
  rl.status = ds.status;
  rl.check_status = ds.status;
  rl.npartials = pl.npartials;
  const GemmJob* jobs = reinterpret_cast<const GemmJob*>(base + pl.off_jobs);
  const GemmTile* tiles = reinterpret_cast<const GemmTile*>(base + pl.off_tiles);
  const bool overwrite = pl.key.kind == kPlanNs || pl.key.kind == kPlanNsTp;  // W = O, not W -= lr O
  size_t li = 0;
  const int ngroups = static_cast<int>(pl.group_begin.size()) - 1;
  for (int g = 0; g < ngroups; ++g) {
    const int i0 = pl.group_begin[g], i1 = pl.group_begin[g + 1];
    if (group_ready) DM_CUDA(cudaStreamWaitEvent(stream, group_ready[g], 0), "wait for a group's gradients");
    RowLaunch rg = rl;
    rg.mats += i0;
    rg.nmats = i1 - i0;
    rg.chunk_prefix += i0;
    rg.tile_prefix += i0;
    rg.norms += i0;
    rg.inv += i0;
    if (rg.norms_out) rg.norms_out += i0;
    rg.chunk_base = pl.chunk_prefix[i0];
    rg.tile_base = pl.tile_prefix[i0];
    const int64_t nchunks = pl.chunk_prefix[i1] - pl.chunk_prefix[i0];
    const int64_t ncast = pl.tile_prefix[i1] - pl.tile_prefix[i0];
    if (pl.key.kind == kPlanNsTp) {
      // One sum of squares per shard and row slab; their fixed-order sum is the one scalar all-reduce.
      const MatInfo& mi = pl.mats[0];
      ShardSumsqLaunch sl;
      std::memset(&sl, 0, sizeof(sl));
      sl.x = mi.M;
      sl.rows = mi.rows;
      sl.cols = mi.cols;
      sl.trans = mi.trans ? 1 : 0;
      sl.shards = pl.key.shards;
      sl.slabs = pl.tp_slabs;
      for (int t = 0; t <= pl.key.shards; ++t) sl.bounds[t] = pl.shard_bounds[t];
      sl.partials = rl.partials;
      DM_CUDA(timed(0, stream, [&] { return launch_shard_sumsq(sl, stream); }), "shard sum-of-squares launch");
    } else {
      DM_CUDA(timed(0, stream, [&] { return launch_momentum_sumsq(rg, nchunks, stream); }),
              "momentum/sum-of-squares launch");
    }
    if (group_read) DM_CUDA(cudaEventRecord(group_read[g], stream), "record a group's gradients as read");
    DM_CUDA(timed(1, stream, [&] { return launch_finalize_norms(rg, stream, true); }), "norm launch");
    // The fused small-matrix kernel normalises and casts as it reads M.
    if (!pl.small_fused)
      DM_CUDA(timed(2, stream, [&] { return launch_normalize_cast(rg, ncast, stream, true); }),
              "normalise/cast launch");
    if (pl.small_fused) {
      SmallLaunch sl;
      std::memset(&sl, 0, sizeof(sl));
      sl.jobs = reinterpret_cast<const SmallJob*>(base + pl.off_small);
      sl.njobs = static_cast<int>(pl.mats.size());
      sl.steps = pl.key.steps;
      sl.restart_mask = pl.restart_mask;
      for (int k = 0; k < 3 * pl.key.steps; ++k) sl.coef[k] = coeffs[k];
      sl.w_alpha = pl.key.kind == kPlanNs ? 0.f : 1.f;
      sl.w_beta = pl.key.kind == kPlanNs ? 1.f : -lr;
      sl.status = ds.status;
      DM_CUDA(timed(3, stream, [&] { return launch_ns_small(sl, ds.sms, stream); }), "small-matrix kernel launch");
      continue;  // a fused plan has one group
    }
    for (; li < pl.launches.size() && pl.launches[li].group == g; ++li) {
      const LaunchRec& L = pl.launches[li];
      if (L.tp_reduce) {
        const MatInfo& mi = pl.mats[L.tp_mat];
        TpReduceLaunch tr;
        tr.P = reinterpret_cast<const float*>(base + mi.P);
        tr.shards = pl.key.shards;
        tr.m = mi.m;
        tr.ldp = mi.ldp;
        tr.plane = mi.m * mi.ldp;
        tr.R = reinterpret_cast<__half*>(base + mi.R);
        tr.ldr = mi.ldm;
        DM_CUDA(timed(5, stream, [&] { return launch_tp_reduce(tr, stream); }), "shard Gram reduction launch");
        continue;
      }
      GemmLaunch gl;
      std::memset(&gl, 0, sizeof(gl));
      gl.jobs = jobs + L.first_job;
      gl.tiles = tiles + L.first_tile;
      gl.ntiles = L.ntiles;
      gl.njobs = L.njobs;
      gl.a = coeffs[3 * L.coef + 0];
      gl.b = coeffs[3 * L.coef + 1];
      gl.c = coeffs[3 * L.coef + 2];
      gl.w_alpha = overwrite ? 0.f : 1.f;
      gl.w_beta = overwrite ? 1.f : -lr;
      gl.status = ds.status;
      const int units = std::min(L.ntiles, gemm_max_units(L.tile, ds.sms));
      DM_CUDA(timed(3, stream, [&] { return launch_gemm(gl, L.tile, units, stream); }), "tensor-core GEMM launch");
    }
  }
  return DMUON_OK;
}

// Make the device's cached plan the one for `key`, building and binding it if it is not. Caller holds g_mu.
// *rebuilt tells whether it had to be built.
int ensure_plan(DeviceState& ds, const PlanKey& key, const std::vector<const void*>& G, const std::vector<float*>& Mom,
                const std::vector<float*>& W, const std::vector<void*>& xout, cudaStream_t stream,
                bool* rebuilt = nullptr) {
  if (rebuilt) *rebuilt = false;
  if (ds.plan.bound && ds.plan.key == key) return DMUON_OK;
  if (rebuilt) *rebuilt = true;
  ++ds.plan_serial;
  ds.plan = Plan();
  int st = build_plan_host(ds.plan, key, G, Mom, W, xout, gemm_max_units(kTilePair256, ds.sms));
  if (st != DMUON_OK) return st;
  st = bind_plan(ds, ds.plan, stream);
  if (st != DMUON_OK) ds.plan = Plan();
  return st;
}

void drop_graph(DeviceState& ds) {
  if (ds.graph) cudaGraphExecDestroy(ds.graph);
  ds.graph = nullptr;
  ds.graph_key = GraphKey();
}

// Capture one run of the cached plan on the library's private stream and instantiate it. On any failure
// the capture is abandoned, the error cleared, and false returned: the caller launches directly instead.
bool capture_plan(DeviceState& ds, const float* coeffs, float lr, float beta, float eps, float* norms_out) {
  drop_graph(ds);
  if (!ds.capture_stream && cudaStreamCreateWithFlags(&ds.capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    ds.capture_stream = nullptr;
    cudaGetLastError();
    return false;
  }
  if (cudaStreamBeginCapture(ds.capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int st = run_plan(ds, ds.plan, coeffs, lr, beta, eps, norms_out, ds.capture_stream);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(ds.capture_stream, &g);
  bool ok = st == DMUON_OK && e == cudaSuccess && g != nullptr &&
            cudaGraphInstantiate(&ds.graph, g, 0) == cudaSuccess;
  if (g) cudaGraphDestroy(g);
  if (!ok) {
    ds.graph = nullptr;
    cudaGetLastError();
  }
  return ok;
}

// Shared body of the plan-based entry points that take device buffers. With graph replay on (the default),
// no per-launch timing and a caller's stream that is not itself being captured, the second consecutive call with the same plan and the same arguments captures
// the plan's launches as a CUDA graph, and every further such call launches that graph on the caller's
// stream: the same kernels with the same arguments, so the same results bit for bit, with the per-launch
// issue cost of the chain of small dependent launches taken off. Any other call launches directly.
int plan_and_run(const PlanKey& key, const std::vector<const void*>& G, const std::vector<float*>& Mom,
                 const std::vector<float*>& W, const std::vector<void*>& xout, const float* coeffs, float lr,
                 float beta, float eps, float* norms_out, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = current_device(&ds);
  if (st != DMUON_OK) return st;
  st = ensure_plan(*ds, key, G, Mom, W, xout, stream);
  if (st != DMUON_OK) return st;
  // A stream the caller is capturing gets the launches themselves, so that they become part of the
  // caller's graph.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;
  }
  if (!g_graphs || g_timing || cs != cudaStreamCaptureStatusNone)
    return run_plan(*ds, ds->plan, coeffs, lr, beta, eps, norms_out, stream);
  GraphKey gk;
  gk.valid = true;
  gk.plan_serial = ds->plan_serial;
  gk.coeffs.assign(coeffs, coeffs + 3 * ds->plan.key.steps);
  gk.lr = lr, gk.beta = beta, gk.eps = eps, gk.norms_out = norms_out;
  if (!(ds->graph && ds->graph_key == gk)) {
    const bool repeat = ds->last_key == gk;
    ds->last_key = gk;
    if (!repeat || !capture_plan(*ds, coeffs, lr, beta, eps, norms_out))
      return run_plan(*ds, ds->plan, coeffs, lr, beta, eps, norms_out, stream);
    ds->graph_key = gk;
  }
  DM_CUDA(cudaGraphLaunch(ds->graph, stream), "cudaGraphLaunch of the cached plan");
  return DMUON_OK;
}

// The copy stream and at least `n` pairs of group events of the host-gradient pipeline.
int ensure_pipeline(DeviceState& ds, size_t n) {
  if (!ds.copy_stream) DM_CUDA(cudaStreamCreateWithFlags(&ds.copy_stream, cudaStreamNonBlocking), "create copy stream");
  if (!ds.entry) DM_CUDA(cudaEventCreateWithFlags(&ds.entry, cudaEventDisableTiming), "create event");
  while (ds.copied.size() < n) {
    cudaEvent_t a = nullptr, b = nullptr;
    DM_CUDA(cudaEventCreateWithFlags(&a, cudaEventDisableTiming), "create event");
    if (cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
      cudaEventDestroy(a);
      return fail(DMUON_ERR_CUDA, "create event failed");
    }
    ds.copied.push_back(a);
    ds.read.push_back(b);
  }
  return DMUON_OK;
}

int check_matrix_list(int count, const int64_t* rows, const int64_t* cols);

// The device gather table for these host -> device copies (built once per set of pointers and sizes).
// Leaves ds.gather_ok false when some host pointer is not readable by the device (pageable memory on a
// device without host page-table access): the caller then copies with the copy engines.
int ensure_gather(DeviceState& ds, int count, const void* const* src, void* const* dst, const int64_t* bytes,
                  cudaStream_t stream) {
  std::vector<uintptr_t> key;
  key.reserve(3 * static_cast<size_t>(count));
  for (int i = 0; i < count; ++i) {
    key.push_back(reinterpret_cast<uintptr_t>(src[i]));
    key.push_back(reinterpret_cast<uintptr_t>(dst[i]));
    key.push_back(static_cast<uintptr_t>(bytes[i]));
  }
  int dev = 0, pageable = 0;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
    cudaGetLastError();
    pageable = 0;
  }
  // The device address of host pointer i, or null when the device cannot read it.
  auto resolve = [&](int i) -> const void* {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, src[i]) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer) return a.devicePointer;  // page-locked, mapped
    if (a.type == cudaMemoryTypeUnregistered && pageable) return src[i];          // through host page tables
    return nullptr;
  };
  if (key == ds.gather_key) {
    // With host page-table access every host address stays readable; without it the same addresses may
    // have been unpinned since the table was built, so they are checked again.
    if (ds.gather_ok && !pageable) {
      for (int i = 0; i < count; ++i)
        if (!resolve(i)) {
          ds.gather_key.clear();
          ds.gather_ok = false;
          return DMUON_OK;
        }
    }
    return DMUON_OK;
  }
  ds.gather_key.clear();
  ds.gather_ok = false;
  std::vector<GatherItem> items(count);
  std::vector<int64_t> prefix(count + 1, 0);
  for (int i = 0; i < count; ++i) {
    const void* s = resolve(i);
    if (!s) {
      ds.gather_key = key;  // remember the outcome for this pointer set
      return DMUON_OK;
    }
    items[i] = GatherItem{s, dst[i], bytes[i]};
    prefix[i + 1] = prefix[i] + (bytes[i] + kGatherChunk - 1) / kGatherChunk;
  }
  if (prefix[count] >= (int64_t(1) << 31)) return fail(DMUON_ERR_UNSUPPORTED, "too many gradient bytes for one gather");
  const size_t need = sizeof(GatherItem) * count + 256 + sizeof(int64_t) * (count + 1);
  // An earlier call, possibly on another stream, may still be reading the old table.
  if (ds.gather_buf) DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize before replacing the gather table");
  if (need > ds.gather_bytes) {
    if (ds.gather_buf) {
      cudaFree(ds.gather_buf);
      ds.gather_buf = nullptr;
      ds.gather_bytes = 0;
    }
    if (cudaMalloc(&ds.gather_buf, need) != cudaSuccess) {
      cudaGetLastError();
      ds.gather_buf = nullptr;
      return fail(DMUON_ERR_OOM, "cudaMalloc of the %zu-byte gather table failed", need);
    }
    ds.gather_bytes = need;
  }
  const size_t off_prefix = (sizeof(GatherItem) * count + 255) / 256 * 256;
  DM_CUDA(cudaMemcpyAsync(ds.gather_buf, items.data(), sizeof(GatherItem) * count, cudaMemcpyHostToDevice, stream),
          "upload gather items");
  DM_CUDA(cudaMemcpyAsync(ds.gather_buf + off_prefix, prefix.data(), sizeof(int64_t) * (count + 1),
                          cudaMemcpyHostToDevice, stream),
          "upload gather prefix");
  DM_CUDA(cudaStreamSynchronize(stream), "cudaStreamSynchronize after the gather table upload");
  ds.gather_chunks = prefix[count];
  ds.gather_key = key;
  ds.gather_ok = true;
  return DMUON_OK;
}

// Validation and key of dmuon_muon_step (shared with dmuon_muon_step_host).
int muon_key(int count, float* const* params, const void* const* grads, int grad_dtype, float* const* momenta,
             const int64_t* rows, const int64_t* cols, float* norms_out, float lr, float beta, const float* coeffs,
             int steps, const int* restarts, int n_restarts, int backend, float eps, PlanKey& key,
             std::vector<const void*>& G, std::vector<float*>& Mo, std::vector<float*>& W) {
  int st = check_matrix_list(count, rows, cols);
  if (st != DMUON_OK) return st;
  if (!params || !grads || !momenta) return fail(DMUON_ERR_INVALID_ARG, "params/grads/momenta arrays are NULL");
  if (grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16)
    return fail(DMUON_ERR_INVALID_ARG, "grad_dtype must be DMUON_F32 (0) or DMUON_BF16 (1)");
  if (!std::isfinite(lr) || !std::isfinite(beta)) return fail(DMUON_ERR_INVALID_ARG, "lr and beta must be finite");
  if (norms_out && (reinterpret_cast<uintptr_t>(norms_out) & 3))
    return fail(DMUON_ERR_INVALID_ARG, "norms_out must be 4-byte aligned");
  st = check_ns_args(coeffs, steps, restarts, n_restarts, backend, eps);
  if (st != DMUON_OK) return st;
  key = PlanKey();
  key.kind = kPlanMuon;
  key.backend = backend;
  key.steps = steps;
  key.gdtype = grad_dtype;
  if (backend != DMUON_NS_DIRECT) key.restarts.assign(restarts, restarts + n_restarts);
  key.rows.assign(rows, rows + count);
  key.cols.assign(cols, cols + count);
  G.assign(count, nullptr);
  Mo.assign(count, nullptr);
  W.assign(count, nullptr);
  for (int i = 0; i < count; ++i) {
    if (!params[i] || !grads[i] || !momenta[i]) return fail(DMUON_ERR_INVALID_ARG, "matrix %d has a NULL pointer", i);
    if (!aligned16(params[i]) || !aligned16(grads[i]) || !aligned16(momenta[i]))
      return fail(DMUON_ERR_INVALID_ARG, "matrix %d: device buffers must be 16-byte aligned", i);
    G[i] = grads[i];
    Mo[i] = momenta[i];
    W[i] = params[i];
    key.ptrs.push_back(reinterpret_cast<uintptr_t>(params[i]));
    key.ptrs.push_back(reinterpret_cast<uintptr_t>(grads[i]));
    key.ptrs.push_back(reinterpret_cast<uintptr_t>(momenta[i]));
  }
  return DMUON_OK;
}

int check_matrix_list(int count, const int64_t* rows, const int64_t* cols) {
  if (count < 1) return fail(DMUON_ERR_INVALID_ARG, "count must be >= 1");
  if (!rows || !cols) return fail(DMUON_ERR_INVALID_ARG, "rows/cols arrays are NULL");
  for (int i = 0; i < count; ++i) {
    if (rows[i] < 1 || cols[i] < 1)
      return fail(DMUON_ERR_INVALID_ARG, "matrix %d has a non-positive size (%lld x %lld)", i, (long long)rows[i],
                  (long long)cols[i]);
    if (rows[i] > kMaxDim || cols[i] > kMaxDim)
      return fail(DMUON_ERR_UNSUPPORTED, "matrix %d is larger than %lld in one dimension", i, (long long)kMaxDim);
  }
  return DMUON_OK;
}

}  // namespace

int set_error(int status, const char* message) { return fail(status, "%s", message); }

}  // namespace dmuon

using namespace dmuon;

extern "C" {

int dmuon_ns(float* x, int64_t m, int64_t n, const float* coeffs, int steps, const int* restarts, int n_restarts,
             int backend, float eps, void* cuda_stream) {
  try {
    if (!x) return fail(DMUON_ERR_INVALID_ARG, "x is NULL");
    if (!aligned16(x)) return fail(DMUON_ERR_INVALID_ARG, "x must be 16-byte aligned");
    int st = check_matrix_list(1, &m, &n);
    if (st != DMUON_OK) return st;
    st = check_ns_args(coeffs, steps, restarts, n_restarts, backend, eps);
    if (st != DMUON_OK) return st;
    PlanKey key;
    key.kind = kPlanNs;
    key.backend = backend;
    key.steps = steps;
    key.gdtype = 0;
    if (backend != DMUON_NS_DIRECT) key.restarts.assign(restarts, restarts + n_restarts);
    key.rows = {m};
    key.cols = {n};
    key.ptrs = {reinterpret_cast<uintptr_t>(x)};
    return plan_and_run(key, {nullptr}, {x}, {x}, {nullptr}, coeffs, 0.f, 0.f, eps, nullptr,
                        static_cast<cudaStream_t>(cuda_stream));
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_ns_tp(float* x, int64_t m, int64_t n, int shards, const float* coeffs, int steps, const int* restarts,
                int n_restarts, float eps, void* cuda_stream) {
  try {
    if (!x) return fail(DMUON_ERR_INVALID_ARG, "x is NULL");
    if (!aligned16(x)) return fail(DMUON_ERR_INVALID_ARG, "x must be 16-byte aligned");
    int st = check_matrix_list(1, &m, &n);
    if (st != DMUON_OK) return st;
    st = check_ns_args(coeffs, steps, restarts, n_restarts, DMUON_NS_GRAM, eps);
    if (st != DMUON_OK) return st;
    if (shards < 1 || shards > kMaxShards) return fail(DMUON_ERR_INVALID_ARG, "shards must be in [1, %d]", kMaxShards);
    if (std::max(m, n) < 16 * static_cast<int64_t>(shards))
      return fail(DMUON_ERR_INVALID_ARG, "each shard needs at least 16 columns of the long side");
    PlanKey key;
    key.kind = kPlanNsTp;
    key.backend = DMUON_NS_GRAM;
    key.steps = steps;
    key.shards = shards;
    key.restarts.assign(restarts, restarts + n_restarts);
    key.rows = {m};
    key.cols = {n};
    key.ptrs = {reinterpret_cast<uintptr_t>(x)};
    return plan_and_run(key, {nullptr}, {x}, {x}, {nullptr}, coeffs, 0.f, 0.f, eps, nullptr,
                        static_cast<cudaStream_t>(cuda_stream));
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_muon_step(int count, float* const* params, const void* const* grads, int grad_dtype, float* const* momenta,
                    const int64_t* rows, const int64_t* cols, float* norms_out, float lr, float beta,
                    const float* coeffs, int steps, const int* restarts, int n_restarts, int backend, float eps,
                    void* cuda_stream) {
  try {
    PlanKey key;
    std::vector<const void*> G;
    std::vector<float*> Mo, W;
    const int st = muon_key(count, params, grads, grad_dtype, momenta, rows, cols, norms_out, lr, beta, coeffs, steps,
                            restarts, n_restarts, backend, eps, key, G, Mo, W);
    if (st != DMUON_OK) return st;
    std::vector<void*> xo(count, nullptr);
    return plan_and_run(key, G, Mo, W, xo, coeffs, lr, beta, eps, norms_out, static_cast<cudaStream_t>(cuda_stream));
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_muon_step_host(int count, float* const* params, const void* const* grads_host, void* const* grads,
                         int grad_dtype, float* const* momenta, const int64_t* rows, const int64_t* cols,
                         float* norms_out, float lr, float beta, const float* coeffs, int steps, const int* restarts,
                         int n_restarts, int backend, float eps, int groups, void* cuda_stream) {
  try {
    PlanKey key;
    std::vector<const void*> G;
    std::vector<float*> Mo, W;
    int st = muon_key(count, params, reinterpret_cast<const void* const*>(grads), grad_dtype, momenta, rows, cols,
                      norms_out, lr, beta, coeffs, steps, restarts, n_restarts, backend, eps, key, G, Mo, W);
    if (st != DMUON_OK) return st;
    if (!grads_host) return fail(DMUON_ERR_INVALID_ARG, "grads_host is NULL");
    for (int i = 0; i < count; ++i)
      if (!grads_host[i]) return fail(DMUON_ERR_INVALID_ARG, "matrix %d has a NULL host gradient", i);
    if (groups > kMaxGroups) return fail(DMUON_ERR_INVALID_ARG, "groups must be at most %d", kMaxGroups);
    const size_t esize = grad_dtype == DMUON_BF16 ? 2 : 4;
    if (groups <= 0) {
      // One group per ~1 GiB of gradients, at most 16: fewer groups leave more of the copy or of the
      // computation exposed at the ends, and every group adds one launch per phase (measured: twelve
      // groups of the 8B set add under 2% to the GEMM time).
      int64_t bytes = 0;
      for (int i = 0; i < count; ++i) bytes += rows[i] * cols[i] * static_cast<int64_t>(esize);
      const int64_t per_group = int64_t(1) << 30;
      groups = static_cast<int>(std::min<int64_t>(16, std::max<int64_t>(1, (bytes + per_group - 1) / per_group)));
    }
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    st = current_device(&ds);
    if (st != DMUON_OK) return st;
    // Many small matrices (here a copy-engine call per matrix costs more host time than its transfer):
    // one gather launch on cuda_stream reads every gradient out of host memory, then the step runs as
    // one group. Needs device-readable host memory; otherwise the copy engines below.
    {
      int64_t total = 0;
      for (int i = 0; i < count; ++i) total += rows[i] * cols[i] * static_cast<int64_t>(esize);
      if (count >= kGatherMinCount && total < static_cast<int64_t>(count) * kGatherMaxAvgBytes) {
        std::vector<int64_t> nbytes(count);
        for (int i = 0; i < count; ++i) nbytes[i] = rows[i] * cols[i] * static_cast<int64_t>(esize);
        st = ensure_gather(*ds, count, grads_host, grads, nbytes.data(), stream);
        if (st != DMUON_OK) return st;
        if (ds->gather_ok) {
          key.groups = 1;
          std::vector<void*> xo(count, nullptr);
          st = ensure_plan(*ds, key, G, Mo, W, xo, stream);
          if (st != DMUON_OK) return st;
          const size_t off_prefix = (sizeof(GatherItem) * count + 255) / 256 * 256;
          DM_CUDA(launch_h2d_gather(reinterpret_cast<const GatherItem*>(ds->gather_buf),
                                    reinterpret_cast<const int64_t*>(ds->gather_buf + off_prefix), count,
                                    ds->gather_chunks, stream),
                  "gradient gather launch");
          return run_plan(*ds, ds->plan, coeffs, lr, beta, eps, norms_out, stream);
        }
      }
    }
    key.groups = groups;
    const size_t prev_groups = ds->copied.size();
    bool rebuilt = false;
    std::vector<void*> xo(count, nullptr);
    st = ensure_plan(*ds, key, G, Mo, W, xo, stream, &rebuilt);
    if (st != DMUON_OK) return st;
    const Plan& pl = ds->plan;
    const size_t ng = pl.group_begin.size() - 1;
    st = ensure_pipeline(*ds, ng);
    if (st != DMUON_OK) return st;
    // Copies follow everything already enqueued on the caller's stream, and each group's copy follows the
    // previous call's momentum pass over the same buffers (every previous group when the grouping changed).
    DM_CUDA(cudaEventRecord(ds->entry, stream), "record entry event");
    DM_CUDA(cudaStreamWaitEvent(ds->copy_stream, ds->entry, 0), "order copies after the caller's stream");
    if (rebuilt)
      for (size_t g = 0; g < prev_groups; ++g)
        DM_CUDA(cudaStreamWaitEvent(ds->copy_stream, ds->read[g], 0), "order copies after the previous call");
    for (size_t g = 0; g < ng; ++g) {
      DM_CUDA(cudaStreamWaitEvent(ds->copy_stream, ds->read[g], 0), "order copies after the previous call");
      for (int i = pl.group_begin[g]; i < pl.group_begin[g + 1]; ++i)
        DM_CUDA(cudaMemcpyAsync(grads[i], grads_host[i], static_cast<size_t>(rows[i] * cols[i]) * esize,
                                cudaMemcpyHostToDevice, ds->copy_stream),
                "gradient copy");
      DM_CUDA(cudaEventRecord(ds->copied[g], ds->copy_stream), "record a group's copy");
    }
    return run_plan(*ds, pl, coeffs, lr, beta, eps, norms_out, stream, ds->copied.data(), ds->read.data());
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_momentum_normalize(int count, const void* const* grads, int grad_dtype, float* const* momenta,
                             const int64_t* rows, const int64_t* cols, void* const* x_out, float* norms_out,
                             float beta, float eps, void* cuda_stream) {
  try {
    int st = check_matrix_list(count, rows, cols);
    if (st != DMUON_OK) return st;
    if (!momenta || !x_out || !norms_out) return fail(DMUON_ERR_INVALID_ARG, "momenta/x_out/norms_out are NULL");
    if (grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16)
      return fail(DMUON_ERR_INVALID_ARG, "grad_dtype must be DMUON_F32 (0) or DMUON_BF16 (1)");
    if (!std::isfinite(beta) || !std::isfinite(eps) || !(eps >= 0.f))
      return fail(DMUON_ERR_INVALID_ARG, "beta must be finite and eps finite and >= 0");
    PlanKey key;
    key.kind = kPlanMomNorm;
    key.gdtype = grad_dtype;
    key.rows.assign(rows, rows + count);
    key.cols.assign(cols, cols + count);
    std::vector<const void*> G(count);
    std::vector<float*> Mo(count), W(count, nullptr);
    std::vector<void*> xo(count);
    for (int i = 0; i < count; ++i) {
      const void* g = grads ? grads[i] : nullptr;
      if (!momenta[i] || !x_out[i]) return fail(DMUON_ERR_INVALID_ARG, "matrix %d has a NULL pointer", i);
      if (!aligned16(momenta[i]) || (g && !aligned16(g)) || !aligned16(x_out[i]))
        return fail(DMUON_ERR_INVALID_ARG, "matrix %d: device buffers must be 16-byte aligned", i);
      G[i] = g;
      Mo[i] = momenta[i];
      xo[i] = x_out[i];
      key.ptrs.push_back(reinterpret_cast<uintptr_t>(g));
      key.ptrs.push_back(reinterpret_cast<uintptr_t>(momenta[i]));
      key.ptrs.push_back(reinterpret_cast<uintptr_t>(x_out[i]));
    }
    const float dummy[3] = {0.f, 0.f, 0.f};
    return plan_and_run(key, G, Mo, W, xo, dummy, 0.f, beta, eps, norms_out, static_cast<cudaStream_t>(cuda_stream));
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   int b_trans, const void* E, int64_t lde, void* D, int64_t ldd, float alpha, float beta, float gamma,
                   int symmetric, void* cuda_stream) {
  try {
    if (M < 1 || N < 1 || K < 1) return fail(DMUON_ERR_INVALID_ARG, "M, N, K must be >= 1");
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return fail(DMUON_ERR_UNSUPPORTED, "dimension above %lld", (long long)kMaxDim);
    if (!A || !B || !D) return fail(DMUON_ERR_INVALID_ARG, "A, B and D must not be NULL");
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (E && !aligned16(E)))
      return fail(DMUON_ERR_INVALID_ARG, "A, B, D, E must be 16-byte aligned");
    if (symmetric && M != N) return fail(DMUON_ERR_INVALID_ARG, "symmetric output needs M == N");
    const int64_t b_row = b_trans ? K : N;
    if (lda < K || ldb < b_row || ldd < N || (E && lde < N))
      return fail(DMUON_ERR_INVALID_ARG, "a leading dimension is smaller than its row length");
    if ((lda | ldb | ldd | (E ? lde : 0)) & 7)
      return fail(DMUON_ERR_INVALID_ARG, "leading dimensions must be multiples of 8 elements (16 bytes)");
    if (!std::isfinite(alpha) || !std::isfinite(beta) || !std::isfinite(gamma))
      return fail(DMUON_ERR_INVALID_ARG, "alpha, beta, gamma must be finite");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    int st = current_device(&ds);
    if (st != DMUON_OK) return st;
    const int tile = pick_tile(static_cast<int>(M), static_cast<int>(N));
    GemmLaunch gl;
    std::memset(&gl, 0, sizeof(gl));
    GemmJob& j = gl.single;
    j.M = static_cast<int>(M), j.N = static_cast<int>(N), j.K = static_cast<int>(K);
    j.recipe = kRecCustom;
    j.flags = (symmetric ? kJobSymmetric : 0) | (b_trans ? 0 : kJobBMnMajor);
    j.D = static_cast<__half*>(D);
    j.E = static_cast<const __half*>(E);
    j.ldd = ldd, j.lde = E ? lde : 0;
    j.tiles_n = static_cast<int>((N + tile_cols(tile) - 1) / tile_cols(tile));
    const char* err = nullptr;
    if (!encode_job_maps(j, A, lda, B, ldb, !b_trans, tile, &err) || !encode_out_maps(j, &err))
      return fail(DMUON_ERR_CUDA, "%s", err);
    gl.jobs = nullptr;
    gl.tiles = nullptr;
    gl.tiles_m = static_cast<int>((M + tile_rows(tile) - 1) / tile_rows(tile));
    const int64_t ntiles = static_cast<int64_t>(gl.tiles_m) * j.tiles_n;
    if (ntiles >= (int64_t(1) << 31)) return fail(DMUON_ERR_UNSUPPORTED, "too many tiles");
    gl.ntiles = static_cast<int>(ntiles);
    gl.alpha = alpha, gl.beta = E ? beta : 0.f, gl.gamma = gamma;
    gl.status = ds->status;
    const int units = static_cast<int>(std::min<int64_t>(ntiles, gemm_max_units(tile, ds->sms)));
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    DM_CUDA(timed(3, stream, [&] { return launch_gemm(gl, tile, units, stream); }), "tensor-core GEMM launch");
    return DMUON_OK;
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_check_status(void* cuda_stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = current_device(&ds);
  if (st != DMUON_OK) return st;
  DM_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)), "cudaStreamSynchronize");
  unsigned word = 0;
  DM_CUDA(cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost), "read device status");
  if (word) DM_CUDA(cudaMemset(ds->status, 0, sizeof(unsigned)), "clear device status");
  if (word & kDevTimeout) return fail(DMUON_ERR_TIMEOUT, "a device-side bounded wait gave up; results are invalid");
  if (word & kDevRange)
    return fail(DMUON_ERR_RANGE, "a device-side range check failed (checked build): an index or tile outside its "
                                 "table or matrix was skipped; results are invalid");
  if (word & kDevNonfinite) return fail(DMUON_ERR_NONFINITE, "an fp16 intermediate overflowed or was NaN");
  return DMUON_OK;
}

int dmuon_adamw_step(int count, float* const* params, const void* const* grads, int grad_dtype, float* const* exp_avg,
                     float* const* exp_avg_sq, const int64_t* numels, double lr, double beta1, double beta2,
                     double eps, double weight_decay, int step, void* cuda_stream) {
  try {
    if (count < 1) return fail(DMUON_ERR_INVALID_ARG, "count must be >= 1");
    if (!params || !grads || !exp_avg || !exp_avg_sq || !numels)
      return fail(DMUON_ERR_INVALID_ARG, "params/grads/exp_avg/exp_avg_sq/numels arrays are NULL");
    if (grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16)
      return fail(DMUON_ERR_INVALID_ARG, "grad_dtype must be DMUON_F32 (0) or DMUON_BF16 (1)");
    if (step < 1) return fail(DMUON_ERR_INVALID_ARG, "step must be >= 1");
    if (!std::isfinite(lr) || !std::isfinite(weight_decay) || !std::isfinite(eps) || !(eps >= 0.0) ||
        !(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
      return fail(DMUON_ERR_INVALID_ARG, "lr, weight_decay, eps must be finite (eps >= 0) and betas in [0, 1)");
    std::vector<uintptr_t> key;
    key.reserve(5 * static_cast<size_t>(count));
    for (int i = 0; i < count; ++i) {
      if (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i])
        return fail(DMUON_ERR_INVALID_ARG, "tensor %d has a NULL pointer", i);
      if (numels[i] < 1) return fail(DMUON_ERR_INVALID_ARG, "tensor %d has no elements", i);
      key.push_back(reinterpret_cast<uintptr_t>(params[i]));
      key.push_back(reinterpret_cast<uintptr_t>(grads[i]));
      key.push_back(reinterpret_cast<uintptr_t>(exp_avg[i]));
      key.push_back(reinterpret_cast<uintptr_t>(exp_avg_sq[i]));
      key.push_back(static_cast<uintptr_t>(numels[i]));
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    int st = current_device(&ds);
    if (st != DMUON_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    AdamPlan& ap = ds->adam;
    if (!(ap.bound && ap.key == key && ap.gdtype == grad_dtype)) {
      ap.bound = false;
      ap.key = key;
      ap.gdtype = grad_dtype;
      ap.tensors.assign(count, AdamTensor{});
      ap.chunk_prefix.assign(count + 1, 0);
      for (int i = 0; i < count; ++i) {
        AdamTensor& t = ap.tensors[i];
        t.p = params[i];
        t.g = grads[i];
        t.m = exp_avg[i];
        t.v = exp_avg_sq[i];
        t.numel = numels[i];
        t.vec_ok = aligned16(params[i]) && aligned16(grads[i]) && aligned16(exp_avg[i]) && aligned16(exp_avg_sq[i]);
        ap.chunk_prefix[i + 1] = ap.chunk_prefix[i] + (numels[i] + kAdamChunkElems - 1) / kAdamChunkElems;
      }
      if (ap.chunk_prefix[count] >= (int64_t(1) << 31)) return fail(DMUON_ERR_UNSUPPORTED, "too many elements");
      Layout lay;
      lay.take(sizeof(AdamTensor) * count);
      ap.off_prefix = lay.take(sizeof(int64_t) * (count + 1));
      if (lay.off > ap.buf_bytes) {
        DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize before re-planning");
        if (ap.buf) cudaFree(ap.buf);
        ap.buf = nullptr;
        ap.buf_bytes = 0;
        if (cudaMalloc(&ap.buf, lay.off) != cudaSuccess) {
          cudaGetLastError();
          ap.buf = nullptr;
          return fail(DMUON_ERR_OOM, "cudaMalloc of %zu bytes for the AdamW table failed", lay.off);
        }
        ap.buf_bytes = lay.off;
      }
      DM_CUDA(cudaMemcpyAsync(ap.buf, ap.tensors.data(), sizeof(AdamTensor) * count, cudaMemcpyHostToDevice, stream),
              "upload AdamW table");
      DM_CUDA(cudaMemcpyAsync(ap.buf + ap.off_prefix, ap.chunk_prefix.data(), sizeof(int64_t) * (count + 1),
                              cudaMemcpyHostToDevice, stream),
              "upload AdamW chunk table");
      ap.bound = true;
    }
    AdamLaunch a;
    std::memset(&a, 0, sizeof(a));
    a.tensors = reinterpret_cast<const AdamTensor*>(ap.buf);
    a.ntensors = count;
    a.chunk_prefix = reinterpret_cast<const int64_t*>(ap.buf + ap.off_prefix);
    a.gdtype = grad_dtype;
    a.decay = static_cast<float>(1.0 - lr * weight_decay);
    a.step_size = static_cast<float>(lr / (1.0 - std::pow(beta1, step)));
    a.inv_bc2 = static_cast<float>(1.0 / std::sqrt(1.0 - std::pow(beta2, step)));
    a.beta1 = static_cast<float>(beta1);
    a.one_minus_beta1 = static_cast<float>(1.0 - beta1);
    a.beta2 = static_cast<float>(beta2);
    a.one_minus_beta2 = static_cast<float>(1.0 - beta2);
    a.eps = static_cast<float>(eps);
    a.status = ds->status;
    const int64_t nchunks = ap.chunk_prefix[count];
    DM_CUDA(timed(4, stream, [&] { return launch_adamw(a, nchunks, stream); }), "AdamW launch");
    return DMUON_OK;
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_set_graph_replay(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_graphs = on != 0;
  return DMUON_OK;
}

int dmuon_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& t : g_timed) {
    cudaEventSynchronize(t.stop);
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_timed.clear();
  g_timing = on != 0;
  return DMUON_OK;
}

int dmuon_timing_read(double* ms_out, int64_t* launches_out) {
  if (!ms_out || !launches_out) return fail(DMUON_ERR_INVALID_ARG, "output arrays are NULL");
  std::lock_guard<std::mutex> lock(g_mu);
  for (int c = 0; c < DMUON_TIMING_CLASSES; ++c) ms_out[c] = 0.0, launches_out[c] = 0;
  int st = DMUON_OK;
  for (auto& t : g_timed) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
    if (e != cudaSuccess && st == DMUON_OK) st = cuda_fail(e, "timing events");
    if (t.cls >= 0 && t.cls < DMUON_TIMING_CLASSES) {
      ms_out[t.cls] += ms;
      launches_out[t.cls] += 1;
    }
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_timed.clear();
  return st;
}

int dmuon_timing_read_launches(int max_launches, double* ms_out, int* class_out, int* count_out) {
  if (!count_out || max_launches < 0 || (max_launches > 0 && (!ms_out || !class_out)))
    return fail(DMUON_ERR_INVALID_ARG, "output arrays are NULL or max_launches is negative");
  std::lock_guard<std::mutex> lock(g_mu);
  int st = DMUON_OK;
  int i = 0;
  for (auto& t : g_timed) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
    if (e != cudaSuccess && st == DMUON_OK) st = cuda_fail(e, "timing events");
    if (i < max_launches) {
      ms_out[i] = ms;
      class_out[i] = t.cls;
    }
    ++i;
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  *count_out = i;
  g_timed.clear();
  return st;
}

int dmuon_selftest_bounded_wait(int64_t limit_ns, void* cuda_stream) {
  if (limit_ns < 1000000 || limit_ns > 2000000000)
    return fail(DMUON_ERR_INVALID_ARG, "limit_ns must be in [1e6, 2e9] (1 ms to 2 s)");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = current_device(&ds);
  if (st != DMUON_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  DM_CUDA(launch_selftest_wait(ds->status, static_cast<unsigned long long>(limit_ns), stream), "self-test launch");
  return DMUON_OK;
}

int dmuon_selftest_range_check(void* cuda_stream) {
  if (!DMUON_DEVICE_CHECKS)
    return fail(DMUON_ERR_UNSUPPORTED, "this library was built without device-side range checks "
                                       "(libdmuon_checked.so has them)");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = current_device(&ds);
  if (st != DMUON_OK) return st;
  // One GEMM launch whose only tile lies outside its product (a product with no rows): the checks skip it
  // in every role before any operand is touched and record the failure.
  GemmLaunch gl;
  std::memset(&gl, 0, sizeof(gl));
  gl.single.M = 0;
  gl.single.N = 128;
  gl.single.K = 64;
  gl.single.tiles_n = 1;
  gl.tiles_m = 1;
  gl.ntiles = 1;
  gl.status = ds->status;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  DM_CUDA(launch_gemm(gl, kTileSingle128, 1, stream), "range self-test launch");
  return DMUON_OK;
}

int dmuon_plan_info(double* exec_flops_out, int64_t* tiles_out, int* gemm_launches_out) {
  if (!exec_flops_out || !tiles_out || !gemm_launches_out) return fail(DMUON_ERR_INVALID_ARG, "outputs are NULL");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  int st = current_device(&ds);
  if (st != DMUON_OK) return st;
  if (!ds->plan.bound) return fail(DMUON_ERR_INVALID_ARG, "no call has been planned on this device");
  const Plan& pl = ds->plan;
  *exec_flops_out = pl.exec_flops;
  *tiles_out = pl.exec_tiles;
  int n = 0;
  for (const LaunchRec& L : pl.launches) n += L.tp_reduce ? 0 : 1;
  *gemm_launches_out = pl.small_fused ? 1 : n;
  return DMUON_OK;
}

const char* dmuon_last_error(void) { return t_last_error.c_str(); }

const char* dmuon_version(void) {
  return DMUON_DEVICE_CHECKS ? "dmuon-gb300 0.2.0 (sm_103a, device-side range checks)" : "dmuon-gb300 0.2.0 (sm_103a)";
}

int dmuon_set_workspace_limit(size_t bytes) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_ws_limit = bytes;
  return DMUON_OK;
}

int dmuon_workspace_size(int count, const int64_t* rows, const int64_t* cols, int backend, size_t* bytes_out) {
  try {
    if (!bytes_out) return fail(DMUON_ERR_INVALID_ARG, "bytes_out is NULL");
    int st = check_matrix_list(count, rows, cols);
    if (st != DMUON_OK) return st;
    if (backend != DMUON_NS_DIRECT && backend != DMUON_NS_GRAM && backend != DMUON_NS_AUTO)
      return fail(DMUON_ERR_INVALID_ARG, "bad backend");
    PlanKey key;
    key.kind = kPlanMuon;
    key.backend = backend;
    key.steps = 5;
    key.restarts = {2};
    key.rows.assign(rows, rows + count);
    key.cols.assign(cols, cols + count);
    Plan pl;
    std::vector<const void*> G(count, nullptr);
    std::vector<float*> Mo(count, nullptr), W(count, nullptr);
    std::vector<void*> xo(count, nullptr);
    // No device here: the tile choice (and so the tile table's size) assumes GB300's 76 CTA pairs.
    st = build_plan_host(pl, key, G, Mo, W, xo, 76);
    if (st != DMUON_OK) return st;
    *bytes_out = pl.bytes;
    return DMUON_OK;
  } catch (const std::exception& e) {
    return fail(DMUON_ERR_OOM, "host exception: %s", e.what());
  }
}

int dmuon_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return DMUON_OK;
  DeviceState& ds = g_dev[dev];
  if (ds.arena) {
    DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    DM_CUDA(cudaFree(ds.arena), "cudaFree(workspace)");
  }
  ds.arena = nullptr;
  ds.arena_bytes = 0;
  ds.plan = Plan();
  ++ds.plan_serial;
  drop_graph(ds);
  ds.last_key = GraphKey();
  if (ds.adam.buf) {
    DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    DM_CUDA(cudaFree(ds.adam.buf), "cudaFree(AdamW table)");
  }
  ds.adam = AdamPlan();
  if (ds.gather_buf) {
    DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    DM_CUDA(cudaFree(ds.gather_buf), "cudaFree(gather table)");
  }
  ds.gather_buf = nullptr;
  ds.gather_bytes = 0;
  ds.gather_key.clear();
  ds.gather_ok = false;
  return DMUON_OK;
}

}  // extern "C"
