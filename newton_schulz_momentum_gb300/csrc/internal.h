// Internal types shared by the host layer (api.cu) and the kernels (gemm_tc.cu, rowwise.cu).
// Nothing here is part of the public C ABI in include/dmuon.h.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace dmuon {

// Bits of the device status word (read and cleared by dmuon_check_status).
enum : unsigned {
  kDevTimeout = 1u,    // a bounded mbarrier wait gave up; the launch's results are invalid
  kDevNonfinite = 2u,  // an fp16 store overflowed or was NaN
  kDevRange = 4u,      // checked build: an index or tile outside its table or matrix was skipped
};

// Device-side range checks: compiled in with -DDMUON_DEVICE_CHECKS=1 (the checked build,
// libdmuon_checked.so), left out otherwise. dev_check(ok, status) is ok in the checked build, recording
// kDevRange in *status (when given) if it is false, so the caller can skip the access; in the regular
// build it is always true and the condition costs nothing.
#ifndef DMUON_DEVICE_CHECKS
#define DMUON_DEVICE_CHECKS 0
#endif
#if defined(__CUDACC__)
__device__ __forceinline__ bool dev_check(bool ok, unsigned* status) {
#if DMUON_DEVICE_CHECKS
  if (!ok && status != nullptr) atomicOr(status, kDevRange);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}
#endif

// ------------------------------------------------------------------------------------------------
// Grouped tensor-core GEMM (gemm_tc.cu).
//
// One launch processes a list of tiles drawn from a list of jobs; each job is one product
// acc = A * Bop on one matrix, with its own operand tensor maps and epilogue. Tiles are 128 x BN
// (BN = 128 or 256) output blocks with fp32 accumulators in tensor memory.
// ------------------------------------------------------------------------------------------------

constexpr int kBM = 128;  // tile rows (tcgen05 M)
constexpr int kBK = 64;   // K per pipeline stage: 64 fp16 = one 128-byte swizzled row

// How the epilogue forms v from the accumulator, the optional addend E and the step's (a, b, c).
enum EpiRecipe : int {
  kRecPlain = 0,   // v = acc
  kRecZ = 1,       // v = c * acc + b * E          (Z = b R + c R^2; acc = R R, E = R)
  kRecAxpy = 2,    // v = acc + a * E              (Z Q + a Q, Z R + a R, S Z + a S, B X + a X)
  kRecCustom = 3,  // v = alpha * acc + beta * E + gamma * [i == j]
};

enum JobFlags : int {
  kJobBMnMajor = 1,    // Bop is stored K x N (N contiguous): B tile loaded MN-major
  kJobSymmetric = 2,   // upper-triangle tiles only; store D[i][j] and D[j][i] for j >= i
  kJobFinal = 4,       // write fp32 W = w_alpha * W + w_beta * v instead of an fp16 D
  kJobFinalTrans = 8,  // with kJobFinal: W is stored transposed (W[j][i])
  kJobD2 = 16,         // also store D2 = v + a * [i == j] (the first Q after a (re)start)
  kJobTmaW = 32,       // with kJobFinal: tmW is valid (W rows 16-byte aligned) -> TMA store / reduce-add
};

struct alignas(128) GemmJob {
  CUtensorMap tmA;   // A: M rows x K cols (K contiguous), box {64, 128}
  CUtensorMap tmB;   // B: N x K (K contiguous) box {64, BN}, or K x N (N contiguous) box {64, 64}
  CUtensorMap tmD;   // D (fp16, M x N, ldd), box {32, 32}, 64-byte swizzle: epilogue TMA stores
  CUtensorMap tmD2;  // D2, same geometry
  CUtensorMap tmW;   // W (fp32, caller orientation), box {32, 32}, 128-byte swizzle (kJobTmaW)
  __half* D;
  __half* D2;
  const __half* E;
  float* W;
  int64_t ldd, lde, ldw;  // leading dimensions in elements
  int M, N, K;
  int recipe, flags;
  int tiles_n;  // number of BN-wide column tiles
};
static_assert(sizeof(GemmJob) % 128 == 0, "GemmJob must keep the tensor maps 128-byte aligned in arrays");

struct GemmTile {
  int job, tm, tn, pad_;
};

struct GemmLaunch {
  // Either a device job table + tile list (grouped launch), or, when jobs == nullptr, the one job in
  // `single` with tiles enumerated row-major over tiles_m x single.tiles_n.
  GemmJob single;
  const GemmJob* jobs;
  const GemmTile* tiles;
  int ntiles;
  int tiles_m;
  float a, b, c;             // this step's coefficients (recipes kRecZ / kRecAxpy / kJobD2)
  float alpha, beta, gamma;  // kRecCustom
  float w_alpha, w_beta;     // kJobFinal
  unsigned* status;
  int njobs;                 // entries of `jobs` (checked build: every tile's job index is tested against it)
};

// Output tile configurations of the GEMM kernel.
enum TileConfig : int {
  kTileSingle128 = 0,  // one CTA, 128 x 128 tile (products with N <= 128)
  kTileSingle256 = 1,  // one CTA, 128 x 256 tile
  kTilePair256 = 2,    // a CTA pair (cluster of 2, tcgen05 cta_group::2), 256 x 256 tile
  kTileSingle64 = 3,   // one CTA, 128 x 64 tile (launches whose 128 x 128 tiles would fill under half the SMs)
};
inline int tile_rows(int tile) { return tile == kTilePair256 ? 256 : 128; }
inline int tile_cols(int tile) { return tile == kTileSingle128 ? 128 : tile == kTileSingle64 ? 64 : 256; }
inline int tile_ctas(int tile) { return tile == kTilePair256 ? 2 : 1; }

// Largest number of persistent workers of a tile configuration that fit on the device at once.
int gemm_max_units(int tile, int sms);
// Launch one grouped GEMM with `units` persistent workers (CTAs, or CTA pairs for kTilePair256).
cudaError_t launch_gemm(const GemmLaunch& p, int tile, int units, cudaStream_t stream);
// Encode the operand tensor maps of a job (host). a/b point to fp16 row-major matrices.
// b_mn_major selects the K x N storage of Bop. Returns false (with a message) on failure.
bool encode_job_maps(GemmJob& job, const void* a, int64_t lda, const void* b, int64_t ldb,
                     bool b_mn_major, int tile, const char** err);
// Encode the epilogue maps of a job from its D, D2, W pointers and leading dimensions (host). Sets
// kJobTmaW when the W map can be built (16-byte aligned base and rows); otherwise the final update
// falls back to direct stores.
bool encode_out_maps(GemmJob& job, const char** err);

// Encode a 2-D tensor map (host): `inner` contiguous elements per row, `outer` rows `row_bytes` apart.
bool encode_tensor_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_outer, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                      const char** err);

// ------------------------------------------------------------------------------------------------
// Fused Newton-Schulz for small matrices (ns_small.cu): m <= 128 rows and n <= 512 columns after
// orientation. One persistent CTA per SM takes one matrix at a time and runs the whole iteration in
// shared memory and tensor memory, ending with the fused weight update: ONE launch for all matrices.
// ------------------------------------------------------------------------------------------------

constexpr int kSmallMaxM = 128;
constexpr int kSmallMaxN = 512;

struct alignas(128) SmallJob {
  CUtensorMap tmW;  // W (fp32, caller orientation), box {32, 32}, 128-byte swizzle (when tma_w)
  const float* M;   // momentum (fp32, caller orientation, leading dimension ldm): X = fp16(M * *inv)
  const float* inv; // 1 / (||M||_F + eps), written by the norm pass
  float* W;
  int64_t ldm, ldw;
  int m, n;
  int trans;   // M and W are stored transposed (the matrix was oriented)
  int vec_m;   // M and its rows 16-byte aligned
  int tma_w;   // tmW valid; otherwise direct stores
  int direct;  // 1: direct iteration, 0: Gram iteration
};

struct SmallLaunch {
  const SmallJob* jobs;
  int njobs;
  int steps;
  unsigned restart_mask;  // bit k: restart before step k (k > 0)
  float coef[3 * 16];     // (a, b, c) per step
  float w_alpha, w_beta;  // W = w_alpha W + w_beta O  (w_alpha 0 or 1)
  unsigned* status;
};

bool encode_small_job(SmallJob& job, const float* M, int64_t ldm, const float* inv, float* W, int64_t ldw, int m,
                      int n, bool trans, bool direct, const char** err);
cudaError_t launch_ns_small(const SmallLaunch& p, int sms, cudaStream_t stream);

// ------------------------------------------------------------------------------------------------
// Row-wise (HBM-bound) kernels (rowwise.cu): momentum + sum of squares, norm finalisation,
// normalise + fp16 cast (+ transpose to the m <= n orientation).
// ------------------------------------------------------------------------------------------------

constexpr int kChunkElems = 65536;  // elements per momentum CTA (multiple of 8 * 256)
constexpr int kCastTile = 64;       // normalise/cast tiles are 64 x 64 elements of M

struct RowMat {
  const void* G;  // gradient (fp32 or bf16), or null: M is only read
  float* M;       // momentum, rows x cols fp32
  __half* X;      // oriented fp16 output, m x n with leading dimension ldx
  int64_t rows, cols, ldx;
  int gdtype;     // 0 fp32, 1 bf16
  int trans;      // rows > cols
  int vec_ok;     // pointers and rows allow 16-byte vector access
  int part_begin, part_count;  // this matrix's partial sums
  int pad_;
  // Elements per momentum chunk of this matrix in the bulk-copy pass (a multiple of 4096). It depends on
  // the matrix alone, so a matrix's norm is summed the same way whatever else is in the call. The
  // vector-load pass of the allocation-free entry uses kChunkElems.
  int64_t chunk;
};

// The bulk-copy pass's chunk for a matrix of `numel` elements: one chunk up to kChunkElems, 64 chunks up
// to 64 kChunkElems (a lone matrix of moderate size is spread over many CTAs instead of a few making
// long trips through their copy ring), kChunkElems beyond.
inline int64_t momentum_chunk(int64_t numel) {
  if (numel <= kChunkElems) return kChunkElems;
  int64_t c = kChunkElems;
  while (c > 4096 && c * 64 > numel) c /= 2;
  return c;
}

struct RowLaunch {
  const RowMat* mats;
  int nmats;
  const int64_t* chunk_prefix;  // nmats + 1 exclusive prefix of momentum chunks
  const int64_t* tile_prefix;   // nmats + 1 exclusive prefix of 64 x 64 cast tiles
  float* partials;              // one per chunk
  float* norms;                 // one per matrix: ||M||_F
  float* inv;                   // one per matrix: 1 / (||M||_F + eps)
  float* norms_out;             // optional user copy of norms
  float beta, eps;
  // A launch may cover a contiguous group of the plan's matrices: `mats`, both prefixes, `norms`,
  // `inv` and `norms_out` then point at the group's first entry, and block b works on momentum chunk
  // chunk_base + b (cast tile tile_base + b) of the plan-wide numbering. Zero for a whole-plan launch.
  int64_t chunk_base = 0, tile_base = 0;
  // Device status word for bounded waits. With it the momentum pass streams M and G through a
  // shared-memory ring of bulk copies; without it (the allocation-free entry) it uses vector loads.
  unsigned* status = nullptr;
  int64_t npartials = 0;  // entries of `partials` (checked build: every partial index is tested against it)
  unsigned* check_status = nullptr;  // checked build: where range failures are recorded (may be null)
};

// ------------------------------------------------------------------------------------------------
// Fused AdamW over many tensors (adamw.cu).
// ------------------------------------------------------------------------------------------------

constexpr int kAdamChunkElems = 16384;  // elements per AdamW CTA (multiple of 8 * 256)

struct AdamTensor {
  float* p;
  const void* g;
  float* m;
  float* v;
  int64_t numel;
  int vec_ok;  // every pointer 16-byte aligned
  int pad_;
};

struct AdamLaunch {
  const AdamTensor* tensors;
  int ntensors;
  const int64_t* chunk_prefix;  // ntensors + 1 exclusive prefix of chunks
  int gdtype;                   // 0 fp32, 1 bf16
  float decay, step_size, inv_bc2, beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
  unsigned* status;             // checked build: where range failures are recorded
};

cudaError_t launch_adamw(const AdamLaunch& a, int64_t nchunks, cudaStream_t stream);

// ------------------------------------------------------------------------------------------------
// Tensor-parallel emulation of the Gram form (rowwise.cu): the matrix split into column shards along
// its long side, per-shard sums of squares and per-shard Gram matrices reduced in a fixed order.
// ------------------------------------------------------------------------------------------------

constexpr int kMaxShards = 64;
constexpr int kShardSlab = 64;  // rows (short side) per shard sum-of-squares CTA

struct ShardSumsqLaunch {
  const float* x;  // caller matrix, rows x cols fp32
  int64_t rows, cols;
  int trans;  // rows > cols: the long side (sharded) is the row index
  int shards, slabs;
  int64_t bounds[kMaxShards + 1];  // shard boundaries along the long side
  float* partials;                 // shards * slabs, shard-major
};

// R[i][j] = fp16(sum over t of P_t[min(i,j)][max(i,j)]), t = 0 .. shards-1 in order.
struct TpReduceLaunch {
  const float* P;  // shards planes of m x ldp fp32
  int shards;
  int64_t m, ldp, plane;
  __half* R;
  int64_t ldr;
};

cudaError_t launch_shard_sumsq(const ShardSumsqLaunch& p, cudaStream_t stream);
cudaError_t launch_tp_reduce(const TpReduceLaunch& p, cudaStream_t stream);

// Host -> device gather of many small buffers in one launch (dmuon_muon_step_host with many small
// matrices, where one copy-engine call per matrix would leave the host issuing copies): item i copies
// bytes[i] from src[i], a device-accessible address of host memory, to dst[i]. Items are split into
// kGatherChunk-byte chunks numbered by `prefix` (n + 1 entries).
struct GatherItem {
  const void* src;
  void* dst;
  int64_t bytes;
};
constexpr int64_t kGatherChunk = 65536;
cudaError_t launch_h2d_gather(const GatherItem* items, const int64_t* prefix, int n, int64_t nchunks,
                              cudaStream_t stream);

// Diagnostic: one bounded wait on an mbarrier phase that nothing completes (records kDevTimeout).
cudaError_t launch_selftest_wait(unsigned* status, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_momentum_sumsq(const RowLaunch& p, int64_t nchunks, cudaStream_t stream);
// programmatic: launched with programmatic stream serialisation (the planned path; the kernels wait for
// the preceding grid themselves). The bulk momentum kernel (RowLaunch.status set) always is.
cudaError_t launch_finalize_norms(const RowLaunch& p, cudaStream_t stream, bool programmatic = false);
cudaError_t launch_normalize_cast(const RowLaunch& p, int64_t ntiles, cudaStream_t stream, bool programmatic = false);

// Record `message` as the calling thread's last error (returned by dmuon_last_error) and return status.
int set_error(int status, const char* message);

}  // namespace dmuon
