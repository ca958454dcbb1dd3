// Allocation-free variant of the momentum / normalise stage for one matrix.
//
// Who needs it: callers whose device memory belongs to someone else -- a framework's caching
// allocator or a fixed memory plan that must account for every byte -- and callers that cannot afford
// the device-wide synchronisation cudaMalloc / cudaFree may cause. dmuon_momentum_normalize grows a
// library workspace with cudaMalloc on first use; this entry point instead keeps its scratch (the matrix
// descriptor, the per-chunk partial sums of M^2 and the norm) in the fixed-size device array below, which
// every GPU that loads the library holds until the process exits.
//
// The array's name in host code is only a host-side stand-in, never a device address: the first call
// on each device (with that device current) asks the runtime for the real address with
// cudaGetSymbolAddress and keeps it, together with the unique id of the CUDA context it was found in.
// When a later call finds another context current on that device (after cudaDeviceReset, for instance,
// the runtime loads the library's device image into a new primary context, where the array may sit
// elsewhere) the address is looked up again. All calls share the one array, so calls whose work
// overlaps on the GPU (different streams, or different host threads on one stream without ordering)
// race on it. Nothing in it needs to start at zero: every call rewrites the descriptor, every partial
// sum it reads and the norm before using them.
#include <cmath>
#include <cstring>
#include <mutex>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
namespace {

constexpr int64_t kNoAllocMaxChunks = (int64_t(DMUON_NOALLOC_MAX_ELEMS) + kChunkElems - 1) / kChunkElems;

struct NoAllocScratch {
  RowMat mat;
  int64_t chunk_prefix[2];
  int64_t tile_prefix[2];
  float norm[1];
  float inv[1];
  float partials[kNoAllocMaxChunks];
};

// Scratch of the allocation-free entry point: sizeof(NoAllocScratch) bytes (about 16.5 KB).
static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

// Writes this call's descriptor tables into the scratch (one thread).
__global__ void noalloc_describe_kernel(NoAllocScratch* s, RowMat mat, int64_t nchunks, int64_t ntiles) {
  s->mat = mat;
  s->chunk_prefix[0] = 0;
  s->chunk_prefix[1] = nchunks;
  s->tile_prefix[0] = 0;
  s->tile_prefix[1] = ntiles;
}

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
NoAllocScratch* g_noalloc_addr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (cuCtxGetCurrent + cuCtxGetId from the driver
// entry points); 0 when no context is current or the driver cannot say.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(a);
      get_id = reinterpret_cast<GetIdFn>(b);
    } else {
      cudaGetLastError();
    }
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device: looked up once per device and context.
int scratch_address(NoAllocScratch** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(DMUON_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return set_error(DMUON_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_noalloc_addr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return set_error(DMUON_ERR_CUDA, "cudaDeviceGetAttribute failed");
    if (major != 10 || minor != 3) return set_error(DMUON_ERR_UNSUPPORTED, "libdmuon is built for sm_103a (GB300)");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return set_error(DMUON_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    g_noalloc_addr[dev] = static_cast<NoAllocScratch*>(ptr);
    g_noalloc_ctx[dev] = current_context_id();  // the lookup made the device's primary context current
  }
  *out = g_noalloc_addr[dev];
  return DMUON_OK;
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" int dmuon_momentum_normalize_noalloc(const void* grad, int grad_dtype, float* momentum, int64_t rows,
                                                int64_t cols, void* x_out, float* norm_out, float beta, float eps,
                                                void* cuda_stream) {
  if (!momentum || !x_out || !norm_out) return set_error(DMUON_ERR_INVALID_ARG, "momentum, x_out and norm_out must not be NULL");
  if (grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16)
    return set_error(DMUON_ERR_INVALID_ARG, "grad_dtype must be DMUON_F32 (0) or DMUON_BF16 (1)");
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(momentum) || misaligned(x_out) || (grad && misaligned(grad)) ||
      (reinterpret_cast<uintptr_t>(norm_out) & 3))
    return set_error(DMUON_ERR_INVALID_ARG, "device buffers must be 16-byte aligned (norm_out 4-byte)");
  if (rows < 1 || cols < 1) return set_error(DMUON_ERR_INVALID_ARG, "rows and cols must be >= 1");
  if (rows > DMUON_NOALLOC_MAX_ELEMS || cols > DMUON_NOALLOC_MAX_ELEMS || rows * cols > DMUON_NOALLOC_MAX_ELEMS)
    return set_error(DMUON_ERR_INVALID_ARG,
                     "matrix has more than DMUON_NOALLOC_MAX_ELEMS (268435456) elements, the fixed scratch limit "
                     "of dmuon_momentum_normalize_noalloc; use dmuon_momentum_normalize");
  if (!std::isfinite(eps) || !(eps >= 0.f) || !std::isfinite(beta))
    return set_error(DMUON_ERR_INVALID_ARG, "beta must be finite and eps finite and >= 0");
  NoAllocScratch* s = nullptr;
  int st = scratch_address(&s);
  if (st != DMUON_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  RowMat mat;
  memset(&mat, 0, sizeof(mat));
  mat.G = grad;
  mat.M = momentum;
  mat.X = static_cast<__half*>(x_out);
  mat.rows = rows;
  mat.cols = cols;
  mat.trans = rows > cols ? 1 : 0;
  mat.ldx = rows > cols ? rows : cols;
  mat.gdtype = grad_dtype;
  mat.vec_ok = 1;
  const int64_t numel = rows * cols;
  const int64_t nchunks = (numel + kChunkElems - 1) / kChunkElems;
  const int64_t ntiles = ((rows + kCastTile - 1) / kCastTile) * ((cols + kCastTile - 1) / kCastTile);
  mat.part_begin = 0;
  mat.part_count = static_cast<int>(nchunks);

  noalloc_describe_kernel<<<1, 1, 0, stream>>>(s, mat, nchunks, ntiles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(DMUON_ERR_CUDA, cudaGetErrorString(e));
  RowLaunch rl;
  rl.mats = &s->mat;
  rl.nmats = 1;
  rl.chunk_prefix = s->chunk_prefix;
  rl.tile_prefix = s->tile_prefix;
  rl.partials = s->partials;
  rl.norms = s->norm;
  rl.inv = s->inv;
  rl.norms_out = norm_out;
  rl.beta = beta;
  rl.eps = eps;
  rl.npartials = nchunks;
  if ((e = launch_momentum_sumsq(rl, nchunks, stream)) != cudaSuccess ||
      (e = launch_finalize_norms(rl, stream)) != cudaSuccess ||
      (e = launch_normalize_cast(rl, ntiles, stream)) != cudaSuccess)
    return set_error(DMUON_ERR_CUDA, cudaGetErrorString(e));
  return DMUON_OK;
}
