// Fused Newton-Schulz for small matrices: the whole iteration of one matrix (m <= 128 rows, n <= 512
// columns after orientation) in one CTA, ending with the weight update -- one launch for every matrix of
// the call ("Newton-Schulz 变体": the Gram iteration of section "Gram 空间 NS" with the restarts of
// section "重启机制", or the direct iteration of section "直接空间 NS（经典）").
//
// Shared memory holds every operand in the 128-byte-swizzled layout tcgen05 reads directly: X (up to
// 8 column blocks of 128 rows x 64 fp16) and R, Z, Q (2 blocks each). A K-major A operand, a K-major B
// operand (rows = output columns) and an MN-major B operand (rows = the contraction index) are all views of
// this one row-major layout, so each product is issued exactly as written: X X^T reads X as a K-major B;
// the m x m products (R R, Z Q, Z R, S Z) read their right factor MN-major, with no assumption that it is
// symmetric; Q X reads X MN-major. Accumulators live in tensor memory (up to 512 fp32 columns).
//
// Each phase: one thread issues the MMAs and commits to an mbarrier; all four warps wait, read their
// 32 accumulator rows with tcgen05.ld, apply the step's fp32 recipe and write the fp16 result back into
// shared memory (in place where the recipe reads the old value: each thread rewrites only its own row,
// after the MMA that read it has completed). Rows and columns beyond the matrix are kept at zero. The
// final Q X (or B X + a X) goes out as W += w_beta * O by TMA reduce-add (TMA store when W is
// overwritten, direct stores when W rows are not 16-byte aligned). Every wait is bounded.
#include <algorithm>

#include "internal.h"
#include "tc_ptx.h"

namespace dmuon {
namespace {

using namespace ptx;

constexpr int kBlk = 16384;       // one operand block: 128 rows x 64 fp16, 128-byte swizzle
constexpr int kXOff = 0;          // X: 8 blocks (512 columns)
constexpr int kROff = 8 * kBlk;   // R, and S while the R update runs (2 blocks)
constexpr int kZOff = 10 * kBlk;  // Z; the weight-update staging area at the end
constexpr int kQOff = 12 * kBlk;  // Q
constexpr int kOpBytes = 14 * kBlk;
constexpr int kSmallSmem = kOpBytes + 256 + 1024;
static_assert(kSmallSmem <= 232448, "shared memory budget");

// Byte offset of element (r, c) in an operand buffer.
__device__ __forceinline__ uint32_t op_off(int r, int c) {
  return static_cast<uint32_t>((c >> 6) * kBlk + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}

__device__ __forceinline__ void load_row32(const uint8_t* buf, int r, int c0, float (&e)[32]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 x = *reinterpret_cast<const uint4*>(buf + op_off(r, c0 + 8 * u));
    const __half2* h = reinterpret_cast<const __half2*>(&x);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(h[k]);
      e[8 * u + 2 * k] = f.x;
      e[8 * u + 2 * k + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store_row32(uint8_t* buf, int r, int c0, const float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<uint4*>(buf + op_off(r, c0 + 8 * u)) =
        make_uint4(pack_half2(v[8 * u + 0], v[8 * u + 1]), pack_half2(v[8 * u + 2], v[8 * u + 3]),
                   pack_half2(v[8 * u + 4], v[8 * u + 5]), pack_half2(v[8 * u + 6], v[8 * u + 7]));
}

// acc[0, N) (+)= A (128 x K, K-major at a) * B; B K-major (rows = output columns) or MN-major (rows = the
// contraction index, output columns across blocks). K a multiple of 16 (<= 512), N a multiple of 16 (<= 256).
__device__ __forceinline__ void issue_product(uint32_t d_tmem, uint32_t a, uint32_t b, int K, int N, bool b_mn) {
  const uint32_t idesc = (1u << 4) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
                         (static_cast<uint32_t>(128 >> 4) << 24);
  for (int kk = 0; kk < K / 16; ++kk) {
    const uint64_t da = smem_desc(a + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
    const uint64_t db = b_mn ? smem_desc(b + kk * 2048, kBlk, 1024) : smem_desc(b + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
    mma_f16(d_tmem, da, db, idesc, kk > 0 ? 1u : 0u);
  }
}

__global__ void __launch_bounds__(128, 1) ns_small_kernel(const __grid_constant__ SmallLaunch p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_x = reinterpret_cast<uint64_t*>(smem + kOpBytes);
  uint64_t* bar_mma = bar_x + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* Xs = smem + kXOff;
  uint8_t* Rs = smem + kROff;
  uint8_t* Zs = smem + kZOff;
  uint8_t* Qs = smem + kQOff;
  const uint32_t sx = smem_u32(Xs), sr = smem_u32(Rs), sz = smem_u32(Zs), sq = smem_u32(Qs);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid;  // tensor-memory lane = output row

  if (tid == 0) {
    mbar_init(bar_x, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t my_tmem = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  uint32_t x_phase = 0, mma_phase = 0;
  bool bad = false;

  // Issue (one thread) and wait for (everyone) one phase's products; smem operands must be fenced and
  // synchronised by the caller. Returns false (uniformly) if a wait gave up.
  auto mma_phase_done = [&]() -> bool {
    bool ok = wait_bounded(bar_mma, mma_phase, abort_flag, p.status, kWaitLimitNs, true);
    mma_phase ^= 1u;
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    return ok;
  };
  // Make this phase's shared-memory writes visible to the tensor cores and release tensor memory.
  auto operands_ready = [&]() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  for (int j = blockIdx.x; j < p.njobs; j += gridDim.x) {
    const SmallJob& job = p.jobs[j];
    const int m = job.m, n = job.n;
    const int nb = (n + 63) / 64;  // column blocks of X
    const int ncols = nb * 64;

    // ---- X into shared memory (rows >= m and columns >= n arrive as zeros)
    if (tid == 0) {
      fence_async_smem();  // the previous matrix's reads of X precede this overwrite
      mbar_arrive_expect_tx(bar_x, static_cast<uint32_t>(nb * kBlk));
      for (int c = 0; c < nb; ++c) tma_load_2d(sx + c * kBlk, &job.tmX, c * 64, 0, bar_x);
    }
    bool ok = wait_bounded(bar_x, x_phase, abort_flag, p.status, kWaitLimitNs, true);
    x_phase ^= 1u;
    if (!__syncthreads_and(ok)) break;

    // R = X X^T, written to Rs (zero outside m x m).
    auto gram_of_x = [&]() -> bool {
      if (tid == 0) {
        tc_fence_after();
        issue_product(tmem, sx, sx, ncols, 128, false);
        mma_commit(bar_mma);
      }
      if (!mma_phase_done()) return false;
      for (int c = 0; c < 128; c += 32) {
        float v[32];
        tmem_ld32(my_tmem + c, v);
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (row >= m || c + k >= m) v[k] = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) bad |= !fp16_ok(v[k]);
        store_row32(Rs, row, c, v);
      }
      operands_ready();
      return true;
    };
    // acc = A * B for an m x m pair (B MN-major), then out = s_acc * acc + s_e * E + s_i * [i == j]
    // (E read from `e` before out is written; out may equal e or be a third buffer).
    auto mm_phase = [&](uint32_t a, uint32_t b, uint8_t* e, uint8_t* out, float s_acc, float s_e, float s_i,
                        uint8_t* out2, float s_i2) -> bool {
      if (tid == 0) {
        tc_fence_after();
        issue_product(tmem, a, b, 128, 128, true);
        mma_commit(bar_mma);
      }
      if (!mma_phase_done()) return false;
      for (int c = 0; c < 128; c += 32) {
        float v[32], ev[32];
        tmem_ld32(my_tmem + c, v);
        if (e) load_row32(e, row, c, ev);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          float x = s_acc * v[k] + (e ? s_e * ev[k] : 0.f);
          if (c + k == row) x += s_i;
          v[k] = (row >= m || c + k >= m) ? 0.f : x;
          bad |= !fp16_ok(v[k]);
        }
        store_row32(out, row, c, v);
        if (out2) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (c + k == row && row < m) v[k] += s_i2;
#pragma unroll
          for (int k = 0; k < 32; ++k) bad |= !fp16_ok(v[k]);
          store_row32(out2, row, c, v);
        }
      }
      operands_ready();
      return true;
    };
    // acc[0, ncols) = A (128 x 128 at a) * X (MN-major).
    auto times_x = [&](uint32_t a) {
      if (tid == 0) {
        tc_fence_after();
        for (int h = 0; h * 256 < ncols; ++h)
          issue_product(tmem + static_cast<uint32_t>(h * 256), a, sx + h * 4 * kBlk, 128, min(256, ncols - h * 256), true);
        mma_commit(bar_mma);
      }
    };
    // X = s_acc * acc + s_e * X over the first ncols columns (zero outside m x n), in place.
    auto x_update = [&](float s_acc, float s_e) {
      for (int c = 0; c < ncols; c += 32) {
        float v[32], ev[32];
        tmem_ld32(my_tmem + c, v);
        if (s_e != 0.f) load_row32(Xs, row, c, ev);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float x = s_acc * v[k] + (s_e != 0.f ? s_e * ev[k] : 0.f);
          v[k] = (row >= m || c + k >= n) ? 0.f : x;
          bad |= !fp16_ok(v[k]);
        }
        store_row32(Xs, row, c, v);
      }
      operands_ready();
    };
    // W += w_beta * (s_acc * acc + s_e * X) (or W = ...), W in the caller's orientation.
    auto w_update = [&](float s_acc, float s_e) {
      uint8_t* stage = Zs + warp * 4096;
      const uint32_t sbuf = smem_u32(stage);
      const int row0 = warp * 32;
      const bool tma_w = job.tma_w && (p.w_alpha == 0.f || p.w_alpha == 1.f);
      if (row0 < m) {
        for (int c = 0; c < ncols && c < n; c += 32) {
          float v[32], ev[32];
          tmem_ld32(my_tmem + c, v);
          if (s_e != 0.f) load_row32(Xs, row, c, ev);
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float x = s_acc * v[k] + (s_e != 0.f ? s_e * ev[k] : 0.f);
            v[k] = (row >= m || c + k >= n) ? 0.f : x;
            bad |= !isfinite(v[k]);
          }
          if (tma_w) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            if (!job.trans) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(stage + sw128_f(lane, 4 * q)) =
                    make_float4(p.w_beta * v[4 * q], p.w_beta * v[4 * q + 1], p.w_beta * v[4 * q + 2], p.w_beta * v[4 * q + 3]);
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k) *reinterpret_cast<float*>(stage + sw128_f(k, lane)) = p.w_beta * v[k];
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int x = job.trans ? row0 : c, y = job.trans ? c : row0;
              if (p.w_alpha == 0.f) tma_store_2d(&job.tmW, sbuf, x, y);
              else tma_reduce_add_2d(&job.tmW, sbuf, x, y);
              bulk_commit();
            }
          } else if (row < m) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (c + k < n) {
                float* w = job.trans ? job.W + static_cast<int64_t>(c + k) * job.ldw + row
                                     : job.W + static_cast<int64_t>(row) * job.ldw + c + k;
                *w = (p.w_alpha != 0.f ? p.w_alpha * *w : 0.f) + p.w_beta * v[k];
              }
            }
          }
        }
      }
      if (lane == 0) bulk_wait_read0();  // the staging area is Z: free it before the next matrix
      tc_fence_before();
      __syncthreads();
    };

    bool alive = true;
    if (!job.direct) {
      // ---- Gram iteration
      if (!gram_of_x()) break;
      bool fresh = true;
      for (int k = 0; alive && k < p.steps; ++k) {
        const float a = p.coef[3 * k], b = p.coef[3 * k + 1], c = p.coef[3 * k + 2];
        if (k > 0 && ((p.restart_mask >> k) & 1u)) {
          times_x(sq);  // X <- Q X
          if (!mma_phase_done()) { alive = false; break; }
          x_update(1.f, 0.f);
          if (!gram_of_x()) { alive = false; break; }
          fresh = true;
        }
        // Z = b R + c R^2 (and Q = Z + a I after a (re)start)
        if (!mm_phase(sr, sr, Rs, Zs, c, b, 0.f, fresh ? Qs : nullptr, a)) { alive = false; break; }
        if (!fresh && !mm_phase(sz, sq, Qs, Qs, 1.f, a, 0.f, nullptr, 0.f)) { alive = false; break; }  // Q = ZQ + aQ
        const bool update_r = k + 1 < p.steps && !((p.restart_mask >> (k + 1)) & 1u);
        if (update_r) {
          if (!mm_phase(sz, sr, Rs, Rs, 1.f, a, 0.f, nullptr, 0.f)) { alive = false; break; }  // S = ZR + aR
          if (!mm_phase(sr, sz, Rs, Rs, 1.f, a, 0.f, nullptr, 0.f)) { alive = false; break; }  // R = SZ + aS
        }
        fresh = false;
      }
      if (!alive) break;
      times_x(sq);  // O = Q X
      if (!mma_phase_done()) break;
      w_update(1.f, 0.f);
    } else {
      // ---- direct iteration
      for (int k = 0; alive && k < p.steps; ++k) {
        const float a = p.coef[3 * k], b = p.coef[3 * k + 1], c = p.coef[3 * k + 2];
        if (!gram_of_x()) { alive = false; break; }                                       // A = X X^T
        if (!mm_phase(sr, sr, Rs, Zs, c, b, 0.f, nullptr, 0.f)) { alive = false; break; }  // B = b A + c A^2
        times_x(sz);                                                                       // B X
        if (!mma_phase_done()) { alive = false; break; }
        if (k + 1 < p.steps) x_update(1.f, a);  // X = B X + a X
        else w_update(1.f, a);
      }
      if (!alive) break;
    }
  }

  if (lane == 0) bulk_wait0();
  if (bad) atomicOr(p.status, kDevNonfinite);
  // After an abort, let any copy or MMA still in flight finish before shared and tensor memory go away.
  if (*abort_flag) {
    if (tid == 0) {
      mma_commit(bar_mma);
      wait_bounded(bar_mma, mma_phase, abort_flag, p.status, kDrainLimitNs, false);
      wait_bounded(bar_x, x_phase ^ 1u, abort_flag, p.status, kDrainLimitNs, false);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

bool encode_small_job(SmallJob& job, const __half* X, int64_t ldx, float* W, int64_t ldw, int m, int n, bool trans,
                      bool direct, const char** err) {
  job.direct = direct ? 1 : 0;
  job.m = m;
  job.n = n;
  job.trans = trans ? 1 : 0;
  job.W = W;
  job.ldw = ldw;
  if (!encode_tensor_2d(&job.tmX, X, static_cast<uint64_t>(n), static_cast<uint64_t>(m), static_cast<uint64_t>(ldx) * 2,
                        64, 128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, err))
    return false;
  job.tma_w = 0;
  if ((reinterpret_cast<uintptr_t>(W) & 15) == 0 && (ldw & 3) == 0) {
    const char* e2 = nullptr;
    const uint64_t inner = static_cast<uint64_t>(trans ? m : n), outer = static_cast<uint64_t>(trans ? n : m);
    if (encode_tensor_2d(&job.tmW, W, inner, outer, static_cast<uint64_t>(ldw) * 4, 32, 32,
                         CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B, &e2))
      job.tma_w = 1;
  }
  return true;
}

cudaError_t launch_ns_small(const SmallLaunch& p, int sms, cudaStream_t stream) {
  if (p.njobs <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
  if (e != cudaSuccess) return e;
  ns_small_kernel<<<std::min(p.njobs, sms), 128, kSmallSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dmuon
