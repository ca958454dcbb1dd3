// Fused Newton-Schulz for small matrices: the whole iteration of one matrix (m <= 128 rows, n <= 512
// columns after orientation) in one CTA, ending with the weight update -- one launch for every matrix of
// the call ("Newton-Schulz 变体": the Gram iteration of section "Gram 空间 NS" with the restarts of
// section "重启机制", or the direct iteration of section "直接空间 NS（经典）").
//
// Shared memory holds every operand in the 128-byte-swizzled layout tcgen05 reads directly: X (up to
// 8 column blocks of 128 rows x 64 fp16) and R, Z, Q (2 blocks each). X is built there from the fp32
// momentum and the norm pass's 1 / (||M|| + eps) (the normalise-and-cast step of the row-wise pass,
// with the same rounding), so no fp16 copy of X goes through HBM. A K-major A operand, a K-major B
// operand (rows = output columns) and an MN-major B operand (rows = the contraction index) are all views of
// this one row-major layout, so each product is issued exactly as written: X X^T reads X as a K-major B;
// the m x m products (R R, Z Q, Z R, S Z) read their right factor MN-major, with no assumption that it is
// symmetric; Q X reads X MN-major. Accumulators live in tensor memory (up to 512 fp32 columns).
//
// Each phase: one thread issues the MMAs and commits them to mbarriers; eight warps finish the phase, two
// per tensor-memory lane quarter (32 rows), one for each half of the output columns. A warp reads its
// accumulator columns with tcgen05.ld (two loads in flight per wait), applies the step's fp32 recipe and
// writes the fp16 result back into shared memory (in place where the recipe reads the old value: a
// thread rewrites only its own row's columns). The issuing thread, at about one MMA per 70 cycles, is the
// limit of the small products, so X X^T and the m x m products are single N = 128 products (all warps
// wait for all of it); the X-wide products (Q X, B X) go in two halves of output columns with a barrier
// each, so the first half's epilogue overlaps the second half's MMAs -- safe in place, because each half
// reads only its own column blocks of X. fp16 overflow is tracked with one packed FMA per pair of
// values. Rows and columns beyond the matrix are kept at zero. The final Q X (or B X + a X) goes out as
// W += w_beta * O by TMA reduce-add (TMA store when W is overwritten, direct stores when W rows are not
// 16-byte aligned); in the Gram form the next matrix's X is built under it (its M was prefetched into L2
// at the start of the current matrix). The launch is programmatic: set-up overlaps the norm pass's tail,
// and the kernel waits for it before touching global memory. Every wait is bounded.
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
constexpr int kSmallThreads = 256;  // 8 warps: two per tensor-memory lane quarter, one per column half
static_assert(kSmallSmem <= 232448, "shared memory budget");

// Byte offset of element (r, c) in an operand buffer.
__device__ __forceinline__ uint32_t op_off(int r, int c) {
  return static_cast<uint32_t>((c >> 6) * kBlk + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}

// 8 consecutive fp16 columns [c0, c0 + 8) of row r of an operand buffer (c0 a multiple of 8), as fp32.
__device__ __forceinline__ void load8(const uint8_t* buf, int r, int c0, float (&e)[8]) {
  const uint4 x = *reinterpret_cast<const uint4*>(buf + op_off(r, c0));
  const __half2* h = reinterpret_cast<const __half2*>(&x);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(h[k]);
    e[2 * k] = f.x;
    e[2 * k + 1] = f.y;
  }
}

// v rounded to fp16 as row r, columns [c0, c0 + 64). chk turns NaN if a value rounded to an infinity or
// was NaN (h * 0 + chk: one packed FMA per pair instead of a test per value).
__device__ __forceinline__ void store_row64(uint8_t* buf, int r, int c0, const float (&v)[64], __half2& chk) {
  const __half2 zero2 = __float2half2_rn(0.f);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(v[8 * u + 2 * q], v[8 * u + 2 * q + 1]);
      chk = __hfma2(h, zero2, chk);
      w[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(buf + op_off(r, c0 + 8 * u)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// X = fp16(M * inv) for X's column blocks [b_lo, b_hi) (zero outside m x n), done by `nth` threads (this one
// is number th; nth is 128 or 256) in part `part` of `nparts` equal shares: the normalise-and-cast step of
// the row-wise pass, done here so that X goes from M straight into shared memory. Every load is
// coalesced and every index is a shift or an increment (the fill is bound by its own instructions):
// M rows -- a warp takes X rows in turn, its lanes 8-column chunks of the row (two 16-byte loads each);
// transposed (X rows are M columns) -- a warp takes (32-row slab, 8-column chunk) units, its lanes the
// slab's rows (eight 4-byte loads each, one per M row). Batches of loads are in flight before any store.
__device__ __forceinline__ void fill_x(uint8_t* Xs, const SmallJob& jb, int b_lo, int b_hi, int th, int nth, int part,
                                       int nparts) {
  if (b_hi <= b_lo) return;
  const int jm = jb.m, jn = jb.n;
  const float* const M = jb.M;
  const int64_t ldm = jb.ldm;
  const bool vec = jb.vec_m != 0;
  const float inv = *jb.inv;
  const int nw = nth >> 5, wid = th >> 5, ln = th & 31;
  const int nch = 8 * (b_hi - b_lo);  // 8-column chunks in the range (8 ... 64)
  if (!jb.trans) {
    constexpr int kRows = 4;
    const int rows_w = 128 / nw;  // rows per warp
    const int i_lo = part * rows_w / nparts, i_hi = (part + 1) * rows_w / nparts;
    for (int i0 = i_lo; i0 < i_hi; i0 += kRows) {
      float4 v[kRows][2][2];
#pragma unroll
      for (int a = 0; a < kRows; ++a) {
        const int r = wid + nw * (i0 + a);
        const bool row_ok = i0 + a < i_hi && r < jm;
        const float* rp = M + static_cast<int64_t>(r) * ldm;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int c = 64 * b_lo + 8 * (ln + 32 * t);
          v[a][t][0] = v[a][t][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_ok && ln + 32 * t < nch && c < jn) {
            if (vec && c + 8 <= jn) {
              v[a][t][0] = __ldcs(reinterpret_cast<const float4*>(rp + c));
              v[a][t][1] = __ldcs(reinterpret_cast<const float4*>(rp + c + 4));
            } else {
              float e[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) e[k] = c + k < jn ? rp[c + k] : 0.f;
              v[a][t][0] = make_float4(e[0], e[1], e[2], e[3]);
              v[a][t][1] = make_float4(e[4], e[5], e[6], e[7]);
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < kRows; ++a) {
        const int r = wid + nw * (i0 + a);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (i0 + a >= i_hi || ln + 32 * t >= nch) continue;
          const float4 x = v[a][t][0], y = v[a][t][1];
          *reinterpret_cast<uint4*>(Xs + op_off(r, 64 * b_lo + 8 * (ln + 32 * t))) =
              make_uint4(pack_half2(x.x * inv, x.y * inv), pack_half2(x.z * inv, x.w * inv),
                         pack_half2(y.x * inv, y.y * inv), pack_half2(y.z * inv, y.w * inv));
        }
      }
    }
  } else {
    constexpr int kUnits = 4;
    const int units_w = 4 * nch / nw;  // (slab, chunk) units per warp: slab = unit & 3, chunk = unit >> 2
    const int i_lo = part * units_w / nparts, i_hi = (part + 1) * units_w / nparts;
    for (int i0 = i_lo; i0 < i_hi; i0 += kUnits) {
      float v[kUnits][8];
#pragma unroll
      for (int a = 0; a < kUnits; ++a) {
        const int k = wid + nw * (i0 + a);
        const int r = 32 * (k & 3) + ln, c = 64 * b_lo + 8 * (k >> 2);
        const bool live = i0 + a < i_hi && r < jm;
        const float* cp = M + static_cast<int64_t>(c) * ldm + r;
#pragma unroll
        for (int e = 0; e < 8; ++e) v[a][e] = live && c + e < jn ? __ldcs(cp + e * ldm) : 0.f;
      }
#pragma unroll
      for (int a = 0; a < kUnits; ++a) {
        if (i0 + a >= i_hi) continue;
        const int k = wid + nw * (i0 + a);
        const int r = 32 * (k & 3) + ln, c = 64 * b_lo + 8 * (k >> 2);
        *reinterpret_cast<uint4*>(Xs + op_off(r, c)) =
            make_uint4(pack_half2(v[a][0] * inv, v[a][1] * inv), pack_half2(v[a][2] * inv, v[a][3] * inv),
                       pack_half2(v[a][4] * inv, v[a][5] * inv), pack_half2(v[a][6] * inv, v[a][7] * inv));
      }
    }
  }
}

// 64 consecutive fp32 accumulator columns of this thread's TMEM lane: both loads in flight, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  tmem_ld32_issue(taddr, r);
  tmem_ld32_issue(taddr + 32, r + 32);
  tmem_ld_wait(r);
#pragma unroll
  for (int k = 0; k < 64; ++k) v[k] = __uint_as_float(r[k]);
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

__global__ void __launch_bounds__(kSmallThreads, 1) ns_small_kernel(const __grid_constant__ SmallLaunch p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(smem + kOpBytes);  // [0]: output columns [0, split); [1]: all
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* const Xs = smem + kXOff;
  uint8_t* const Rs = smem + kROff;  // R, and S while the R update runs
  uint8_t* const Zs = smem + kZOff;  // Z; with R, the staging area of the weight update
  uint8_t* const Qs = smem + kQOff;
  const uint32_t sx = smem_u32(Xs), sq = smem_u32(Qs);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;  // tensor-memory lanes 32 * quarter ... : the rows this warp owns
  const int half = warp >> 2;    // which half of each product's output columns this warp finishes
  const int row = quarter * 32 + lane;

  griddep_launch_dependents();
  if (tid == 0) {
    mbar_init(&bar_mma[0], 1);
    mbar_init(&bar_mma[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t my_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  griddep_wait();  // the norm pass's results are complete and visible before any global access
#if DMUON_DEVICE_CHECKS
  // Checked build: every job's sizes within the kernel's limits, or the launch does nothing.
  {
    bool ok = true;
    for (int j = tid; j < p.njobs; j += kSmallThreads) {
      const SmallJob& jb = p.jobs[j];
      ok &= jb.m >= 1 && jb.m <= kSmallMaxM && jb.n >= 1 && jb.n <= kSmallMaxN;
    }
    if (!__syncthreads_and(dev_check(ok, p.status))) {
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (warp == 0) tmem_dealloc(tmem, 512);
      return;
    }
  }
#endif

  uint32_t mma_phase = 0;
  bool bad = false;
  __half2 chk16 = __float2half2_rn(0.f);  // NaN once an fp16 operand overflowed
  float chk32 = 0.f;                      // NaN once an fp32 output was not finite

  // Wait for this warp's half of the phase's products, or for all of them (the second barrier is
  // committed after both halves).
  auto wait_half = [&](bool all = false) -> bool {
    const bool ok = wait_bounded(&bar_mma[all ? 1 : half], mma_phase, abort_flag, p.status, kWaitLimitNs, true);
    mma_phase ^= 1u;
    tc_fence_after();
    return ok;
  };
  // End of a phase: shared-memory results visible to the tensor core, tensor-memory reads done, every
  // thread here. False (uniformly) if some wait gave up.
  auto phase_end = [&](bool ok) -> bool {
    fence_async_smem();
    tc_fence_before();
    return __syncthreads_and(ok) != 0;
  };

  bool x_ready = false;  // X of the next matrix already in shared memory (filled under the weight update)
  for (int j = blockIdx.x; j < p.njobs; j += gridDim.x) {
    const SmallJob& job = p.jobs[j];
    const int m = job.m, n = job.n;
    const int nb = (n + 63) / 64;  // column blocks of X
    const int ncols = nb * 64;
    const int split = ((nb + 1) >> 1) * 64;  // X-wide products: columns [0, split) then [split, ncols)
    const int c_lo = half ? split : 0, c_hi = half ? ncols : split;
    const int c_mm = 64 * half;  // m x m products: this warp's 64 columns
    const bool has_next = j + static_cast<int>(gridDim.x) < p.njobs;

    if (!x_ready) {  // the first matrix, or one after a direct-form matrix: all threads fill X
      fill_x(Xs, job, 0, nb, tid, kSmallThreads, 0, 1);
      fence_async_smem();
      __syncthreads();
    }
    x_ready = false;
    const int nb_next = has_next ? (p.jobs[j + gridDim.x].n + 63) / 64 : 0;
    // The next matrix's M is read at the end of this one, when every CTA is busy with memory at once;
    // bring it into L2 now, under this matrix's products (M is contiguous: rows x ldm floats).
    if (has_next && warp == 7) {
      const SmallJob& nj = p.jobs[j + gridDim.x];
      const int64_t bytes = static_cast<int64_t>(nj.trans ? nj.n : nj.m) * nj.ldm * 4 & ~int64_t(15);
      for (int64_t off = static_cast<int64_t>(lane) * 16384; off < bytes; off += 32 * 16384)
        bulk_prefetch_l2(reinterpret_cast<const char*>(nj.M) + off, static_cast<uint32_t>(bytes - off < 16384 ? bytes - off : 16384));
    }

    // Products, issued by one thread. R = X X^T and the m x m products are one N = 128 product each,
    // committed to both barriers: the issuing thread is the limit, so fewer, wider MMAs win over an
    // early start for half of the columns.
    auto issue_gram = [&]() {
      tc_fence_after();
      issue_product(tmem, sx, sx, ncols, 128, false);
      mma_commit(&bar_mma[0]);
      mma_commit(&bar_mma[1]);
    };
    // acc = A * B for m x m operands, B MN-major.
    auto issue_mm = [&](uint32_t a, uint32_t b) {
      tc_fence_after();
      issue_product(tmem, a, b, 128, 128, true);
      mma_commit(&bar_mma[0]);
      mma_commit(&bar_mma[1]);
    };
    // acc[0, ncols) = A (128 x 128 at a) * X (MN-major), in two halves of output columns, each committed
    // to its own barrier (N up to 256 per half).
    auto issue_times_x = [&](uint32_t a) {
      tc_fence_after();
      issue_product(tmem, a, sx, 128, split, true);
      mma_commit(&bar_mma[0]);
      if (ncols > split)
        issue_product(tmem + static_cast<uint32_t>(split), a, sx + (split / 64) * kBlk, 128, ncols - split, true);
      mma_commit(&bar_mma[1]);
    };

    // R = X X^T, written to Rs (zero outside m x m).
    auto gram_of_x = [&]() -> bool {
      if (tid == 0) issue_gram();
      bool good = wait_half();
      if (good) {
        float v[64];
        tmem_ld64(my_tmem + c_mm, v);
        if (m < 128) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (row >= m || c_mm + k >= m) v[k] = 0.f;
        }
        store_row64(Rs, row, c_mm, v, chk16);
      }
      return phase_end(good);
    };
    // acc = A * B for an m x m pair (B MN-major), then out = s_acc * acc + s_e * E (E read from `e`; out
    // may equal e, since every product of the phase is complete when a thread rewrites its own row's
    // columns) and, when out2 is given, out2 = out + s_i2 I.
    auto mm_phase = [&](uint8_t* a, uint8_t* b, uint8_t* e, uint8_t* out, float s_acc, float s_e, uint8_t* out2,
                        float s_i2) -> bool {
      if (tid == 0) issue_mm(smem_u32(a), smem_u32(b));
      bool good = wait_half();
      if (good) {
        float v[64];
        tmem_ld64(my_tmem + c_mm, v);
        if (e) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float ev[8];
            load8(e, row, c_mm + 8 * u, ev);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[8 * u + k] = s_acc * v[8 * u + k] + s_e * ev[k];
          }
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) v[k] *= s_acc;
        }
        if (m < 128) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (row >= m || c_mm + k >= m) v[k] = 0.f;
        }
        store_row64(out, row, c_mm, v, chk16);
        if (out2) {
          if (row < m && row >= c_mm && row < c_mm + 64) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (c_mm + k == row) v[k] += s_i2;
          }
          store_row64(out2, row, c_mm, v, chk16);
        }
      }
      return phase_end(good);
    };
    // Q = Z Q + a Q and S = Z R + a R together (both need only Z): one wait and one epilogue for two
    // products, in tensor-memory columns [0, 128) and [128, 256).
    auto zq_zr_phase = [&](float a) -> bool {
      if (tid == 0) {
        tc_fence_after();
        issue_product(tmem, smem_u32(Zs), smem_u32(Qs), 128, 128, true);
        issue_product(tmem + 128, smem_u32(Zs), smem_u32(Rs), 128, 128, true);
        mma_commit(&bar_mma[0]);
        mma_commit(&bar_mma[1]);
      }
      bool good = wait_half();
      if (good) {
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          uint8_t* o = t ? Rs : Qs;
          float v[64];
          tmem_ld64(my_tmem + 128 * t + c_mm, v);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float ev[8];
            load8(o, row, c_mm + 8 * u, ev);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[8 * u + k] = v[8 * u + k] + a * ev[k];
          }
          if (m < 128) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (row >= m || c_mm + k >= m) v[k] = 0.f;
          }
          store_row64(o, row, c_mm, v, chk16);
        }
      }
      return phase_end(good);
    };
    // X = s_acc * acc + s_e * X over this warp's columns (zero outside m x n), in place: the other half's
    // products read only the other half's column blocks of X.
    auto x_update = [&](float s_acc, float s_e) -> bool {
      bool good = wait_half();
      if (good) {
        for (int c = c_lo; c < c_hi; c += 64) {
          float v[64];
          tmem_ld64(my_tmem + c, v);
          if (s_e != 0.f) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float ev[8];
              load8(Xs, row, c + 8 * u, ev);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[8 * u + k] = s_acc * v[8 * u + k] + s_e * ev[k];
            }
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) v[k] *= s_acc;
          }
          if (row >= m || c + 64 > n) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (row >= m || c + k >= n) v[k] = 0.f;
          }
          store_row64(Xs, row, c, v, chk16);
        }
      }
      return phase_end(good);
    };
    // W += w_beta * (s_acc * acc + s_e * X) (or W = ...), W in the caller's orientation. The R and Z
    // buffers (64 KB, free by now) stage two 32 x 32 fp32 tiles per warp for the TMA reduce-adds. (The
    // TMA unit moves about 20 bytes per cycle here whatever the box: 32 x 128 boxes filled by four warps
    // together were slower, having fewer boxes in flight.)
    // With fill_next, each half also fills its own column blocks of the next matrix's X (the products
    // that read them are done) in shares between its groups, so the loads overlap the TMA's drain.
    auto w_update = [&](float s_acc, float s_e, bool good, bool fill_next) -> bool {
      uint8_t* stage = smem + kROff + warp * 8192;
      const uint32_t sbuf = smem_u32(stage);
      const int row0 = quarter * 32;
      const bool tma_w = job.tma_w && (p.w_alpha == 0.f || p.w_alpha == 1.f);
      const SmallJob* nj = good && fill_next ? &p.jobs[j + gridDim.x] : nullptr;
      const int fb_lo = half ? split / 64 : 0, fb_hi = half ? nb_next : min(split / 64, nb_next);
      const int groups = max(0, (min(c_hi, n) - c_lo + 63) / 64), nparts = max(1, groups);
      int filled = 0;
      if (good && row0 < m) {
        for (int c = c_lo; c < c_hi && c < n; c += 64) {
          float v[64];
          tmem_ld64(my_tmem + c, v);
          if (s_e != 0.f) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float ev[8];
              load8(Xs, row, c + 8 * u, ev);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[8 * u + k] = s_acc * v[8 * u + k] + s_e * ev[k];
            }
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) v[k] *= s_acc;
          }
          if (row >= m || c + 64 > n) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (row >= m || c + k >= n) v[k] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 64; ++k) chk32 = fmaf(v[k], 0.f, chk32);
          if (tma_w) {
            if (lane == 0) bulk_wait_read0();  // the previous group's tiles have left the staging area
            __syncwarp();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              uint8_t* tile = stage + t * 4096;
              if (!job.trans) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  *reinterpret_cast<float4*>(tile + sw128_f(lane, 4 * q)) =
                      make_float4(p.w_beta * v[32 * t + 4 * q], p.w_beta * v[32 * t + 4 * q + 1],
                                  p.w_beta * v[32 * t + 4 * q + 2], p.w_beta * v[32 * t + 4 * q + 3]);
              } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) *reinterpret_cast<float*>(tile + sw128_f(k, lane)) = p.w_beta * v[32 * t + k];
              }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              for (int t = 0; t < 2 && c + 32 * t < n; ++t) {
                const int cc = c + 32 * t;
                const int x = job.trans ? row0 : cc, y = job.trans ? cc : row0;
                if (p.w_alpha == 0.f) tma_store_2d(&job.tmW, sbuf + t * 4096, x, y);
                else tma_reduce_add_2d(&job.tmW, sbuf + t * 4096, x, y);
              }
              bulk_commit();
            }
            if (nj) fill_x(Xs, *nj, fb_lo, fb_hi, quarter * 32 + lane, 128, filled++, nparts);
          } else if (row < m) {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              if (c + k < n) {
                float* w = job.trans ? job.W + static_cast<int64_t>(c + k) * job.ldw + row
                                     : job.W + static_cast<int64_t>(row) * job.ldw + c + k;
                *w = (p.w_alpha != 0.f ? p.w_alpha * *w : 0.f) + p.w_beta * v[k];
              }
            }
          }
        }
      }
      if (nj)
        for (; filled < nparts; ++filled) fill_x(Xs, *nj, fb_lo, fb_hi, quarter * 32 + lane, 128, filled, nparts);
      if (lane == 0) bulk_wait_read0();  // the staging area is R and Z: free it before the next matrix
      return phase_end(good);
    };

    bool alive = true;
    if (!job.direct) {
      // ---- Gram iteration
      if (!gram_of_x()) break;
      bool fresh = true;
      for (int k = 0; alive && k < p.steps; ++k) {
        const float a = p.coef[3 * k], b = p.coef[3 * k + 1], c = p.coef[3 * k + 2];
        if (k > 0 && ((p.restart_mask >> k) & 1u)) {
          if (tid == 0) issue_times_x(sq);  // X <- Q X
          if (!x_update(1.f, 0.f) || !gram_of_x()) { alive = false; break; }
          fresh = true;
        }
        // Z = b R + c R^2 (and Q = Z + a I after a (re)start)
        if (!mm_phase(Rs, Rs, Rs, Zs, c, b, fresh ? Qs : nullptr, a)) { alive = false; break; }
        const bool update_r = k + 1 < p.steps && !((p.restart_mask >> (k + 1)) & 1u);
        if (!fresh && update_r) {
          if (!zq_zr_phase(a)) { alive = false; break; }  // Q = ZQ + aQ, S = ZR + aR
        } else {
          if (!fresh && !mm_phase(Zs, Qs, Qs, Qs, 1.f, a, nullptr, 0.f)) { alive = false; break; }  // Q = ZQ + aQ
          if (update_r && !mm_phase(Zs, Rs, Rs, Rs, 1.f, a, nullptr, 0.f)) { alive = false; break; }  // S = ZR + aR
        }
        if (update_r && !mm_phase(Rs, Zs, Rs, Rs, 1.f, a, nullptr, 0.f)) { alive = false; break; }  // R = SZ + aS
        fresh = false;
      }
      if (!alive) break;
      if (tid == 0) issue_times_x(sq);  // O = Q X
      const bool good = wait_half();
      if (!w_update(1.f, 0.f, good, has_next)) break;
      x_ready = has_next;
    } else {
      // ---- direct iteration
      for (int k = 0; alive && k < p.steps; ++k) {
        const float a = p.coef[3 * k], b = p.coef[3 * k + 1], c = p.coef[3 * k + 2];
        if (!gram_of_x()) { alive = false; break; }                                       // A = X X^T
        if (!mm_phase(Rs, Rs, Rs, Zs, c, b, nullptr, 0.f)) { alive = false; break; }  // B = b A + c A^2
        if (tid == 0) issue_times_x(smem_u32(Zs));                                         // B X
        if (k + 1 < p.steps) {
          if (!x_update(1.f, a)) { alive = false; break; }  // X = B X + a X
        } else if (!w_update(1.f, a, wait_half(true), false)) {  // Z, in the staging area, is read by both halves
          alive = false;
          break;
        }
      }
      if (!alive) break;
    }
  }

  if (lane == 0) bulk_wait0();
  bad |= __hisnan(__low2half(chk16)) || __hisnan(__high2half(chk16)) || chk32 != chk32;
  if (bad) atomicOr(p.status, kDevNonfinite);
  // After an abort, let any copy or MMA still in flight finish before shared and tensor memory go away.
  // Every thread waited once per product, so the last product's phase has parity mma_phase ^ 1 and may
  // still be pending; the drain commit completes the phase after it. A wait on the drain's parity alone
  // would return at once while the product's phase is open (it names the completed phase before), so
  // both phases are waited for, in order.
  if (*abort_flag) {
    if (tid == 0) {
      mma_commit(&bar_mma[1]);
      wait_bounded(&bar_mma[1], mma_phase ^ 1u, abort_flag, p.status, kDrainLimitNs, false);
      wait_bounded(&bar_mma[1], mma_phase, abort_flag, p.status, kDrainLimitNs, false);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

bool encode_small_job(SmallJob& job, const float* M, int64_t ldm, const float* inv, float* W, int64_t ldw, int m,
                      int n, bool trans, bool direct, const char** err) {
  job.direct = direct ? 1 : 0;
  job.m = m;
  job.n = n;
  job.trans = trans ? 1 : 0;
  job.M = M;
  job.ldm = ldm;
  job.inv = inv;
  job.vec_m = (reinterpret_cast<uintptr_t>(M) & 15) == 0 && (ldm & 3) == 0;
  job.W = W;
  job.ldw = ldw;
  job.tma_w = 0;
  if ((reinterpret_cast<uintptr_t>(W) & 15) == 0 && (ldw & 3) == 0) {
    const char* e2 = nullptr;
    const uint64_t inner = static_cast<uint64_t>(trans ? m : n), outer = static_cast<uint64_t>(trans ? n : m);
    if (encode_tensor_2d(&job.tmW, W, inner, outer, static_cast<uint64_t>(ldw) * 4, 32, 32,
                         CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B, &e2))
      job.tma_w = 1;
  }
  (void)err;
  return true;
}

cudaError_t launch_ns_small(const SmallLaunch& p, int sms, cudaStream_t stream) {
  if (p.njobs <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
  if (e != cudaSuccess) return e;
  // Programmatic stream serialisation: launch and set-up overlap the norm pass's tail; the kernel waits
  // for it before touching global memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(p.njobs, sms)), 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmallSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, ns_small_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dmuon
