// Grouped fp16 tensor-core GEMM / SYRK for sm_103a: TMA -> shared memory ring -> tcgen05.mma with
// fp32 accumulators in tensor memory -> tcgen05.ld epilogue.
//
// Every product of both Newton-Schulz forms runs here ("Newton-Schulz 变体" page: X X^T and R^2 as
// symmetric products -- "R 是对称的 ... SYRK" in section "Gram 空间 NS" -- plus Z Q, Z R, S Z, Q X,
// and B X for the direct form). One launch walks a list of 128 x BN output tiles drawn from many
// jobs (one job = one product on one matrix), so all matrices a rank owns advance one phase per
// launch.
//
// CTA layout (192 threads, one persistent CTA per SM):
//   warp 0      TMA producer: one thread streams 128 x 64 A tiles and BN x 64 B tiles into a
//               STAGES-deep ring of 128-byte-swizzled shared memory buffers.
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma (M=128, N=BN, K=16) into one
//               of two BN-column fp32 accumulators and commits completion to mbarriers.
//   warps 2-5   epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..+31, i.e.
//               one output row per thread), combine with the step's scalars and an optional fp16
//               addend, store fp16 (mirrored for symmetric outputs) or update the fp32 weights.
// The accumulator is double-buffered so a tile's epilogue overlaps the next tile's main loop.
//
// Every mbarrier wait is bounded: after kWaitLimitNs the waiting thread raises a CTA-wide abort
// flag and sets kDevTimeout in the device status word, all roles leave their loops, in-flight copies
// and MMAs are drained (again with a bound), tensor memory is freed and the kernel returns.
#include <cstdio>

#include "internal.h"

namespace dmuon {
namespace {

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s: far above any legitimate wait
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s for draining after an abort

template <int BN>
struct Cfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kABytes = kBM * kBK * 2;  // 16 KB
  static constexpr int kBBytes = BN * kBK * 2;   // 32 KB or 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators of BN fp32 columns
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");
  static_assert((2 * kStages + 5) * 8 + 8 <= kBarrierBytes, "barrier area too small");
};

// ---------------------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with parity `parity` of `bar` to complete. Returns false if the CTA is aborting
// or the wait exceeded `limit_ns` (which starts the abort). `honour_abort` = false is used when
// draining after an abort.
__device__ __noinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status, unsigned long long limit_ns,
                                          bool honour_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        if (honour_abort) {
          *abort_flag = 1;
          atomicOr(status, kDevTimeout);
        }
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading / stride byte offsets (all >> 4),
// descriptor version 1 at bit 46, 128-byte swizzle (layout type 2) at bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16: fp32 accumulator (bit 4), A and B fp16 (format 0), A K-major,
// B K-major or MN-major (bit 16), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int BN>
__device__ __forceinline__ uint32_t instr_desc(bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

// ---------------------------------------------------------------------------- tile bookkeeping

struct TileRef {
  const GemmJob* job;
  int tm, tn;
  bool skip;  // a lower-triangle tile of a symmetric single-job launch: nobody touches it
};

__device__ __forceinline__ TileRef tile_at(const GemmLaunch& p, int t, int bn) {
  TileRef r;
  if (p.jobs != nullptr) {
    const GemmTile g = p.tiles[t];
    r.job = p.jobs + g.job;
    r.tm = g.tm;
    r.tn = g.tn;
    r.skip = false;
  } else {
    r.job = &p.single;
    r.tm = t / p.single.tiles_n;
    r.tn = t - r.tm * p.single.tiles_n;
    r.skip = (p.single.flags & kJobSymmetric) && (r.tn * bn + bn - 1 < r.tm * kBM);
  }
  return r;
}

// ---------------------------------------------------------------------------- epilogue

struct Scalars {
  float acc, e, diag, d2;
};

__device__ __forceinline__ Scalars recipe_scalars(const GemmLaunch& p, int recipe) {
  switch (recipe) {
    case kRecZ: return {p.c, p.b, 0.f, p.a};
    case kRecAxpy: return {1.f, p.a, 0.f, 0.f};
    case kRecCustom: return {p.alpha, p.beta, p.gamma, 0.f};
    default: return {1.f, 0.f, 0.f, 0.f};
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ bool fp16_ok(float x) { return fabsf(x) < 65520.f; }  // false for NaN too

// Store 32 fp16 values of row i, columns j0.. (all in bounds, 16-byte aligned).
__device__ __forceinline__ void store_row32(__half* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d[q] = make_uint4(pack_half2(v[8 * q + 0], v[8 * q + 1]), pack_half2(v[8 * q + 2], v[8 * q + 3]),
                      pack_half2(v[8 * q + 4], v[8 * q + 5]), pack_half2(v[8 * q + 6], v[8 * q + 7]));
  }
}

template <int BN>
__device__ void epilogue_tile(const GemmLaunch& p, const GemmJob& job, int tm, int tn, int quarter,
                              int lane, uint32_t taddr, bool& bad) {
  const int row0 = tm * kBM + quarter * 32;  // first row handled by this warp
  const int i = row0 + lane;
  const bool sym = (job.flags & kJobSymmetric) != 0;
  const bool final_out = (job.flags & kJobFinal) != 0;
  const bool final_trans = (job.flags & kJobFinalTrans) != 0;
  const bool has_d2 = (job.flags & kJobD2) != 0;
  const Scalars s = recipe_scalars(p, job.recipe);
  const bool has_e = job.E != nullptr && s.e != 0.f;
  const bool row_ok = i < job.M;

  for (int c = 0; c < BN; c += 32) {
    const int j0 = tn * BN + c;
    if (j0 >= job.N) break;              // warp-uniform
    if (sym && j0 < row0) continue;      // whole chunk below the diagonal for every row of this warp
    float v[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c), v);
    if (!row_ok) continue;
    const bool full = j0 + 32 <= job.N;

    if (has_e) {
      const __half* erow = job.E + static_cast<int64_t>(i) * job.lde + j0;
      if (full) {
        const uint4* e4 = reinterpret_cast<const uint4*>(erow);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u = e4[q];
          const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float2 f = __half22float2(h[k]);
            v[8 * q + 2 * k] = fmaf(s.acc, v[8 * q + 2 * k], s.e * f.x);
            v[8 * q + 2 * k + 1] = fmaf(s.acc, v[8 * q + 2 * k + 1], s.e * f.y);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float e = (j0 + k < job.N) ? __half2float(erow[k]) : 0.f;
          v[k] = fmaf(s.acc, v[k], s.e * e);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= s.acc;
    }
    if (s.diag != 0.f) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (j0 + k == i) v[k] += s.diag;
    }

    if (final_out) {
      // W = w_alpha * W + w_beta * v, W in the caller's orientation.
      if (!final_trans) {
        float* wrow = job.W + static_cast<int64_t>(i) * job.ldw + j0;
        const bool vec = full && ((job.ldw & 3) == 0) && ((reinterpret_cast<uintptr_t>(job.W) & 15) == 0);
        if (vec) {
          float4* w4 = reinterpret_cast<float4*>(wrow);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 w = p.w_alpha != 0.f ? w4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            w.x = p.w_alpha * w.x + p.w_beta * v[4 * q + 0];
            w.y = p.w_alpha * w.y + p.w_beta * v[4 * q + 1];
            w.z = p.w_alpha * w.z + p.w_beta * v[4 * q + 2];
            w.w = p.w_alpha * w.w + p.w_beta * v[4 * q + 3];
            bad |= !(isfinite(w.x) && isfinite(w.y) && isfinite(w.z) && isfinite(w.w));
            w4[q] = w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            if (j0 + k < job.N) {
              const float w = (p.w_alpha != 0.f ? p.w_alpha * wrow[k] : 0.f) + p.w_beta * v[k];
              bad |= !isfinite(w);
              wrow[k] = w;
            }
          }
        }
      } else {
        // Kernel row i is the caller's column i: consecutive lanes write consecutive addresses.
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (j0 + k < job.N) {
            float* w = job.W + static_cast<int64_t>(j0 + k) * job.ldw + i;
            const float nw = (p.w_alpha != 0.f ? p.w_alpha * *w : 0.f) + p.w_beta * v[k];
            bad |= !isfinite(nw);
            *w = nw;
          }
        }
      }
      continue;
    }

#pragma unroll
    for (int k = 0; k < 32; ++k) bad |= !fp16_ok(v[k]);

    // Symmetric outputs: chunks with j0 > row0 lie strictly above the diagonal for every row here.
    const bool upper_chunk = sym && j0 > row0;
    const bool diag_chunk = sym && j0 == row0;
    for (int pass = 0; pass < (has_d2 ? 2 : 1); ++pass) {
      __half* out = pass == 0 ? job.D : job.D2;
      if (pass == 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (j0 + k == i) {
            v[k] += s.d2;
            bad |= !fp16_ok(v[k]);
          }
        }
      }
      __half* orow = out + static_cast<int64_t>(i) * job.ldd + j0;
      if (!sym || upper_chunk) {
        if (full) {
          store_row32(orow, v);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j0 + k < job.N) orow[k] = __float2half_rn(v[k]);
        }
        if (upper_chunk) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j0 + k < job.N) out[static_cast<int64_t>(j0 + k) * job.ldd + i] = __float2half_rn(v[k]);
        }
      } else if (diag_chunk) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = j0 + k;
          if (j < job.N && j >= i) {
            const __half h = __float2half_rn(v[k]);
            orow[k] = h;
            if (j > i) out[static_cast<int64_t>(j) * job.ldd + i] = h;
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------- the kernel

template <int BN>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GemmLaunch p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[C::kStages];
      uint32_t issued_parity[C::kStages];
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) issued[s] = 0, issued_parity[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x) {
        const TileRef tr = tile_at(p, t, BN);
        if (tr.skip) continue;
        const GemmJob* job = tr.job;
        const int nkb = (job->K + kBK - 1) / kBK;
        const bool bmn = (job->flags & kJobBMnMajor) != 0;
        const int m0 = tr.tm * kBM;
        const int n0 = tr.tn * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, kWaitLimitNs, true)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          tma_load_2d(sa, &job->tmA, kb * kBK, m0, &full[stage]);
          if (!bmn) {
            tma_load_2d(sb, &job->tmB, kb * kBK, n0, &full[stage]);
          } else {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) tma_load_2d(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, &full[stage]);
          }
          issued[stage] = 1;
          issued_parity[stage] = phase;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Aborting: let every copy already issued land before the CTA's shared memory is released.
        for (int s = 0; s < C::kStages; ++s)
          if (issued[s]) wait_bounded(&full[s], issued_parity[s], abort_flag, p.status, kDrainLimitNs, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x) {
        const TileRef tr = tile_at(p, t, BN);
        if (tr.skip) continue;
        const GemmJob* job = tr.job;
        const int nkb = (job->K + kBK - 1) / kBK;
        const bool bmn = (job->flags & kJobBMnMajor) != 0;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, kWaitLimitNs, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t idesc = instr_desc<BN>(bmn);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p.status, kWaitLimitNs, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // A (K-major): advance 16 fp16 = 32 bytes along the swizzled row; 8-row groups 1024 B apart.
            const uint64_t da = smem_desc(sa + k * 32, 16, 1024);
            // B K-major: as A. B MN-major: 16 K-rows = two 8-row groups of 1024 B; 64-column groups
            // (one TMA box each) 8192 B apart.
            const uint64_t db = bmn ? smem_desc(sb + k * 2048, 8192, 1024) : smem_desc(sb + k * 32, 16, 1024);
            mma_f16(d_tmem, da, db, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Make sure every MMA this thread issued has completed before tensor memory is freed.
      mma_commit(drain);
      wait_bounded(drain, 0, abort_flag, p.status, kDrainLimitNs, false);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    bool bad = false;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
      const TileRef tr = tile_at(p, t, BN);
      if (tr.skip) continue;
      bool ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, p.status, kWaitLimitNs, true);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      epilogue_tile<BN>(p, *tr.job, tr.tm, tr.tn, quarter, lane, taddr, bad);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (bad) atomicOr(p.status, kDevNonfinite);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D fp16 map: `inner` contiguous elements per row, `outer` rows `row_bytes` apart.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer, const char** err) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled is not available from the CUDA driver";
    return false;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled rejected an operand (alignment, stride or size)";
    return false;
  }
  return true;
}

}  // namespace

int gemm_smem_bytes(int bn) { return bn == 256 ? Cfg<256>::kSmemBytes : Cfg<128>::kSmemBytes; }

bool encode_job_maps(GemmJob& job, const void* a, int64_t lda, const void* b, int64_t ldb, bool b_mn_major,
                     int bn, const char** err) {
  if (!encode_2d(&job.tmA, a, static_cast<uint64_t>(job.K), static_cast<uint64_t>(job.M),
                 static_cast<uint64_t>(lda) * 2, kBK, kBM, err))
    return false;
  if (!b_mn_major)
    return encode_2d(&job.tmB, b, static_cast<uint64_t>(job.K), static_cast<uint64_t>(job.N),
                     static_cast<uint64_t>(ldb) * 2, kBK, static_cast<uint32_t>(bn), err);
  return encode_2d(&job.tmB, b, static_cast<uint64_t>(job.N), static_cast<uint64_t>(job.K),
                   static_cast<uint64_t>(ldb) * 2, 64, kBK, err);
}

cudaError_t launch_gemm(const GemmLaunch& p, int bn, int grid, cudaStream_t stream) {
  if (p.ntiles <= 0) return cudaSuccess;
  cudaError_t e;
  if (bn == 256) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<256>::kSmemBytes);
    if (e != cudaSuccess) return e;
    gemm_tc_kernel<256><<<grid, 192, Cfg<256>::kSmemBytes, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    gemm_tc_kernel<128><<<grid, 192, Cfg<128>::kSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dmuon
