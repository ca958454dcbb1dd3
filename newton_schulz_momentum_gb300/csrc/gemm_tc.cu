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
#include <algorithm>
#include <cstdio>

#include "internal.h"

namespace dmuon {
namespace {

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s: far above any legitimate wait
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s for draining after an abort

// BN: output tile width. CG: CTAs per MMA (1, or 2 for a CTA pair sharing one 256 x BN tile with
// tcgen05.mma.cta_group::2; each CTA then holds 128 rows of A and BN / 2 rows of B per stage).
template <int BN, int CG>
struct Cfg {
  static constexpr int kBRows = BN / CG;         // rows of the B tile held by one CTA
  static constexpr int kTileM = kBM * CG;        // output rows per tile
  static constexpr int kABytes = kBM * kBK * 2;  // 16 KB
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (kStageBytes <= 32768) ? 6 : 4;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators of BN fp32 columns
  static constexpr int kEpiBytes = 4 * 4096;  // one 4 KB staging buffer per epilogue warp
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiBytes + kBarrierBytes + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");
  static_assert((2 * kStages + 5) * 8 + 8 <= kBarrierBytes, "barrier area too small");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
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

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of this CTA's shared variable at `addr` as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// CTA-pair load: the data lands in this CTA's shared memory, completion is signalled on the mbarrier at
// shared::cluster address `mbar` (the pair's leader).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t mbar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar_cluster_addr) : "memory");
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
template <int BM, int BN>
__device__ __forceinline__ uint32_t instr_desc(bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
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

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this shared offset in both CTAs of the pair once this thread's MMAs finish.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Completion of this thread's CTA-pair MMAs, signalled on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
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

// CTA-pair allocation: executed by one warp in each CTA of the pair; the same columns are allocated in
// both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
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

__device__ __forceinline__ TileRef tile_at(const GemmLaunch& p, int t, int bn, int tile_m) {
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
    r.skip = (p.single.flags & kJobSymmetric) && (r.tn * bn + bn - 1 < r.tm * tile_m);
  }
  return r;
}

// ---------------------------------------------------------------------------- epilogue
//
// Each epilogue warp owns 32 rows of the tile and walks it in 32-column chunks. A chunk's values are
// combined in registers, written into the warp's 4 KB staging buffer in shared memory (swizzled so the
// writes are bank-conflict free) and sent out by one lane with a TMA bulk store: the 32 x 32 fp16 block
// of D (plus, for symmetric outputs, its transpose at the mirrored position), or, for the final
// update, the fp32 block reduce-added into W (stored, when W is overwritten). The fp16 addend E of the
// next chunk is loaded while the current chunk is processed.

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t smem_src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(smem_src)
               : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t smem_src, int c0, int c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(smem_src)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Byte offset of element (r, c) of a 32 x 32 fp16 block: 64-byte rows, 16-byte units swizzled by the
// TMA 64-byte pattern (unit ^= (r >> 1) & 3). Buffers are 1024-byte aligned.
__device__ __forceinline__ uint32_t sw64_h(int r, int c) {
  return static_cast<uint32_t>(r * 64 + ((((c >> 3) ^ (r >> 1)) & 3) << 4) + ((c & 7) << 1));
}
// Byte offset of element (r, c) of a 32 x 32 fp32 block: 128-byte rows, 128-byte swizzle (unit ^= r & 7).
__device__ __forceinline__ uint32_t sw128_f(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((((c >> 2) ^ r) & 7) << 4) + ((c & 3) << 2));
}

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

template <int BN>
__device__ void epilogue_tile(const GemmLaunch& p, const GemmJob& job, int tile_row0, int tn, int quarter,
                              int lane, uint32_t taddr, uint8_t* stage, bool& bad) {
  const int row0 = tile_row0 + quarter * 32;  // first row handled by this warp
  if (row0 >= job.M) return;                  // all 32 rows past the edge: nothing to read or store
  const int i = row0 + lane;
  const bool sym = (job.flags & kJobSymmetric) != 0;
  const bool final_out = (job.flags & kJobFinal) != 0;
  const bool final_trans = (job.flags & kJobFinalTrans) != 0;
  const bool has_d2 = (job.flags & kJobD2) != 0;
  const bool tma_w = final_out && (job.flags & kJobTmaW) && (p.w_alpha == 0.f || p.w_alpha == 1.f);
  const Scalars s = recipe_scalars(p, job.recipe);
  const bool row_ok = i < job.M;
  const __half* erow = (job.E != nullptr && s.e != 0.f && row_ok) ? job.E + static_cast<int64_t>(i) * job.lde : nullptr;
  const bool has_e = job.E != nullptr && s.e != 0.f;
  const uint32_t sbuf = smem_u32(stage);

  // Symmetric outputs: chunks left of the diagonal block are produced by the mirrored stores of other
  // tiles, so this warp starts at its diagonal block (row0 and tn*BN are multiples of 32).
  int c = sym ? max(0, row0 - tn * BN) : 0;
  uint4 ecur[4], enext[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) ecur[q] = make_uint4(0, 0, 0, 0), enext[q] = ecur[q];
  if (erow && c < BN && tn * BN + c + 32 <= job.N) {
    const uint4* e4 = reinterpret_cast<const uint4*>(erow + tn * BN + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) ecur[q] = e4[q];
  }

  for (; c < BN; c += 32) {
    const int j0 = tn * BN + c;
    if (j0 >= job.N) break;  // warp-uniform
    const bool full = j0 + 32 <= job.N;
    const bool prefetch = erow != nullptr && c + 32 < BN && j0 + 64 <= job.N;
    if (prefetch) {
      const uint4* e4 = reinterpret_cast<const uint4*>(erow + j0 + 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) enext[q] = e4[q];
    }
    float v[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c), v);

    if (!row_ok) {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = 0.f;
    } else if (has_e) {
      if (full) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __half2* h = reinterpret_cast<const __half2*>(&ecur[q]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(h[k]);
            v[8 * q + 2 * k] = fmaf(s.acc, v[8 * q + 2 * k], s.e * f.x);
            v[8 * q + 2 * k + 1] = fmaf(s.acc, v[8 * q + 2 * k + 1], s.e * f.y);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float e = (j0 + k < job.N) ? __half2float(erow[j0 + k]) : 0.f;
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
    if (prefetch) {
#pragma unroll
      for (int q = 0; q < 4; ++q) ecur[q] = enext[q];
    }

    if (final_out) {
#pragma unroll
      for (int k = 0; k < 32; ++k) bad |= (j0 + k < job.N) && !isfinite(v[k]);
      if (tma_w) {
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        if (!final_trans) {
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
          const int x = final_trans ? row0 : j0;
          const int y = final_trans ? j0 : row0;
          if (p.w_alpha == 0.f) tma_store_2d(&job.tmW, sbuf, x, y);
          else tma_reduce_add_2d(&job.tmW, sbuf, x, y);
          bulk_commit();
        }
      } else if (row_ok) {
        // W rows not 16-byte aligned: direct read-modify-write.
        if (!final_trans) {
          float* wrow = job.W + static_cast<int64_t>(i) * job.ldw + j0;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j0 + k < job.N) wrow[k] = (p.w_alpha != 0.f ? p.w_alpha * wrow[k] : 0.f) + p.w_beta * v[k];
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            if (j0 + k < job.N) {
              float* w = job.W + static_cast<int64_t>(j0 + k) * job.ldw + i;
              *w = (p.w_alpha != 0.f ? p.w_alpha * *w : 0.f) + p.w_beta * v[k];
            }
          }
        }
      }
      continue;
    }

#pragma unroll
    for (int k = 0; k < 32; ++k) bad |= (j0 + k < job.N) && !fp16_ok(v[k]);
    const bool upper = sym && j0 > row0;  // strictly above the diagonal for every row of the block
    const bool on_diag = j0 == row0;      // the block holds the diagonal elements i == j

    if (lane == 0) bulk_wait_read0();  // the previous chunk's stores have read the buffer
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stage + sw64_h(lane, 8 * q)) =
          make_uint4(pack_half2(v[8 * q + 0], v[8 * q + 1]), pack_half2(v[8 * q + 2], v[8 * q + 3]),
                     pack_half2(v[8 * q + 4], v[8 * q + 5]), pack_half2(v[8 * q + 6], v[8 * q + 7]));
    if (upper) {
#pragma unroll
      for (int k = 0; k < 32; ++k) *reinterpret_cast<__half*>(stage + 2048 + sw64_h(k, lane)) = __float2half_rn(v[k]);
    }
    __syncwarp();
    if (sym && on_diag) {
      // Lower triangle of the diagonal block takes the upper-triangle values (exact symmetry).
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k < lane) *reinterpret_cast<__half*>(stage + sw64_h(lane, k)) = *reinterpret_cast<const __half*>(stage + sw64_h(k, lane));
      __syncwarp();
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&job.tmD, sbuf, j0, row0);
      if (upper) tma_store_2d(&job.tmD, sbuf + 2048, row0, j0);
      if (has_d2 && !on_diag) {
        tma_store_2d(&job.tmD2, sbuf, j0, row0);
        if (upper) tma_store_2d(&job.tmD2, sbuf + 2048, row0, j0);
      }
      bulk_commit();
    }
    if (has_d2 && on_diag) {
      // D2 = D + a I: only the diagonal elements of this block differ.
      float dv = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k == lane) dv = v[k] + s.d2;
      bad |= row_ok && !fp16_ok(dv);
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
      *reinterpret_cast<__half*>(stage + sw64_h(lane, lane)) = __float2half_rn(dv);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&job.tmD2, sbuf, j0, row0);
        bulk_commit();
      }
    }
  }
}

// ---------------------------------------------------------------------------- the kernel

template <int BN, int CG>
__device__ __forceinline__ void gemm_tc_body(const GemmLaunch& p) {
  using C = Cfg<BN, CG>;
  constexpr bool kPair = CG == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi_stage = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + C::kEpiBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0 = the pair's leader (issues the MMAs)
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nunits = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * CG);  // every epilogue warp of the pair releases the accumulator
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) tmem_alloc_pair(tmem_slot, C::kTmemCols);
    else tmem_alloc(tmem_slot, C::kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers are initialised before anyone signals them
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
      for (int t = unit; ok && t < p.ntiles; t += nunits) {
        const TileRef tr = tile_at(p, t, BN, C::kTileM);
        if (tr.skip) continue;
        const GemmJob* job = tr.job;
        const int nkb = (job->K + kBK - 1) / kBK;
        const bool bmn = (job->flags & kJobBMnMajor) != 0;
        const int m0 = tr.tm * C::kTileM + static_cast<int>(rank) * kBM;   // this CTA's 128 rows of A
        const int n0 = tr.tn * BN + static_cast<int>(rank) * C::kBRows;   // this CTA's rows of B
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, kWaitLimitNs, true)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          if constexpr (kPair) {
            // Both CTAs' copies complete on the leader's full barrier; the leader expects both.
            const uint32_t bar = map_shared(smem_u32(&full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
            tma_load_2d_pair(sa, &job->tmA, kb * kBK, m0, bar);
            if (!bmn) {
              tma_load_2d_pair(sb, &job->tmB, kb * kBK, n0, bar);
            } else {
#pragma unroll
              for (int q = 0; q < C::kBRows / 64; ++q)
                tma_load_2d_pair(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, bar);
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
            tma_load_2d(sa, &job->tmA, kb * kBK, m0, &full[stage]);
            if (!bmn) {
              tma_load_2d(sb, &job->tmB, kb * kBK, n0, &full[stage]);
            } else {
#pragma unroll
              for (int q = 0; q < C::kBRows / 64; ++q) tma_load_2d(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, &full[stage]);
            }
          }
          issued[stage] = 1;
          issued_parity[stage] = phase;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && !kPair) {
        // Aborting: let every copy already issued land before the CTA's shared memory is released.
        for (int s = 0; s < C::kStages; ++s)
          if (issued[s]) wait_bounded(&full[s], issued_parity[s], abort_flag, p.status, kDrainLimitNs, false);
      }
      // (A pair's copies complete on the leader's barriers; the closing cluster barrier plus the
      // leader's drain keep both CTAs resident until then.)
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (the leader only)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = unit; ok && t < p.ntiles; t += nunits) {
        const TileRef tr = tile_at(p, t, BN, C::kTileM);
        if (tr.skip) continue;
        const GemmJob* job = tr.job;
        const int nkb = (job->K + kBK - 1) / kBK;
        const bool bmn = (job->flags & kJobBMnMajor) != 0;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, kWaitLimitNs, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t idesc = instr_desc<C::kTileM, BN>(bmn);
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
            if constexpr (kPair) mma_f16_pair(d_tmem, da, db, idesc, (kb > 0 || k > 0) ? 1u : 0u);
            else mma_f16(d_tmem, da, db, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          if constexpr (kPair) mma_commit_pair(&empty[stage]);
          else mma_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair) mma_commit_pair(&tfull[acc]);
        else mma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Make sure every MMA this thread issued has completed before tensor memory is freed.
      if constexpr (kPair) mma_commit_pair_local(drain);
      else mma_commit(drain);
      wait_bounded(drain, 0, abort_flag, p.status, kDrainLimitNs, false);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    bool bad = false;
    for (int t = unit; t < p.ntiles; t += nunits) {
      const TileRef tr = tile_at(p, t, BN, C::kTileM);
      if (tr.skip) continue;
      bool ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, p.status, kWaitLimitNs, true);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      epilogue_tile<BN>(p, *tr.job, tr.tm * C::kTileM + static_cast<int>(rank) * kBM, tr.tn, quarter, lane, taddr,
                        epi_stage + (warp - 2) * 4096, bad);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair) mbar_arrive_cluster(map_shared(smem_u32(&tempty[acc]), 0));
        else mbar_arrive(&tempty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait0();  // every bulk store / reduce of this warp has completed
    if (bad) atomicOr(p.status, kDevNonfinite);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) {
    // After an abort a pair CTA cannot see its own copies land (they signal the leader's barrier):
    // give any copy still in flight time to finish before shared memory is released.
    if (*abort_flag) {
      const unsigned long long t0 = globaltimer();
      while (globaltimer() - t0 < 2000000ull) __nanosleep(10000);
    }
    cluster_sync_all();  // neither CTA leaves while its peer may still signal it
  }
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GemmLaunch p) {
  gemm_tc_body<BN, 1>(p);
}

// CTA pairs: a 256 x 256 output tile per pair, one tcgen05.mma.cta_group::2 stream issued by the leader.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1) gemm_tc_pair_kernel(const __grid_constant__ GemmLaunch p) {
  gemm_tc_body<256, 2>(p);
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

// 2-D map: `inner` contiguous elements per row, `outer` rows `row_bytes` apart.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer, const char** err,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled is not available from the CUDA driver";
    return false;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled rejected an operand (alignment, stride or size)";
    return false;
  }
  return true;
}

}  // namespace

bool encode_job_maps(GemmJob& job, const void* a, int64_t lda, const void* b, int64_t ldb, bool b_mn_major,
                     int tile, const char** err) {
  const int b_rows = tile_cols(tile) / tile_ctas(tile);  // rows of the K-major B box one CTA loads
  if (!encode_2d(&job.tmA, a, static_cast<uint64_t>(job.K), static_cast<uint64_t>(job.M),
                 static_cast<uint64_t>(lda) * 2, kBK, kBM, err))
    return false;
  if (!b_mn_major)
    return encode_2d(&job.tmB, b, static_cast<uint64_t>(job.K), static_cast<uint64_t>(job.N),
                     static_cast<uint64_t>(ldb) * 2, kBK, static_cast<uint32_t>(b_rows), err);
  return encode_2d(&job.tmB, b, static_cast<uint64_t>(job.N), static_cast<uint64_t>(job.K),
                   static_cast<uint64_t>(ldb) * 2, 64, kBK, err);
}

bool encode_out_maps(GemmJob& job, const char** err) {
  if (job.D && !encode_2d(&job.tmD, job.D, static_cast<uint64_t>(job.N), static_cast<uint64_t>(job.M),
                          static_cast<uint64_t>(job.ldd) * 2, 32, 32, err, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_64B))
    return false;
  if (job.D2 && !encode_2d(&job.tmD2, job.D2, static_cast<uint64_t>(job.N), static_cast<uint64_t>(job.M),
                           static_cast<uint64_t>(job.ldd) * 2, 32, 32, err, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           CU_TENSOR_MAP_SWIZZLE_64B))
    return false;
  job.flags &= ~kJobTmaW;
  if ((job.flags & kJobFinal) && job.W && (reinterpret_cast<uintptr_t>(job.W) & 15) == 0 && (job.ldw & 3) == 0) {
    // W in the caller's orientation: M x N, or N x M when the matrix was worked on transposed.
    const bool tr = (job.flags & kJobFinalTrans) != 0;
    const uint64_t inner = static_cast<uint64_t>(tr ? job.M : job.N);
    const uint64_t outer = static_cast<uint64_t>(tr ? job.N : job.M);
    const char* e2 = nullptr;
    if (encode_2d(&job.tmW, job.W, inner, outer, static_cast<uint64_t>(job.ldw) * 4, 32, 32, &e2,
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B))
      job.flags |= kJobTmaW;
  }
  return true;
}

int gemm_max_units(int tile, int sms) {
  if (tile != kTilePair256) return sms;
  // CTA pairs need two SMs of one GPC each: ask how many such clusters fit at once.
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sms / 2;
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(gemm_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<256, 2>::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return sms / 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = Cfg<256, 2>::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  cached[dev] = std::min(n, sms / 2);
  return cached[dev];
}

cudaError_t launch_gemm(const GemmLaunch& p, int tile, int units, cudaStream_t stream) {
  if (p.ntiles <= 0) return cudaSuccess;
  cudaError_t e;
  switch (tile) {
    case kTilePair256:
      e = cudaFuncSetAttribute(gemm_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<256, 2>::kSmemBytes);
      if (e != cudaSuccess) return e;
      gemm_tc_pair_kernel<<<2 * units, 192, Cfg<256, 2>::kSmemBytes, stream>>>(p);
      break;
    case kTileSingle256:
      e = cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<256, 1>::kSmemBytes);
      if (e != cudaSuccess) return e;
      gemm_tc_kernel<256><<<units, 192, Cfg<256, 1>::kSmemBytes, stream>>>(p);
      break;
    default:
      e = cudaFuncSetAttribute(gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<128, 1>::kSmemBytes);
      if (e != cudaSuccess) return e;
      gemm_tc_kernel<128><<<units, 192, Cfg<128, 1>::kSmemBytes, stream>>>(p);
      break;
  }
  return cudaGetLastError();
}

}  // namespace dmuon
