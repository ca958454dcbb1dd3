// Grouped fp16 tensor-core GEMM / SYRK for sm_103a: TMA -> shared memory ring -> tcgen05.mma with
// fp32 accumulators in tensor memory -> tcgen05.ld epilogue.
//
// Every product of both Newton-Schulz forms runs here ("Newton-Schulz 变体" page: X X^T and R^2 as
// symmetric products -- "R 是对称的 ... SYRK" in section "Gram 空间 NS" -- plus Z Q, Z R, S Z, Q X,
// and B X for the direct form). One launch walks a list of 128 x BN output tiles drawn from many
// jobs (one job = one product on one matrix), so all matrices a rank owns advance one phase per
// launch.
//
// CTA layout (192 threads, or 320 for 128 x 128 and 128 x 64 tiles; one persistent CTA per SM):
//   warp 0      TMA producer: one thread streams 128 x 64 A tiles and BN x 64 B tiles into a
//               STAGES-deep ring of 128-byte-swizzled shared memory buffers.
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma (M=128, N=BN, K=16) into one
//               of two BN-column fp32 accumulators and commits completion to mbarriers.
//   warps 2-5   epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..+31, i.e.
//               one output row per thread), combine with the step's scalars and an optional fp16
//               addend, store fp16 (mirrored for symmetric outputs) or update the fp32 weights.
//               128 x 128 and 128 x 64 tiles run only in launches too small to fill the machine,
//               where the epilogue is the critical path: warps 2-9, two per lane quarter, each half the
//               columns.
// The accumulator is double-buffered so a tile's epilogue overlaps the next tile's main loop.
// Four tile configurations: 256 x 256 tiles on CTA pairs (a cluster of two; tcgen05.mma.cta_group::2,
// each CTA holding half of A and half of B per stage), 128 x 256, 128 x 128 and 128 x 64 on single CTAs;
// the planner takes the pair tiles unless a launch could not fill the pairs or its products are at most
// 128 wide, and halves 128 x 128 tiles to 128 x 64 when they would fill under half of the SMs. Launches are programmatic: a grid lets the next phase be scheduled at entry, and sets up its
// barriers and tensor memory (and prefetches its first tensor maps) before waiting for the previous
// grid.
//
// Every mbarrier wait is bounded: after kWaitLimitNs the waiting thread raises a CTA-wide abort
// flag and sets kDevTimeout in the device status word, all roles leave their loops, in-flight copies
// and MMAs are drained (again with a bound), tensor memory is freed and the kernel returns.
#include <algorithm>
#include <cstdio>

#include "internal.h"
#include "tc_ptx.h"

namespace dmuon {
namespace {

using namespace ptx;

// BN: output tile width. CG: CTAs per MMA (1, or 2 for a CTA pair sharing one 256 x BN tile with
// tcgen05.mma.cta_group::2; each CTA then holds 128 rows of A and BN / 2 rows of B per stage).
template <int BN, int CG>
struct Cfg {
  static constexpr int kBRows = BN / CG;         // rows of the B tile held by one CTA
  static constexpr int kTileM = kBM * CG;        // output rows per tile
  static constexpr int kABytes = kBM * kBK * 2;  // 16 KB
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // Epilogue warps: one per TMEM lane quarter, or two (each draining half of the tile's columns) for the
  // 128 x 128 and 128 x 64 tiles of launches too small to fill the machine, whose epilogue is their
  // critical path; those also double-buffer their staging (a chunk is written while the previous one's
  // stores read the other buffer) and keep fewer ring stages to make room.
  static constexpr bool kSmallTile = BN <= 128 && CG == 1;
  static constexpr int kStages = kSmallTile ? (BN == 64 ? 6 : 5) : (kStageBytes <= 32768) ? 6 : 4;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators of BN fp32 columns
  static constexpr int kEpiWarps = kSmallTile ? 8 : 4;
  static constexpr int kEpiBufs = kSmallTile ? 2 : 1;  // 4 KB staging buffers per epilogue warp
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kEpiBytes = kEpiWarps * 4096 * kEpiBufs;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiBytes + kBarrierBytes + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");
  static_assert(kStages >= 3, "the MMA issuer checks three ring slots at a time");
  static_assert((2 * kStages + 5) * 8 + 8 <= kBarrierBytes, "barrier area too small");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// ---------------------------------------------------------------------------- tile bookkeeping

constexpr int kSingleBand = 8;  // tile rows per raster band of a single-job launch
// L2 priorities of the TMA traffic: operand loads that other tiles of the launch re-read are kept
// (evict_last), epilogue stores and reduce-adds are streamed through (evict_first).
constexpr bool kKeepA = true;
constexpr bool kKeepB = true;
constexpr bool kStreamOut = true;

struct TileRef {
  const GemmJob* job;
  int tm, tn;
  bool skip;  // a lower-triangle tile of a symmetric single-job launch: nobody touches it
};

// Tile t of the launch. In the checked build a tile whose job index lies outside the job table, or which
// does not intersect its product's output (or whose product has no K), is skipped by every role alike and
// recorded as a range failure.
__device__ __forceinline__ TileRef tile_at(const GemmLaunch& p, int t, int bn, int tile_m) {
  TileRef r;
  if (p.jobs != nullptr) {
    const GemmTile g = p.tiles[t];
    const bool job_ok = dev_check(g.job >= 0 && g.job < p.njobs, p.status);
    r.job = p.jobs + (job_ok ? g.job : 0);
    r.tm = g.tm;
    r.tn = g.tn;
    r.skip = !job_ok;
  } else {
    // One job: bands of kSingleBand tile rows, walked column by column, so the tiles in flight at
    // once form a near-square block whose A and B panels stay in L2 together.
    r.job = &p.single;
    const int tiles_n = p.single.tiles_n;
    const int g0 = (t / (kSingleBand * tiles_n)) * kSingleBand;
    const int bh = min(kSingleBand, p.tiles_m - g0);
    const int u = t - g0 * tiles_n;
    r.tn = u / bh;
    r.tm = g0 + (u - r.tn * bh);
    r.skip = (p.single.flags & kJobSymmetric) && (r.tn * bn + bn - 1 < r.tm * tile_m);
  }
  if (!r.skip)
    r.skip = !dev_check(r.tm >= 0 && r.tn >= 0 && r.tm * tile_m < r.job->M && r.tn * bn < r.job->N && r.job->K > 0,
                        p.status);
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


__device__ __forceinline__ void store_out(const CUtensorMap* map, uint32_t src, int c0, int c1, uint64_t pol) {
  if constexpr (kStreamOut) tma_store_2d_hint(map, src, c0, c1, pol);
  else tma_store_2d(map, src, c0, c1);
}
__device__ __forceinline__ void reduce_out(const CUtensorMap* map, uint32_t src, int c0, int c1, uint64_t pol) {
  if constexpr (kStreamOut) tma_reduce_add_2d_hint(map, src, c0, c1, pol);
  else tma_reduce_add_2d(map, src, c0, c1);
}

// The addend of this warp's first chunk of a tile (zeros when there is none). It was written by an earlier
// launch, so it is loaded before the tile's products complete and its latency hides behind them.
template <int BN>
__device__ __forceinline__ void load_first_e(const GemmLaunch& p, const GemmJob& job, int tile_row0, int tn,
                                             int quarter, int c_lo, int c_hi, int lane, uint4 (&e)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) e[q] = make_uint4(0, 0, 0, 0);
  const int row0 = tile_row0 + quarter * 32;
  const int i = row0 + lane;
  if (row0 >= job.M || i >= job.M || job.E == nullptr || recipe_scalars(p, job.recipe).e == 0.f) return;
  const int c = (job.flags & kJobSymmetric) ? max(c_lo, row0 - tn * BN) : c_lo;
  if (c < c_hi && tn * BN + c + 32 <= job.N) {
    const uint4* e4 = reinterpret_cast<const uint4*>(job.E + static_cast<int64_t>(i) * job.lde + tn * BN + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = e4[q];
  }
}

// One warp's share of a tile: the 32 rows of TMEM lane quarter `quarter`, columns [c_lo, c_hi) of the tile.
// `ecur` holds the first chunk's addend (load_first_e). With kBufs = 2 the warp's staging is two 4 KB
// buffers used in turn (`chunk` counts this warp's chunks across tiles), otherwise one.
template <int BN, int kBufs>
__device__ void epilogue_tile(const GemmLaunch& p, const GemmJob& job, int tile_row0, int tn, int quarter,
                              int c_lo, int c_hi, int lane, uint32_t taddr, uint8_t* stage_base, int& chunk,
                              uint4 (&ecur)[4], bool& bad, uint64_t pol_out) {
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
  const bool scale = s.acc != 1.f;
  // Overflow / NaN detection without per-element compares: an fp16 (or, for the final output, fp32)
  // value that is inf or NaN times zero is NaN, so one packed FMA per pair of outputs folds the check into
  // an accumulator tested once per tile. Columns past N hold zeros (out-of-range operand boxes are
  // zero-filled by TMA), so they never raise it.
  const __half2 zero2 = __float2half2_rn(0.f);
  __half2 chk16 = zero2;
  float chk32 = 0.f;

  // Symmetric outputs: chunks left of the diagonal block are produced by the mirrored stores of other
  // tiles, so this warp starts at its diagonal block (row0 and tn*BN are multiples of 32).
  int c = sym ? max(c_lo, row0 - tn * BN) : c_lo;
  uint4 enext[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) enext[q] = make_uint4(0, 0, 0, 0);

  for (; c < c_hi; c += 32) {
    const int j0 = tn * BN + c;
    if (j0 >= job.N) break;  // warp-uniform
    uint8_t* const stage = stage_base + (kBufs > 1 ? (chunk & 1) * 4096 : 0);
    const uint32_t sbuf = smem_u32(stage);
    ++chunk;
    const bool full = j0 + 32 <= job.N;
    const bool prefetch = erow != nullptr && c + 32 < c_hi && j0 + 64 <= job.N;
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
    } else if (scale) {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= s.acc;
    }
    if (s.diag != 0.f && j0 == row0) {  // only the block on the diagonal holds elements with j == i
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
      for (int k = 0; k < 32; ++k) chk32 = fmaf(v[k], 0.f, chk32);
      if (tma_w) {
        if (lane == 0) bulk_wait_read_allow<kBufs - 1>();  // this buffer's previous stores have read it
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
          if (p.w_alpha == 0.f) store_out(&job.tmW, sbuf, x, y, pol_out);
          else reduce_out(&job.tmW, sbuf, x, y, pol_out);
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

    uint32_t pk[16];  // the chunk's row rounded to fp16, two columns per word
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      pk[q] = pack_half2(v[2 * q], v[2 * q + 1]);
      chk16 = __hfma2(*reinterpret_cast<const __half2*>(&pk[q]), zero2, chk16);
    }
    const bool upper = sym && j0 > row0;  // strictly above the diagonal for every row of the block
    const bool on_diag = j0 == row0;      // the block holds the diagonal elements i == j

    if (lane == 0) bulk_wait_read_allow<kBufs - 1>();  // this buffer's previous stores have read it
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stage + sw64_h(lane, 8 * q)) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    if (upper) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        *reinterpret_cast<uint16_t*>(stage + 2048 + sw64_h(k, lane)) =
            static_cast<uint16_t>((k & 1) ? (pk[k >> 1] >> 16) : pk[k >> 1]);
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
      store_out(&job.tmD, sbuf, j0, row0, pol_out);
      if (upper) store_out(&job.tmD, sbuf + 2048, row0, j0, pol_out);
      if (has_d2 && !on_diag) {
        store_out(&job.tmD2, sbuf, j0, row0, pol_out);
        if (upper) store_out(&job.tmD2, sbuf + 2048, row0, j0, pol_out);
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
        store_out(&job.tmD2, sbuf, j0, row0, pol_out);
        bulk_commit();
      }
    }
  }
  bad |= __hisnan(__low2half(chk16)) || __hisnan(__high2half(chk16)) || chk32 != chk32;
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

  griddep_launch_dependents();  // the next phase's CTAs may start their set-up as this grid's SMs free up
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], C::kEpiWarps * CG);  // every epilogue warp of the pair releases the accumulator
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
  // The tile list and the tensor maps were written when the plan was bound, never by a kernel: fetch the
  // first tile's maps while the previous grid finishes.
  if (warp == 0 && lane == 0 && unit < p.ntiles) {
    const TileRef tr0 = tile_at(p, unit, BN, C::kTileM);
    if (!tr0.skip) prefetch_tensormap(&tr0.job->tmA);
    if (!tr0.skip) {
      prefetch_tensormap(&tr0.job->tmB);
      if (tr0.job->flags & kJobFinal) {
        if (tr0.job->flags & kJobTmaW) prefetch_tensormap(&tr0.job->tmW);
      } else {
        prefetch_tensormap(&tr0.job->tmD);
      }
    }
  }
  griddep_wait();  // the previous phase's outputs are complete and visible before any other global access

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per ring slot: a copy was issued / with which parity
      bool ok = true;
      // The leader's full barriers as seen from either CTA of a pair (consecutive 8-byte words).
      const uint32_t full_leader = kPair ? map_shared(smem_u32(&full[0]), 0) : 0u;
      const uint64_t pol_keep = l2_policy_evict_last();
      for (int t = unit; ok && t < p.ntiles; t += nunits) {
        const TileRef tr = tile_at(p, t, BN, C::kTileM);
        if (tr.skip) continue;
        const GemmJob* job = tr.job;
        const int nkb = (job->K + kBK - 1) / kBK;
        const bool bmn = (job->flags & kJobBMnMajor) != 0;
        const int m0 = tr.tm * C::kTileM + static_cast<int>(rank) * kBM;   // this CTA's 128 rows of A
        const int n0 = tr.tn * BN + static_cast<int>(rank) * C::kBRows;   // this CTA's rows of B
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          if constexpr (kPair) {
            // Both CTAs' copies complete on the leader's full barrier; the leader expects both.
            const uint32_t bar = full_leader + 8u * static_cast<uint32_t>(stage);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
            if constexpr (kKeepA) tma_load_2d_pair_hint(sa, &job->tmA, kb * kBK, m0, bar, pol_keep);
            else tma_load_2d_pair(sa, &job->tmA, kb * kBK, m0, bar);
            if (!bmn) {
              if constexpr (kKeepB) tma_load_2d_pair_hint(sb, &job->tmB, kb * kBK, n0, bar, pol_keep);
              else tma_load_2d_pair(sb, &job->tmB, kb * kBK, n0, bar);
            } else {
#pragma unroll
              for (int q = 0; q < C::kBRows / 64; ++q) {
                if constexpr (kKeepB) tma_load_2d_pair_hint(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, bar, pol_keep);
                else tma_load_2d_pair(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, bar);
              }
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
            if constexpr (kKeepA) tma_load_2d_hint(sa, &job->tmA, kb * kBK, m0, &full[stage], pol_keep);
            else tma_load_2d(sa, &job->tmA, kb * kBK, m0, &full[stage]);
            if (!bmn) {
              if constexpr (kKeepB) tma_load_2d_hint(sb, &job->tmB, kb * kBK, n0, &full[stage], pol_keep);
              else tma_load_2d(sb, &job->tmB, kb * kBK, n0, &full[stage]);
            } else {
#pragma unroll
              for (int q = 0; q < C::kBRows / 64; ++q) {
                if constexpr (kKeepB) tma_load_2d_hint(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, &full[stage], pol_keep);
                else tma_load_2d(sb + q * 8192, &job->tmB, n0 + q * 64, kb * kBK, &full[stage]);
              }
            }
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && !kPair) {
        // Aborting: let every copy already issued land before the CTA's shared memory is released.
        for (int s = 0; s < C::kStages; ++s)
          if ((issued >> s) & 1u)
            wait_bounded(&full[s], (issued_parity >> s) & 1u, abort_flag, p.status, kDrainLimitNs, false);
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
          // Full barriers are checked three ring slots at a time (this slot and the next two of the tile):
          // the probes overlap one another, and the MMA issue is interrupted by a barrier check once per
          // twelve MMAs instead of once per four. Short contractions (at most 8 slots) check slot by slot:
          // there the first MMAs issue as soon as their own slot lands rather than two slots later.
          const bool per_slot = nkb <= 8;
          if (per_slot || kb % 3 == 0) {
            const int s1 = stage + 1 == C::kStages ? 0 : stage + 1;
            const uint32_t p1 = stage + 1 == C::kStages ? phase ^ 1u : phase;
            const int s2 = s1 + 1 == C::kStages ? 0 : s1 + 1;
            const uint32_t p2 = s1 + 1 == C::kStages ? p1 ^ 1u : p1;
            const bool r0 = mbar_try_wait(&full[stage], phase);
            const bool r1 = per_slot || kb + 1 >= nkb || mbar_try_wait(&full[s1], p1);
            const bool r2 = per_slot || kb + 2 >= nkb || mbar_try_wait(&full[s2], p2);
            if (!(r0 && r1 && r2)) {
              if ((!r0 && !wait_bounded(&full[stage], phase, abort_flag, p.status, kWaitLimitNs, true)) ||
                  (!r1 && !wait_bounded(&full[s1], p1, abort_flag, p.status, kWaitLimitNs, true)) ||
                  (!r2 && !wait_bounded(&full[s2], p2, abort_flag, p.status, kWaitLimitNs, true))) {
                ok = false;
                break;
              }
            }
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
    // ------------------------------------------------------------------ epilogue (warps 2 .. 1 + kEpiWarps)
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    constexpr int kSpan = BN / (C::kEpiWarps / 4);    // columns per warp
    const int c_lo = ((warp - 2) >> 2) * kSpan;
    const uint64_t pol_out = l2_policy_evict_first();
    int acc = 0;
    uint32_t acc_phase = 0;
    bool bad = false;
    int chunk = 0;  // this warp's chunks so far (which staging buffer is next)
    for (int t = unit; t < p.ntiles; t += nunits) {
      const TileRef tr = tile_at(p, t, BN, C::kTileM);
      if (tr.skip) continue;
      const int tile_row0 = tr.tm * C::kTileM + static_cast<int>(rank) * kBM;
      uint4 efirst[4];
      load_first_e<BN>(p, *tr.job, tile_row0, tr.tn, quarter, c_lo, c_lo + kSpan, lane, efirst);
      bool ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, p.status, kWaitLimitNs, true);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      epilogue_tile<BN, C::kEpiBufs>(p, *tr.job, tile_row0, tr.tn, quarter, c_lo, c_lo + kSpan, lane, taddr,
                                     epi_stage + (warp - 2) * 4096 * C::kEpiBufs, chunk, efirst, bad, pol_out);
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
__global__ void __launch_bounds__(Cfg<BN, 1>::kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmLaunch p) {
  gemm_tc_body<BN, 1>(p);
}

// CTA pairs: a 256 x 256 output tile per pair, one tcgen05.mma.cta_group::2 stream issued by the leader.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<256, 2>::kThreads, 1) gemm_tc_pair_kernel(const __grid_constant__ GemmLaunch p) {
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

bool encode_tensor_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_outer, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                      const char** err) {
  return encode_2d(map, base, inner, outer, row_bytes, box_inner, box_outer, err, dtype, swizzle);
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
  cfg.blockDim = dim3(Cfg<256, 2>::kThreads, 1, 1);
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

// Launched with programmatic stream serialisation: consecutive phases overlap launch and set-up (the
// kernel waits for the previous grid before touching global memory).
template <typename Kernel>
cudaError_t launch_programmatic(Kernel kernel, unsigned grid, unsigned threads, unsigned smem, const GemmLaunch& p,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_gemm(const GemmLaunch& p, int tile, int units, cudaStream_t stream) {
  if (p.ntiles <= 0) return cudaSuccess;
  cudaError_t e;
  switch (tile) {
    case kTilePair256:
      e = cudaFuncSetAttribute(gemm_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<256, 2>::kSmemBytes);
      if (e != cudaSuccess) return e;
      e = launch_programmatic(gemm_tc_pair_kernel, 2 * units, Cfg<256, 2>::kThreads, Cfg<256, 2>::kSmemBytes, p, stream);
      break;
    case kTileSingle256:
      e = cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<256, 1>::kSmemBytes);
      if (e != cudaSuccess) return e;
      e = launch_programmatic(gemm_tc_kernel<256>, units, Cfg<256, 1>::kThreads, Cfg<256, 1>::kSmemBytes, p, stream);
      break;
    case kTileSingle64:
      e = cudaFuncSetAttribute(gemm_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<64, 1>::kSmemBytes);
      if (e != cudaSuccess) return e;
      e = launch_programmatic(gemm_tc_kernel<64>, units, Cfg<64, 1>::kThreads, Cfg<64, 1>::kSmemBytes, p, stream);
      break;
    default:
      e = cudaFuncSetAttribute(gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<128, 1>::kSmemBytes);
      if (e != cudaSuccess) return e;
      e = launch_programmatic(gemm_tc_kernel<128>, units, Cfg<128, 1>::kThreads, Cfg<128, 1>::kSmemBytes, p, stream);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dmuon
