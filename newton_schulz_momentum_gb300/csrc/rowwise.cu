// HBM-bound stages of the Muon update, grouped over all matrices of a call:
//   1. momentum_sumsq   M <- beta * M + G and per-chunk partial sums of M^2 (pwwt.cn post, section 2:
//                       keep a momentum of the gradient);
//   2. finalize_norms   ||M||_F = sqrt(sum of partials) per matrix, in a fixed order, and
//                       inv = 1 / (||M||_F + eps) ("Newton-Schulz 变体", section "精度流水线");
//   3. normalize_cast   X = fp16(M * inv), written in the m <= n orientation (tall matrices are
//                       transposed through shared memory) -- the fp16 input of the iteration.
// Reductions are deterministic: fixed chunking (per matrix, so a matrix's norm does not depend on the
// rest of the call), fixed tree order, no atomics. The planned path launches all three programmatically
// (each waits for the preceding grid before touching global memory); the allocation-free entry launches
// the same bodies plainly.
#include "internal.h"
#include "tc_ptx.h"

namespace dmuon {
namespace {

constexpr int kThreads = 256;

// Index of the matrix whose [prefix[i], prefix[i+1]) range holds `item`.
__device__ __forceinline__ int find_matrix(const int64_t* prefix, int n, int64_t item) {
  int lo = 0, hi = n;  // prefix[lo] <= item < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void load8_grad(const void* g, int gdtype, int64_t e, float (&out)[8]) {
  if (gdtype == 1) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(g) + e));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = __uint_as_float(w[k] << 16);
      out[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e + 4));
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  }
}

__device__ __forceinline__ float load1_grad(const void* g, int gdtype, int64_t e) {
  if (gdtype == 1) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(g)[e]) << 16);
  return static_cast<const float*>(g)[e];
}

template <typename T>
__device__ __forceinline__ T block_sum(T v, T* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  T total = 0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kThreads / 32; ++w) total += scratch[w];
  }
  return total;  // valid in thread 0
}

__global__ void __launch_bounds__(kThreads) momentum_sumsq_kernel(const RowLaunch p) {
  __shared__ float red[kThreads / 32];
  const int64_t chunk = p.chunk_base + blockIdx.x;
  const int mi = find_matrix(p.chunk_prefix, p.nmats, chunk);
  if (!dev_check(mi >= 0 && mi < p.nmats, p.check_status)) return;
  const RowMat mt = p.mats[mi];
  const int64_t local = chunk - p.chunk_prefix[mi];
  if (!dev_check(local >= 0 && local < mt.part_count && mt.part_begin + local < p.npartials, p.check_status)) return;
  const int64_t numel = mt.rows * mt.cols;
  const int64_t begin = local * kChunkElems;
  const int64_t end = min(begin + static_cast<int64_t>(kChunkElems), numel);
  const bool has_g = mt.G != nullptr;
  const float beta = p.beta;
  float acc = 0.f;
  int64_t scalar_from = begin;
  if (mt.vec_ok) {
    const int64_t vend = begin + ((end - begin) / 8) * 8;
    // 4 groups of 8 elements in flight per thread.
    int64_t e = begin + threadIdx.x * 8;
    for (; e + 3 * kThreads * 8 + 8 <= vend; e += 4 * kThreads * 8) {
      float g[4][8];
      float4 m[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t eu = e + u * kThreads * 8;
        if (has_g) load8_grad(mt.G, mt.gdtype, eu, g[u]);
        m[u][0] = *reinterpret_cast<const float4*>(mt.M + eu);
        m[u][1] = *reinterpret_cast<const float4*>(mt.M + eu + 4);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float* mv = reinterpret_cast<float*>(m[u]);
        if (has_g) {
#pragma unroll
          for (int k = 0; k < 8; ++k) mv[k] = fmaf(beta, mv[k], g[u][k]);
          const int64_t eu = e + u * kThreads * 8;
          *reinterpret_cast<float4*>(mt.M + eu) = m[u][0];
          *reinterpret_cast<float4*>(mt.M + eu + 4) = m[u][1];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(mv[k], mv[k], acc);
      }
    }
    for (; e + 8 <= vend; e += kThreads * 8) {
      float g[8];
      float4 m[2];
      if (has_g) load8_grad(mt.G, mt.gdtype, e, g);
      m[0] = *reinterpret_cast<const float4*>(mt.M + e);
      m[1] = *reinterpret_cast<const float4*>(mt.M + e + 4);
      float* mv = reinterpret_cast<float*>(m);
      if (has_g) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mv[k] = fmaf(beta, mv[k], g[k]);
        *reinterpret_cast<float4*>(mt.M + e) = m[0];
        *reinterpret_cast<float4*>(mt.M + e + 4) = m[1];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(mv[k], mv[k], acc);
    }
    scalar_from = vend;
  }
  for (int64_t e = scalar_from + threadIdx.x; e < end; e += kThreads) {
    float m = mt.M[e];
    if (has_g) {
      m = fmaf(beta, m, load1_grad(mt.G, mt.gdtype, e));
      mt.M[e] = m;
    }
    acc = fmaf(m, m, acc);
  }
  const float total = block_sum(acc, red);
  if (threadIdx.x == 0) p.partials[mt.part_begin + local] = total;
}

// The momentum pass streamed through shared memory: one thread moves 4096-element slices of M and G
// into a ring of kRingSlots slots with bulk copies (cp.async.bulk, completion on an mbarrier), and the
// CTA updates M from the slot and writes it back with coalesced 16-byte stores. The bytes in flight are
// set by the ring, not by registers: up to 3 x 24 KB per CTA with bf16 gradients, two CTAs per SM. Every
// wait is bounded; on expiry the CTA sets kDevTimeout, lets its copies land and returns.
constexpr int kSub = 4096;       // elements per ring slot
constexpr int kRingSlots = 3;
constexpr int kSlotBytes = kSub * 4 * 2;  // M (fp32) and G (up to fp32)
constexpr int kBulkSmem = kRingSlots * kSlotBytes + 64;
static_assert(kChunkElems % kSub == 0, "a chunk is a whole number of slots");

__global__ void __launch_bounds__(kThreads, 2) momentum_sumsq_bulk_kernel(const RowLaunch p) {
  // Launched with programmatic stream serialisation: the next pass may be scheduled now; this one waits
  // for the preceding grid before touching global memory.
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ float red[kThreads / 32];
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRingSlots * kSlotBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kRingSlots);
  const int64_t chunk = p.chunk_base + blockIdx.x;
  const int mi = find_matrix(p.chunk_prefix, p.nmats, chunk);
  if (!dev_check(mi >= 0 && mi < p.nmats, p.check_status)) return;
  const RowMat mt = p.mats[mi];
  const int64_t local = chunk - p.chunk_prefix[mi];
  if (!dev_check(local >= 0 && local < mt.part_count && mt.part_begin + local < p.npartials && mt.chunk > 0,
                 p.check_status))
    return;
  const int64_t numel = mt.rows * mt.cols;
  const int64_t begin = local * mt.chunk;
  const int64_t end = min(begin + mt.chunk, numel);
  const bool has_g = mt.G != nullptr;
  const int gsize = mt.gdtype == 1 ? 2 : 4;
  const float beta = p.beta;
  // Slices cover a multiple of 8 elements (whole 16-byte units of either gradient type); the last
  // few elements of a matrix go through plain loads below.
  // Rows that are not 16-byte vectorisable never reach the bulk copies (plain loads for the whole chunk).
  const int64_t nbulk = mt.vec_ok ? ((end - begin) & ~int64_t(7)) : 0;
  const int nsub = static_cast<int>((nbulk + kSub - 1) / kSub);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingSlots; ++s) ptx::mbar_init(&full[s], 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  uint64_t policy = 0;
  if (threadIdx.x == 0) policy = ptx::l2_policy_evict_first();
  auto issue = [&](int i) {  // thread 0: slice i into slot i % kRingSlots
    const int s = i % kRingSlots;
    const int64_t e0 = begin + static_cast<int64_t>(i) * kSub;
    const uint32_t cnt = static_cast<uint32_t>(min(static_cast<int64_t>(kSub), nbulk - static_cast<int64_t>(i) * kSub));
    const uint32_t mb = cnt * 4u, gb = has_g ? cnt * static_cast<uint32_t>(gsize) : 0u;
    uint8_t* slot = ring + s * kSlotBytes;
    ptx::mbar_arrive_expect_tx(&full[s], mb + gb);
    ptx::bulk_load_hint(ptx::smem_u32(slot), mt.M + e0, mb, &full[s], policy);
    if (has_g)
      ptx::bulk_load_hint(ptx::smem_u32(slot + kSub * 4), static_cast<const uint8_t*>(mt.G) + e0 * gsize, gb, &full[s],
                          policy);
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < min(kRingSlots, nsub); ++issued) issue(issued);

  float acc = 0.f;
  bool ok = true;
  int done = 0;
  for (; done < nsub; ++done) {
    const int s = done % kRingSlots;
    const uint32_t parity = static_cast<uint32_t>(done / kRingSlots) & 1u;
    const bool got = ptx::wait_bounded(&full[s], parity, abort_flag, p.status, ptx::kWaitLimitNs, true);
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    const int64_t e0 = begin + static_cast<int64_t>(done) * kSub;
    const int cnt4 = static_cast<int>(min(static_cast<int64_t>(kSub), nbulk - static_cast<int64_t>(done) * kSub)) / 4;
    const float4* sm = reinterpret_cast<const float4*>(ring + s * kSlotBytes);
    const uint8_t* sg = ring + s * kSlotBytes + kSub * 4;
    for (int q = threadIdx.x; q < cnt4; q += kThreads) {
      float4 m = sm[q];
      if (has_g) {
        float g[4];
        if (mt.gdtype == 1) {
          const uint2 u = reinterpret_cast<const uint2*>(sg)[q];
          g[0] = __uint_as_float(u.x << 16), g[1] = __uint_as_float(u.x & 0xFFFF0000u);
          g[2] = __uint_as_float(u.y << 16), g[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
          const float4 v = reinterpret_cast<const float4*>(sg)[q];
          g[0] = v.x, g[1] = v.y, g[2] = v.z, g[3] = v.w;
        }
        m.x = fmaf(beta, m.x, g[0]);
        m.y = fmaf(beta, m.y, g[1]);
        m.z = fmaf(beta, m.z, g[2]);
        m.w = fmaf(beta, m.w, g[3]);
        __stcs(reinterpret_cast<float4*>(mt.M + e0) + q, m);
      }
      acc = fmaf(m.x, m.x, acc);
      acc = fmaf(m.y, m.y, acc);
      acc = fmaf(m.z, m.z, acc);
      acc = fmaf(m.w, m.w, acc);
    }
    __syncthreads();  // every thread is done with slot s
    if (threadIdx.x == 0 && issued < nsub) issue(issued++);
  }
  if (!ok) {
    // Let every copy already issued land before the CTA's shared memory is released.
    if (threadIdx.x == 0)
      for (int i = done; i < issued; ++i)
        ptx::wait_bounded(&full[i % kRingSlots], static_cast<uint32_t>(i / kRingSlots) & 1u, abort_flag, p.status,
                          ptx::kDrainLimitNs, false);
    __syncthreads();
    return;
  }
  for (int64_t e = begin + nbulk + threadIdx.x; e < end; e += kThreads) {
    float m = mt.M[e];
    if (has_g) {
      m = fmaf(beta, m, load1_grad(mt.G, mt.gdtype, e));
      mt.M[e] = m;
    }
    acc = fmaf(m, m, acc);
  }
  const float total = block_sum(acc, red);
  if (threadIdx.x == 0) p.partials[mt.part_begin + local] = total;
}

__device__ __forceinline__ void finalize_norms_body(const RowLaunch& p) {
  __shared__ double red[kThreads / 32];
  if (!dev_check(static_cast<int>(blockIdx.x) < p.nmats, p.check_status)) return;
  const RowMat mt = p.mats[blockIdx.x];
  if (!dev_check(mt.part_begin >= 0 && mt.part_begin + mt.part_count <= p.npartials, p.check_status)) return;
  double s = 0.0;
  for (int k = threadIdx.x; k < mt.part_count; k += kThreads) s += static_cast<double>(p.partials[mt.part_begin + k]);
  const double total = block_sum(s, red);
  if (threadIdx.x == 0) {
    const double norm = sqrt(total);
    p.norms[blockIdx.x] = static_cast<float>(norm);
    p.inv[blockIdx.x] = static_cast<float>(1.0 / (norm + static_cast<double>(p.eps)));
    if (p.norms_out) p.norms_out[blockIdx.x] = static_cast<float>(norm);
  }
}

__global__ void __launch_bounds__(kThreads) finalize_norms_kernel(const RowLaunch p) { finalize_norms_body(p); }

// The same, launched with programmatic stream serialisation (the planned path).
__global__ void __launch_bounds__(kThreads) finalize_norms_pdl_kernel(const RowLaunch p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  finalize_norms_body(p);
}

__device__ __forceinline__ void store_half4(__half* dst, float a, float b, float c, float d) {
  __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = u;
}

__device__ __forceinline__ void normalize_cast_body(const RowLaunch& p) {
  __shared__ float tile[kCastTile][kCastTile + 1];
  const int64_t t = p.tile_base + blockIdx.x;
  const int mi = find_matrix(p.tile_prefix, p.nmats, t);
  if (!dev_check(mi >= 0 && mi < p.nmats, p.check_status)) return;
  const RowMat mt = p.mats[mi];
  const int64_t local = t - p.tile_prefix[mi];
  const int64_t tiles_c = (mt.cols + kCastTile - 1) / kCastTile;
  const int64_t r0 = (local / tiles_c) * kCastTile;
  const int64_t c0 = (local % tiles_c) * kCastTile;
  if (!dev_check(local >= 0 && r0 < mt.rows && c0 < mt.cols, p.check_status)) return;
  const float inv = p.inv[mi];
  // 16-byte loads of M need rows of a multiple of 4 floats; 8-byte stores of X need rows of X
  // (ldx halves) of a multiple of 4. Either condition failing falls back to scalar accesses.
  const bool vec_in = mt.vec_ok && (mt.cols & 3) == 0;
  const bool vec_out = (mt.ldx & 3) == 0 && (reinterpret_cast<uintptr_t>(mt.X) & 7) == 0;
  const int tx = threadIdx.x & 15;   // 4-column group within the tile
  const int ty = threadIdx.x >> 4;   // row within a 16-row pass

  constexpr int kPasses = kCastTile / 16;
  const int64_t c = c0 + tx * 4;
  // Interior tiles (every row and column in range, 16-byte rows): all of a thread's loads are issued
  // before any use, so each thread keeps kPasses 16-byte reads in flight.
  const bool interior = vec_in && r0 + kCastTile <= mt.rows && c0 + kCastTile <= mt.cols;

  if (!mt.trans) {
    if (interior && vec_out) {
      float4 v[kPasses];
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass)
        v[pass] = __ldcs(reinterpret_cast<const float4*>(mt.M + (r0 + pass * 16 + ty) * mt.cols + c));
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass)
        store_half4(mt.X + (r0 + pass * 16 + ty) * mt.ldx + c, v[pass].x * inv, v[pass].y * inv, v[pass].z * inv,
                    v[pass].w * inv);
      return;
    }
    for (int pass = 0; pass < kPasses; ++pass) {
      const int64_t r = r0 + pass * 16 + ty;
      if (r >= mt.rows) continue;
      const float* src = mt.M + r * mt.cols + c;
      __half* dst = mt.X + r * mt.ldx + c;
      if (vec_in && vec_out && c + 4 <= mt.cols) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        store_half4(dst, v.x * inv, v.y * inv, v.z * inv, v.w * inv);
      } else {
        for (int k = 0; k < 4; ++k)
          if (c + k < mt.cols) dst[k] = __float2half_rn(src[k] * inv);
      }
    }
    return;
  }

  // Tall matrix: X (cols x rows) = (M * inv)^T.
  if (interior) {
    float4 v[kPasses];
#pragma unroll
    for (int pass = 0; pass < kPasses; ++pass)
      v[pass] = __ldcs(reinterpret_cast<const float4*>(mt.M + (r0 + pass * 16 + ty) * mt.cols + c));
#pragma unroll
    for (int pass = 0; pass < kPasses; ++pass) {
      const int rr = pass * 16 + ty;
      tile[rr][tx * 4 + 0] = v[pass].x;
      tile[rr][tx * 4 + 1] = v[pass].y;
      tile[rr][tx * 4 + 2] = v[pass].z;
      tile[rr][tx * 4 + 3] = v[pass].w;
    }
  } else {
    for (int pass = 0; pass < kPasses; ++pass) {
      const int rr = pass * 16 + ty;
      const int64_t r = r0 + rr;
      if (r >= mt.rows) continue;
      const float* src = mt.M + r * mt.cols + c;
      if (vec_in && c + 4 <= mt.cols) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        tile[rr][tx * 4 + 0] = v.x;
        tile[rr][tx * 4 + 1] = v.y;
        tile[rr][tx * 4 + 2] = v.z;
        tile[rr][tx * 4 + 3] = v.w;
      } else {
        for (int k = 0; k < 4; ++k)
          if (c + k < mt.cols) tile[rr][tx * 4 + k] = src[k];
      }
    }
  }
  __syncthreads();
  for (int pass = 0; pass < kCastTile / 16; ++pass) {
    const int cc = pass * 16 + ty;      // row of X (column of M)
    const int rr = tx * 4;              // first of 4 consecutive columns of X (rows of M)
    const int64_t xr = c0 + cc;
    const int64_t xc = r0 + rr;
    if (xr >= mt.cols) continue;
    __half* dst = mt.X + xr * mt.ldx + xc;
    if (vec_out && xc + 4 <= mt.rows) {
      store_half4(dst, tile[rr][cc] * inv, tile[rr + 1][cc] * inv, tile[rr + 2][cc] * inv, tile[rr + 3][cc] * inv);
    } else {
      for (int k = 0; k < 4; ++k)
        if (xc + k < mt.rows) dst[k] = __float2half_rn(tile[rr + k][cc] * inv);
    }
  }
}

__global__ void __launch_bounds__(kThreads) normalize_cast_kernel(const RowLaunch p) { normalize_cast_body(p); }

// The same, launched with programmatic stream serialisation (the planned path).
__global__ void __launch_bounds__(kThreads) normalize_cast_pdl_kernel(const RowLaunch p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  normalize_cast_body(p);
}

// Sum of squares of one shard (columns [bounds[t], bounds[t+1]) of the oriented matrix) over one slab of
// kShardSlab oriented rows. Consecutive threads read consecutive addresses in both orientations.
__global__ void __launch_bounds__(kThreads) shard_sumsq_kernel(const ShardSumsqLaunch p) {
  __shared__ float red[kThreads / 32];
  const int t = blockIdx.y, s = blockIdx.x;
  const int64_t m = p.trans ? p.cols : p.rows;
  const int64_t c0 = p.bounds[t], c1 = p.bounds[t + 1];
  const int64_t r0 = static_cast<int64_t>(s) * kShardSlab, r1 = min(r0 + kShardSlab, m);
  const int64_t w = c1 - c0, h = r1 - r0;
  float acc = 0.f;
  for (int64_t e = threadIdx.x; e < w * h; e += kThreads) {
    float v;
    if (!p.trans) v = p.x[(r0 + e / w) * p.cols + c0 + e % w];   // oriented (i, j) = caller (i, j)
    else v = p.x[(c0 + e / h) * p.cols + r0 + e % h];           // oriented (i, j) = caller (j, i)
    acc = fmaf(v, v, acc);
  }
  const float total = block_sum(acc, red);
  if (threadIdx.x == 0) p.partials[t * p.slabs + s] = total;
}

__global__ void __launch_bounds__(kThreads) tp_reduce_kernel(const TpReduceLaunch p) {
  const int64_t i = blockIdx.x;
  for (int64_t j = threadIdx.x; j < p.m; j += kThreads) {
    const int64_t a = min(i, j), b = max(i, j);
    float acc = 0.f;
    for (int t = 0; t < p.shards; ++t) acc += p.P[t * p.plane + a * p.ldp + b];
    p.R[i * p.ldr + j] = __float2half_rn(acc);
  }
}

// One 64 KB chunk of one gather item per CTA. With both addresses 16-byte aligned each thread issues
// four 16-byte host loads before their stores (16 KB in flight per CTA and round, four rounds per
// chunk) to cover the host link's latency; the unaligned remainder goes byte by byte.
__global__ void __launch_bounds__(kThreads) h2d_gather_kernel(const GatherItem* items, const int64_t* prefix, int n) {
  static_assert(kGatherChunk % (int64_t(kThreads) * 16 * 4) == 0, "a chunk is whole rounds of four 16-byte loads");
  const int64_t chunk = blockIdx.x;
  const int i = find_matrix(prefix, n, chunk);
  const GatherItem it = items[i];
  const int64_t begin = (chunk - prefix[i]) * kGatherChunk;
  const int64_t end = min(begin + kGatherChunk, it.bytes);
  const uint8_t* __restrict__ src = static_cast<const uint8_t*>(it.src);
  uint8_t* __restrict__ dst = static_cast<uint8_t*>(it.dst);
  int64_t from = begin;
  if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
    const int64_t vend = begin + ((end - begin) & ~int64_t(15));
    constexpr int64_t kStride = int64_t(kThreads) * 16;
    for (int64_t b0 = begin + threadIdx.x * 16; b0 < vend; b0 += 4 * kStride) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (b0 + u * kStride < vend) v[u] = __ldcs(reinterpret_cast<const uint4*>(src + b0 + u * kStride));
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (b0 + u * kStride < vend) *reinterpret_cast<uint4*>(dst + b0 + u * kStride) = v[u];
    }
    from = vend;
  }
  for (int64_t b = from + threadIdx.x; b < end; b += kThreads) dst[b] = src[b];
}

// One thread waits, through the same bounded wait the library's kernels use, on an mbarrier phase that
// nothing completes: after limit_ns it gives up and records kDevTimeout in the status word.

__global__ void selftest_wait_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) ptx::wait_bounded(&bar, 0, &abort_flag, status, limit_ns, true);
}

}  // namespace

cudaError_t launch_shard_sumsq(const ShardSumsqLaunch& p, cudaStream_t stream) {
  shard_sumsq_kernel<<<dim3(static_cast<unsigned>(p.slabs), static_cast<unsigned>(p.shards)), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tp_reduce(const TpReduceLaunch& p, cudaStream_t stream) {
  tp_reduce_kernel<<<static_cast<unsigned>(p.m), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_h2d_gather(const GatherItem* items, const int64_t* prefix, int n, int64_t nchunks,
                              cudaStream_t stream) {
  if (nchunks <= 0) return cudaSuccess;
  h2d_gather_kernel<<<static_cast<unsigned>(nchunks), kThreads, 0, stream>>>(items, prefix, n);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned* status, unsigned long long limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

// A launch with programmatic stream serialisation (the kernel waits for the preceding grid itself).
template <typename Kernel>
cudaError_t launch_programmatic(Kernel kernel, unsigned grid, unsigned smem, const RowLaunch& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_momentum_sumsq(const RowLaunch& p, int64_t nchunks, cudaStream_t stream) {
  if (nchunks <= 0) return cudaSuccess;
  if (p.status) {
    cudaError_t e = cudaFuncSetAttribute(momentum_sumsq_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBulkSmem);
    if (e != cudaSuccess) return e;
    e = launch_programmatic(momentum_sumsq_bulk_kernel, static_cast<unsigned>(nchunks), kBulkSmem, p, stream);
    if (e != cudaSuccess) return e;
  } else {
    momentum_sumsq_kernel<<<static_cast<unsigned>(nchunks), kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize_norms(const RowLaunch& p, cudaStream_t stream, bool programmatic) {
  if (programmatic) {
    const cudaError_t e = launch_programmatic(finalize_norms_pdl_kernel, static_cast<unsigned>(p.nmats), 0, p, stream);
    if (e != cudaSuccess) return e;
  } else {
    finalize_norms_kernel<<<p.nmats, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_normalize_cast(const RowLaunch& p, int64_t ntiles, cudaStream_t stream, bool programmatic) {
  if (ntiles <= 0) return cudaSuccess;
  if (programmatic) {
    const cudaError_t e = launch_programmatic(normalize_cast_pdl_kernel, static_cast<unsigned>(ntiles), 0, p, stream);
    if (e != cudaSuccess) return e;
  } else {
    normalize_cast_kernel<<<static_cast<unsigned>(ntiles), kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dmuon
