// Fused AdamW over many tensors in one launch (DMuon "Core Concepts", section "1. Dedicated Ownership",
// step 6: every rank updates the parameters that are not Muon targets with AdamW). HBM-bound: per
// element it reads p, g, m, v once and writes p, m, v once (26 bytes with bf16 gradients, 28 with fp32).
//
// For step t, with decay = 1 - lr * weight_decay, step_size = lr / (1 - beta1^t), inv_bc2 =
// 1 / sqrt(1 - beta2^t) and 1 - beta1, 1 - beta2 formed in double on the host:
//   p <- p * decay;  m <- beta1 m + (1 - beta1) g;  v <- beta2 v + (1 - beta2) g^2;
//   p <- p - step_size * m / (sqrt(v) * inv_bc2 + eps)
#include "internal.h"

namespace dmuon {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int find_tensor(const int64_t* prefix, int n, int64_t item) {
  int lo = 0, hi = n;  // prefix[lo] <= item < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

struct AdamScalars {
  float decay, step_size, inv_bc2, beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
};

__device__ __forceinline__ void adam_update(float& p, float& m, float& v, float g, const AdamScalars& s) {
  p *= s.decay;
  m = fmaf(s.beta1, m, s.one_minus_beta1 * g);
  v = fmaf(s.beta2, v, s.one_minus_beta2 * g * g);
  p -= s.step_size * m / fmaf(sqrtf(v), s.inv_bc2, s.eps);
}

__global__ void __launch_bounds__(kThreads) adamw_kernel(const AdamLaunch a) {
  const int64_t chunk = blockIdx.x;
  const int ti = find_tensor(a.chunk_prefix, a.ntensors, chunk);
  if (!dev_check(ti >= 0 && ti < a.ntensors, a.status)) return;
  const AdamTensor t = a.tensors[ti];
  const int64_t begin = (chunk - a.chunk_prefix[ti]) * kAdamChunkElems;
  if (!dev_check(begin >= 0 && begin < t.numel, a.status)) return;
  const int64_t end = min(begin + static_cast<int64_t>(kAdamChunkElems), t.numel);
  const AdamScalars s{a.decay, a.step_size, a.inv_bc2, a.beta1, a.one_minus_beta1, a.beta2, a.one_minus_beta2, a.eps};
  int64_t scalar_from = begin;
  if (t.vec_ok) {
    const int64_t vend = begin + ((end - begin) / 8) * 8;
    for (int64_t e = begin + threadIdx.x * 8; e + 8 <= vend; e += kThreads * 8) {
      float g[8];
      if (a.gdtype == 1) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(t.g) + e));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          g[2 * k] = __uint_as_float(w[k] << 16);
          g[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
      } else {
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(t.g) + e));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(t.g) + e + 4));
        g[0] = g0.x, g[1] = g0.y, g[2] = g0.z, g[3] = g0.w, g[4] = g1.x, g[5] = g1.y, g[6] = g1.z, g[7] = g1.w;
      }
      float4 p4[2], m4[2], v4[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p4[h] = *reinterpret_cast<const float4*>(t.p + e + 4 * h);
        m4[h] = *reinterpret_cast<const float4*>(t.m + e + 4 * h);
        v4[h] = *reinterpret_cast<const float4*>(t.v + e + 4 * h);
      }
      float* pp = reinterpret_cast<float*>(p4);
      float* mm = reinterpret_cast<float*>(m4);
      float* vv = reinterpret_cast<float*>(v4);
#pragma unroll
      for (int k = 0; k < 8; ++k) adam_update(pp[k], mm[k], vv[k], g[k], s);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        *reinterpret_cast<float4*>(t.p + e + 4 * h) = p4[h];
        *reinterpret_cast<float4*>(t.m + e + 4 * h) = m4[h];
        *reinterpret_cast<float4*>(t.v + e + 4 * h) = v4[h];
      }
    }
    scalar_from = vend;
  }
  for (int64_t e = scalar_from + threadIdx.x; e < end; e += kThreads) {
    const float g = a.gdtype == 1 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(t.g)[e]) << 16)
                                  : static_cast<const float*>(t.g)[e];
    float p = t.p[e], m = t.m[e], v = t.v[e];
    adam_update(p, m, v, g, s);
    t.p[e] = p;
    t.m[e] = m;
    t.v[e] = v;
  }
}

}  // namespace

cudaError_t launch_adamw(const AdamLaunch& a, int64_t nchunks, cudaStream_t stream) {
  if (nchunks <= 0) return cudaSuccess;
  adamw_kernel<<<static_cast<unsigned>(nchunks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dmuon
