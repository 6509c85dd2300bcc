// fp32 attention on plain fp32 arithmetic (no tensor cores), for fp32 inputs.
//
// Forward: one warp per query row; keys are taken 32 at a time (one key per
// lane for the score, every lane for a slice of the accumulator) with the
// online-softmax update of "Phase T14: 融合 Flash-Attention Kernel", section
// 什么是 flash-attention (running max m, running sum l, rescaled
// accumulator, out = acc / l, L = m + log l).
//
// Backward: recomputes p_ij = exp(s_ij - L_i) and uses D_i = <dO_i, O_i>
// (precomputed) with ds_ij = p_ij (dp_ij - D_i) (same page, backward
// formulas). dQ is gathered per query row and dK/dV per key row (summed over
// the key/value head's query-head group), so no atomics are needed.
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxPer = 4;   // d / 32 <= 4

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float dot_row(const float* a, const float* b, int d) {
  float acc = 0.f;
  for (int e = 0; e < d; ++e) acc = fmaf(a[e], b[e], acc);
  return acc;
}

__global__ void __launch_bounds__(kWarps * 32) fwd_simt(const SimtParams p) {
  __shared__ float qs[kWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  const int d = p.d, per = d / 32;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const float* qrow = p.q + (static_cast<size_t>(bh) * p.Sq + (i < p.Sq ? i : 0)) * d;
  for (int e = lane; e < d; e += 32) qs[warp][e] = qrow[e];
  __syncwarp();
  if (i >= p.Sq) return;
  const float* kh = p.k + static_cast<size_t>(b * p.Hkv + g) * p.Skv * d;
  const float* vh = p.v + static_cast<size_t>(b * p.Hkv + g) * p.Skv * d;
  const int n = p.causal ? i + 1 + p.kv_offset : p.Skv;   // visible keys
  float m = -INFINITY, l = 0.f, acc[kMaxPer] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const float s = j < n ? p.scale * dot_row(qs[warp], kh + static_cast<size_t>(j) * d, d) : -INFINITY;
    const float m_new = fmaxf(m, warp_max(s));
    const float alpha = expf(m - m_new);
    const float pj = j < n ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
    for (int u = 0; u < per; ++u) acc[u] *= alpha;
    const int cnt = min(32, n - j0);
    for (int t = 0; t < cnt; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pj, t);
      const float* vr = vh + static_cast<size_t>(j0 + t) * d;
      for (int u = 0; u < per; ++u) acc[u] = fmaf(pt, vr[lane + 32 * u], acc[u]);
    }
    m = m_new;
  }
  float* orow = p.o_out + (static_cast<size_t>(bh) * p.Sq + i) * d;
  for (int u = 0; u < per; ++u) orow[lane + 32 * u] = acc[u] / l;
  if (lane == 0) p.lse_out[static_cast<size_t>(bh) * p.Sq + i] = m + logf(l);
}

// dQ_i = scale * sum_j p_ij (dp_ij - D_i) K_j, one warp per query row.
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_simt(const SimtParams p, int Sq_pad) {
  __shared__ float qs[kWarps][128], dos[kWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  const int d = p.d, per = d / 32;
  const int ii = i < p.Sq ? i : 0;
  const size_t rowoff = (static_cast<size_t>(bh) * p.Sq + ii) * d;
  for (int e = lane; e < d; e += 32) {
    qs[warp][e] = p.q[rowoff + e];
    dos[warp][e] = p.dout[rowoff + e];
  }
  __syncwarp();
  if (i >= p.Sq) return;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const float* kh = p.k + static_cast<size_t>(b * p.Hkv + g) * p.Skv * d;
  const float* vh = p.v + static_cast<size_t>(b * p.Hkv + g) * p.Skv * d;
  const float L = p.lse[static_cast<size_t>(bh) * p.Sq + i];
  const float Di = p.delta[static_cast<size_t>(bh) * Sq_pad + i];
  const int n = p.causal ? i + 1 + p.kv_offset : p.Skv;
  float acc[kMaxPer] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    float ds = 0.f;
    if (j < n) {
      const float s = p.scale * dot_row(qs[warp], kh + static_cast<size_t>(j) * d, d);
      const float pj = expf(s - L);
      const float dp = dot_row(dos[warp], vh + static_cast<size_t>(j) * d, d);
      ds = pj * (dp - Di);
    }
    const int cnt = min(32, n - j0);
    for (int t = 0; t < cnt; ++t) {
      const float dst = __shfl_sync(0xffffffffu, ds, t);
      const float* kr = kh + static_cast<size_t>(j0 + t) * d;
      for (int u = 0; u < per; ++u) acc[u] = fmaf(dst, kr[lane + 32 * u], acc[u]);
    }
  }
  float* out = p.dq + (static_cast<size_t>(bh) * p.Sq + i) * d;
  for (int u = 0; u < per; ++u) out[lane + 32 * u] = p.scale * acc[u];
}

// dK_j = scale * sum_{h in group, i} ds_ij Q_i and dV_j = sum p_ij dO_i, one
// warp per key row.
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_simt(const SimtParams p, int Sq_pad) {
  __shared__ float ks[kWarps][128], vs[kWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bkv = blockIdx.y;   // b * Hkv + g
  const int j = blockIdx.x * kWarps + warp;
  const int d = p.d, per = d / 32;
  const int jj = j < p.Skv ? j : 0;
  const size_t rowoff = (static_cast<size_t>(bkv) * p.Skv + jj) * d;
  for (int e = lane; e < d; e += 32) {
    ks[warp][e] = p.k[rowoff + e];
    vs[warp][e] = p.v[rowoff + e];
  }
  __syncwarp();
  if (j >= p.Skv) return;
  const int b = bkv / p.Hkv, g = bkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  float dk[kMaxPer] = {0.f, 0.f, 0.f, 0.f}, dv[kMaxPer] = {0.f, 0.f, 0.f, 0.f};
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const int bh = b * p.Hq + h;
    const float* qh = p.q + static_cast<size_t>(bh) * p.Sq * d;
    const float* doh = p.dout + static_cast<size_t>(bh) * p.Sq * d;
    // causal: query rows at positions i + kv_offset >= j see key j
    const int i_start = p.causal ? max(0, j - p.kv_offset) : 0;
    for (int i0 = i_start; i0 < p.Sq; i0 += 32) {
      const int i = i0 + lane;
      float pij = 0.f, ds = 0.f;
      if (i < p.Sq) {
        const float s = p.scale * dot_row(qh + static_cast<size_t>(i) * d, ks[warp], d);
        pij = expf(s - p.lse[static_cast<size_t>(bh) * p.Sq + i]);
        const float dp = dot_row(doh + static_cast<size_t>(i) * d, vs[warp], d);
        ds = pij * (dp - p.delta[static_cast<size_t>(bh) * Sq_pad + i]);
      }
      const int cnt = min(32, p.Sq - i0);
      for (int t = 0; t < cnt; ++t) {
        const float pt = __shfl_sync(0xffffffffu, pij, t);
        const float dt = __shfl_sync(0xffffffffu, ds, t);
        const float* qr = qh + static_cast<size_t>(i0 + t) * d;
        const float* dr = doh + static_cast<size_t>(i0 + t) * d;
        for (int u = 0; u < per; ++u) {
          dv[u] = fmaf(pt, dr[lane + 32 * u], dv[u]);
          dk[u] = fmaf(dt, qr[lane + 32 * u], dk[u]);
        }
      }
    }
  }
  float* dko = p.dk + rowoff;
  float* dvo = p.dv + rowoff;
  for (int u = 0; u < per; ++u) {
    dko[lane + 32 * u] = p.scale * dk[u];
    dvo[lane + 32 * u] = dv[u];
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const SimtParams& p, cudaStream_t stream) {
  dim3 grid((p.Sq + kWarps - 1) / kWarps, p.B * p.Hq);
  fwd_simt<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const SimtParams& p, cudaStream_t stream) {
  const int Sq_pad = (p.Sq + kTileM - 1) / kTileM * kTileM;
  dim3 g1((p.Sq + kWarps - 1) / kWarps, p.B * p.Hq);
  bwd_dq_simt<<<g1, kWarps * 32, 0, stream>>>(p, Sq_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((p.Skv + kWarps - 1) / kWarps, p.B * p.Hkv);
  bwd_dkdv_simt<<<g2, kWarps * 32, 0, stream>>>(p, Sq_pad);
  return cudaGetLastError();
}

}  // namespace fa
