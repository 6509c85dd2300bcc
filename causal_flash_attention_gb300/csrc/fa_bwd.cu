// Backward pass of causal flash attention on sm_103a.
//
// Follows the recomputation scheme of "Phase T14: 融合 Flash-Attention
// Kernel", section 什么是 flash-attention (backward formulas) and its Key
// Design Decisions item 3: with D_i = <dO_i, O_i>,
//   p_ij = exp(s_ij - L_i), dp_ij = <dO_i, V_j>, ds_ij = p_ij (dp_ij - D_i),
//   dQ_i = scale sum_j ds_ij K_j, dK_j = scale sum_i ds_ij Q_i, dV_j = sum_i p_ij dO_i.
//
// Three kernels on one stream:
//   1. bwd_pre:    D_i, L_i * log2(e) (padded rows: D = 0, L = +inf), a zeroed
//                  fp32 dQ accumulator and a zeroed work-item counter.
//                  Bandwidth-bound.
//   2. bwd_main:   persistent, one CTA per SM. A work item is one (batch, key/value
//                  head, 128-row key tile j); CTAs claim items from the counter,
//                  lowest j (most work under the causal mask) first. K_j and
//                  V_j stay in shared memory, dK_j and dV_j stay in tensor memory
//                  for the whole item (so no atomics for them), and the CTA walks
//                  every query tile that can see a key of tile j (causal: rows
//                  at positions i + kv_offset >= the tile's first key, with
//                  kv_offset = Skv - Sq) of every query head of the group. An
//                  item's dK, dV write-out overlaps the next item's K, V loads
//                  and first products.
//                  Per step, on the tensor cores:
//                    S^T  = K_j Q_i^T          -> TMEM (kv rows x q cols)
//                    dP^T = V_j dO_i^T         -> TMEM
//                    [softmax warps: P^T = 2^(S^T*c - L*log2e), masked; written as
//                     16-bit into TMEM; dS^T = P^T (dP^T - D) written to smem]
//                    dV  += P^T dO_i           (P^T from TMEM)
//                    dK  += dS^T Q_i
//                    dQ   = dS K_j             -> TMEM, then added into the fp32
//                                                 dQ accumulator by bulk tensor
//                                                 reduce-adds of boxes staged in
//                                                 shared memory
//   3. dq_convert: dq = scale * accumulator, rounded to the input type.
//
// Warp roles of bwd_main (320 threads): warp 0 TMA producer (K_j, V_j once per item;
// Q_i with L_i, D_i through a 2-slot ring, dO_i through one slot at d = 128;
// three slots each at d = 64), warp 1 MMA issuer and TMEM
// owner, warps 2-9 compute P^T and dS^T (one thread per key row, two warps per
// TMEM lane quarter splitting the step's 128 query columns) and then move
// their half of dQ from TMEM into the global accumulator; at the end of an
// item warps 2-5 write dK and warps 6-9 write dV (bulk tensor stores staged
// in shared memory the warp owns).
//
// Tensor memory: dK [0,d), dV [128,128+d), S^T / P^T [256,384),
// dP^T / dQ [384,512). dQ reuses dP^T's columns once the softmax warps have
// read dP^T; S^T(i+1) is issued only after dV(i), which reads P^T(i), is done.
// At d = 64, P^T [64,128) and dQ [192,256) have columns of their own instead:
// S^T(i+1) is issued once the compute warps have read S^T(i), dP^T(i+1)
// right after dQ(i), and the warps read dQ(i) out after P^T(i+1).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 320;
constexpr float kLog2eF = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  // d = 64 leaves 128 of the 512 TMEM columns free: packed P^T (64-127) and
  // dQ (192-255) get their own instead of going over S^T and dP^T. S^T(n+1)
  // then waits only for S^T(n) to have been read (not for dV(n)), dP^T(n+1)
  // not for the dQ(n) read-out, and the compute warps read dQ(n) out after
  // P^T(n+1), by when the product has long completed
  static constexpr bool kSepQ = (D == 64);
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTileM * D * 2;        // one 128 x D tile
  // Q_i (with its L and D rows) is live from S^T(i), issued during the step
  // before, to dK(i): two or three slots. dO_i is live from dP^T(i) to dV(i),
  // which follow each other: d = 128 keeps one slot and spends the space on
  // the dQ staging of the bulk reductions.
  static constexpr int kQStages = (D == 128) ? 2 : 3;
  static constexpr int kDoStages = (D == 128) ? 1 : 3;
  static constexpr int kDsBytes = kTileN * kTileM * 2;     // dS^T, 128 x 128 16-bit
  static constexpr int kDqStageBytes = 32 * 32 * 4;        // per compute warp: 32 rows x 32 fp32
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // [kQStages]
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;     // [kDoStages]
  static constexpr int kOffDS = kOffDO + kDoStages * kTileBytes;
  static constexpr int kOffDqS = kOffDS + kDsBytes;                // [8 warps] (d = 128)
  static constexpr int kOffRow = kOffDqS + 8 * kDqStageBytes;     // [kQStages] x (L2 | D) x 128 f32
  static constexpr int kOffBar = kOffRow + kQStages * 1024;
  // kv_full, kv_empty, q_full[NQ], q_empty[NQ], do_full[ND], do_empty[ND], s_full,
  // dp_full, p_full, ds_full, dv_done, dq_full, dq_empty, ds_empty, kd_done, drain
  static constexpr int kNumBars = 2 + 2 * kQStages + 2 * kDoStages + 10 + (kSepQ ? 1 : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) {
      atomicOr(status, kStatusWaitTimeout);
      return;
    }
  }
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// ------------------------------------------------------------------ pre --
// Rows [0, BH * Sq_pad): D = <dO, O> in fp32, L * log2(e), and a zeroed dQ
// accumulator row. Bandwidth-bound, so every access is a 16-byte vector and
// the grid is one wave of warps striding over the rows: a row is U = d *
// sizeof(T) / 16 lanes (4 to 32), a warp takes 32 / U rows per pass.
template <typename T>
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b) {
  const T* x = reinterpret_cast<const T*>(&a);
  const T* y = reinterpret_cast<const T*>(&b);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < static_cast<int>(16 / sizeof(T)); ++e) s = fmaf(to_f(x[e]), to_f(y[e]), s);
  return s;
}

template <typename T>
__global__ void __launch_bounds__(256, 8) bwd_pre_kernel(const BwdPreParams p) {
  // the main kernel (launched as this grid's programmatic dependent) may be
  // scheduled now: its prologue overlaps this pass, and it waits for this
  // grid's completion before it reads anything this pass writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int U = p.d * static_cast<int>(sizeof(T)) / 16;   // power of two, divides 32
  const int rpw = 32 / U;
  const int sub = lane / U, u = lane % U;
  const long long total = static_cast<long long>(p.BH) * p.Sq_pad;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long row0 = warp0 * rpw; row0 < total; row0 += nwarps * rpw) {   // warp-uniform
    const long long row = row0 + sub;                                       // bh * Sq_pad + i
    const bool live = row < total;
    const int bh = live ? static_cast<int>(row / p.Sq_pad) : 0;
    const int i = live ? static_cast<int>(row % p.Sq_pad) : 0;
    float dsum = 0.f;
    if (live && i < p.Sq) {
      const size_t off = (static_cast<size_t>(bh) * p.Sq + i) * p.d * sizeof(T);
      const uint4 ov = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.out) + off)[u];
      const uint4 gv = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.dout) + off)[u];
      dsum = dot16<T>(ov, gv);
    }
    for (int sft = U / 2; sft > 0; sft >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, sft);
    if (live && u == 0) {
      p.delta[row] = (i < p.Sq) ? dsum : 0.f;
      p.lse2[row] = (i < p.Sq) ? p.lse[static_cast<size_t>(bh) * p.Sq + i] * kLog2eF : INFINITY;
    }
    if (p.dq_acc && live) {
      float4* acc = reinterpret_cast<float4*>(p.dq_acc + static_cast<size_t>(row) * p.d);
      for (int e = u; e < p.d / 4; e += U) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (p.work && blockIdx.x == 0 && threadIdx.x == 0) *p.work = 0;
}

// -------------------------------------------------------------- convert --
// dq = scale * dq_acc (rows < Sq), 8 elements per thread.
template <bool kBf16>
__global__ void __launch_bounds__(256, 8) dq_convert_kernel(const DqConvertParams p) {
  // launched as the main kernel's programmatic dependent: wait for that grid
  // (and the pre-pass before it) to complete and its writes to be visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long n8 = static_cast<long long>(p.BH) * p.Sq * p.d / 8;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long e = t * 8;
    const long long rowd = e / p.d;                      // bh * Sq + i
    const int col = static_cast<int>(e % p.d);
    const long long bh = rowd / p.Sq, i = rowd % p.Sq;
    const float4* src =
        reinterpret_cast<const float4*>(p.dq_acc + (bh * p.Sq_pad + i) * p.d + col);
    const float4 a = src[0], b = src[1];
    uint4 w;
    w.x = pack2<kBf16>(a.x * p.scale, a.y * p.scale);
    w.y = pack2<kBf16>(a.z * p.scale, a.w * p.scale);
    w.z = pack2<kBf16>(b.x * p.scale, b.y * p.scale);
    w.w = pack2<kBf16>(b.z * p.scale, b.w * p.scale);
    reinterpret_cast<uint4*>(p.dq)[t] = w;
  }
}

// ----------------------------------------------------------------- main --
// A work item is one key tile j of one (batch, key/value head): item
// w = j * B * Hkv + (b * Hkv + g), so that low j (most query tiles under the
// causal mask) comes first.
struct BwdItem {
  int j, bkv, b, g;
  int i_start, n_i, n_iter;
};

__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int w) {
  BwdItem it;
  const int BHkv = p.B * p.Hkv;
  it.j = w / BHkv;
  it.bkv = w % BHkv;
  it.b = it.bkv / p.Hkv;
  it.g = it.bkv % p.Hkv;
  // causal: the first query tile holding a row at position >= this tile's
  // first key (query row i stands at position i + kv_offset)
  it.i_start = p.causal ? max(0, it.j * kTileN - p.kv_offset) / kTileM : 0;
  it.n_i = p.n_q_tiles - it.i_start;
  it.n_iter = (p.Hq / p.Hkv) * it.n_i;
  return it;
}

template <int D, bool kBf16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int NQ = Cfg::kQStages;
  constexpr int ND = Cfg::kDoStages;
  // dQ = dS K_j lands in TMEM with lanes = query rows, so each compute thread
  // holds D/2 consecutive accumulator entries of one query row. Each warp
  // stages them as boxes of 32 rows x 32 fp32 (128-byte rows, 128-byte
  // swizzle: 16-byte stores, conflict-free) and one lane adds a box into the
  // accumulator with a bulk tensor reduce.
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {   // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadLaunch);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  // the work item whose K_j, V_j the current kv_full phase delivers
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  const uint32_t bar0 = sbase + Cfg::kOffBar;
  const uint32_t kv_full = bar0;
  const uint32_t kv_empty = bar0 + 8;
  auto q_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto q_empty = [&](int s) { return bar0 + 8 * (2 + NQ + s); };
  auto do_full = [&](int s) { return bar0 + 8 * (2 + 2 * NQ + s); };
  auto do_empty = [&](int s) { return bar0 + 8 * (2 + 2 * NQ + ND + s); };
  const uint32_t s_full = bar0 + 8 * (2 + 2 * NQ + 2 * ND);
  const uint32_t dp_full = s_full + 8;
  const uint32_t p_full = s_full + 16;
  const uint32_t ds_full = s_full + 24;
  const uint32_t dv_done = s_full + 32;
  const uint32_t dq_full = s_full + 40;
  const uint32_t dq_empty = s_full + 48;
  const uint32_t ds_empty = s_full + 56;
  const uint32_t kd_done = s_full + 64;
  const uint32_t drain = s_full + 72;
  const uint32_t s_free = s_full + 80;   // kSepQ: the compute warps have read S^T

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int n_items = p.n_kv_tiles * p.B * p.Hkv;
  if (threadIdx.x == 0) {
    trace_span(p.trace, 0, clock64());
    trace_span(p.trace, 1, smid());
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(q_full(s), 1);
      mbar_init(q_empty(s), 1 + 8);   // MMA commit + one per compute warp (L, D rows)
    }
    for (int s = 0; s < ND; ++s) {
      mbar_init(do_full(s), 1);
      mbar_init(do_empty(s), 1);      // MMA commit after dV
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 8);
    mbar_init(ds_full, 8);
    mbar_init(dv_done, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 8);
    mbar_init(ds_empty, 1);
    mbar_init(kd_done, 1);
    mbar_init(drain, 1);
    if (Cfg::kSepQ) mbar_init(s_free, 8);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as the pre-pass's programmatic dependent: everything above ran
  // alongside it; the D, L, zeroed dQ rows and the zeroed item counter it
  // writes are read below
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Steps (one query tile of one query head against the item's key tile) are
  // counted across the CTA's items, so every ring slot and barrier phase
  // below follows a global step count.
  if (warp == 0) {
    // ===================== TMA producer =====================
    // Claims items from the launch's counter. The next item's first Q and dO
    // go out as soon as their ring slots free, then its K_j, V_j once the
    // current item's last products have read K and V (kv_empty); the item
    // index is published with the kv_full arrival (an index past the last
    // item, with no bytes, ends the consumers' loops).
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_dk);
      tma_prefetch_desc(&p.tm_dv);
      Tracer tr(p.trace, 0);
      int nq = 0, ndo = 0;   // Q and dO tiles issued
      int kv_pending = -1;   // kv_full phase whose K, V loads may be in flight
      bool ok = true;
      // one step's Q (with its L, D rows) and dO
      auto load_step = [&](const BwdItem& I, int s) -> bool {
        const int bh = I.b * p.Hq + I.g * (p.Hq / p.Hkv) + s / I.n_i;
        const int i = I.i_start + s % I.n_i;
        const int sq = nq % NQ;
        if (nq >= NQ &&
            !mbar_wait(q_empty(sq), static_cast<uint32_t>(nq / NQ - 1) & 1, abort_flag, p.status))
          return false;
        tr(41);
        const uint32_t fq = q_full(sq);
        mbar_arrive_expect_tx(fq, Cfg::kTileBytes + 1024);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(sbase + Cfg::kOffQ + sq * Cfg::kTileBytes + c * (kTileM * 128), &p.tm_q, fq,
                      c * kChunk, i * kTileM, bh);
        const size_t roff = static_cast<size_t>(bh) * p.Sq_pad + static_cast<size_t>(i) * kTileM;
        bulk_load(sbase + Cfg::kOffRow + sq * 1024, p.lse2 + roff, 512, fq);
        bulk_load(sbase + Cfg::kOffRow + sq * 1024 + 512, p.delta + roff, 512, fq);
        ++nq;
        const int sd = ndo % ND;
        if (ndo >= ND &&
            !mbar_wait(do_empty(sd), static_cast<uint32_t>(ndo / ND - 1) & 1, abort_flag, p.status))
          return false;
        const uint32_t fd = do_full(sd);
        mbar_arrive_expect_tx(fd, Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(sbase + Cfg::kOffDO + sd * Cfg::kTileBytes + c * (kTileM * 128), &p.tm_do,
                      fd, c * kChunk, i * kTileM, bh);
        ++ndo;
        tr(40);
        return true;
      };
      int w = atomicAdd(p.work, 1);
      for (int k = 0; ok; ++k) {
        BwdItem I{};
        if (w < n_items) {
          I = bwd_item(p, w);
          if (!(ok = load_step(I, 0))) break;
        }
        if (k > 0) {
          if (!(ok = mbar_wait(kv_empty, (k - 1) & 1, abort_flag, p.status))) break;
          kv_pending = -1;
        }
        tr(95);
        *item_slot = w;
        if (w >= n_items) {
          mbar_arrive(kv_full);
          break;
        }
        mbar_arrive_expect_tx(kv_full, 2 * Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c) {
          tma_load_3d(sbase + Cfg::kOffK + c * (kTileN * 128), &p.tm_k, kv_full, c * kChunk,
                      I.j * kTileN, I.bkv);
          tma_load_3d(sbase + Cfg::kOffV + c * (kTileN * 128), &p.tm_v, kv_full, c * kChunk,
                      I.j * kTileN, I.bkv);
        }
        kv_pending = k;
        for (int s = 1; ok && s < I.n_iter; ++s) ok = load_step(I, s);
        if (!ok) break;
        w = atomicAdd(p.work, 1);
        if (w < n_items) {   // the next item's K_j, V_j into L2 while this item runs
          const BwdItem J = bwd_item(p, w);
          for (int c = 0; c < Cfg::kChunks; ++c) {
            tma_prefetch_l2_3d(&p.tm_k, c * kChunk, J.j * kTileN, J.bkv);
            tma_prefetch_l2_3d(&p.tm_v, c * kChunk, J.j * kTileN, J.bkv);
          }
        }
      }
      if (*abort_flag) {
        if (kv_pending >= 0) drain_wait(kv_full, static_cast<uint32_t>(kv_pending) & 1, p.status);
        for (int jj = max(0, nq - NQ); jj < nq; ++jj)
          drain_wait(q_full(jj % NQ), static_cast<uint32_t>(jj / NQ) & 1, p.status);
        for (int jj = max(0, ndo - ND); jj < ndo; ++jj)
          drain_wait(do_full(jj % ND), static_cast<uint32_t>(jj / ND) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    // Issue order per step n (dQ(n) first, so that its read-out and dP^T(n+1)
    // follow soon after dS(n); S^T(n+1) as soon as dV(n) has read P^T(n)):
    //   dV(n) [P(n) ready]  dQ(n) [dS(n) ready]  S^T(n+1) [dV(n) done]
    //   dK(n)  dP^T(n+1) [dQ(n) read out of TMEM]
    // d = 64 (own P^T and dQ columns):
    //   S^T(n+1) [S^T(n) read]  dV(n) [P(n) ready]
    //   dQ(n) [dS(n) ready, dQ(n-1) read out]  dP^T(n+1)  dK(n)
    // After an item's last step: kv_empty (K, V read for the last time by
    // that dQ), dK, kd_done; the next item's S^T and dP^T once its K, V land.
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, kTileM, kBf16, false, false);  // S^T, dP^T
      constexpr uint32_t idesc_kv = make_idesc(128, D, kBf16, false, true);       // dV, dK
      constexpr uint32_t idesc_q = make_idesc(128, D, kBf16, true, true);         // dQ
      const uint32_t t_dk = tmem, t_dv = tmem + 128, t_s = tmem + 256, t_dp = tmem + 384;
      const uint32_t t_dq = Cfg::kSepQ ? tmem + 192 : t_dp;
      const uint32_t t_p = Cfg::kSepQ ? tmem + 64 : t_s;   // packed P^T
      const uint32_t k_s = sbase + Cfg::kOffK, v_s = sbase + Cfg::kOffV;
      const uint32_t ds_s = sbase + Cfg::kOffDS;
      auto q_s = [&](int st) { return sbase + Cfg::kOffQ + st * Cfg::kTileBytes; };
      auto do_s = [&](int sd) { return sbase + Cfg::kOffDO + sd * Cfg::kTileBytes; };

      // Every operand descriptor is formed once; each product is issued from
      // one asm block with the K-step offsets as immediates (the issuing
      // thread would otherwise spend longer forming descriptors than the
      // tensor core spends on a step).
      const uint64_t k_desc = make_sdesc(k_s, 16, 1024);              // K_j, K-major (S^T)
      const uint64_t k_desc_mn = make_sdesc(k_s, kTileN * 128, 1024); // K_j, MN-major (dQ)
      const uint64_t v_desc = make_sdesc(v_s, 16, 1024);              // V_j, K-major (dP^T)
      const uint64_t ds_desc = make_sdesc(ds_s, 16, 1024);            // dS^T, K-major (dK)
      const uint64_t ds_desc_mn = make_sdesc(ds_s, kTileN * 128, 1024);   // dS, MN-major (dQ)
      // slot s of the Q and dO rings: the slot-0 descriptor plus s tiles
      // (the start-address field counts 16-byte units and cannot overflow
      // inside the 227 KB of shared memory)
      const uint64_t q_desc0 = make_sdesc(q_s(0), 16, 1024);
      const uint64_t q_desc0_mn = make_sdesc(q_s(0), kTileM * 128, 1024);
      const uint64_t do_desc0 = make_sdesc(do_s(0), 16, 1024);
      const uint64_t do_desc0_mn = make_sdesc(do_s(0), kTileM * 128, 1024);
      constexpr uint64_t kSlot = Cfg::kTileBytes >> 4;
      auto q_desc = [&](int s) { return q_desc0 + s * kSlot; };
      auto q_desc_mn = [&](int s) { return q_desc0_mn + s * kSlot; };
      auto do_desc = [&](int s) { return do_desc0 + s * kSlot; };
      auto do_desc_mn = [&](int s) { return do_desc0_mn + s * kSlot; };
      constexpr int kCB = kTileN * 128;   // bytes of one 64-column chunk of a 128-row tile

      Tracer tr(p.trace, 1);
      // S^T(g) = K_j Q_i^T once Q_i has landed and dV(g-1) has read P^T(g-1)
      auto issue_s = [&](int g) -> bool {
        if (!mbar_wait(q_full(g % NQ), static_cast<uint32_t>(g / NQ) & 1, abort_flag, p.status))
          return false;
        if (g > 0 && !mbar_wait(Cfg::kSepQ ? s_free : dv_done, (g - 1) & 1, abort_flag, p.status))
          return false;
        tr(5);
        tc_fence_after();
        mma_ss_product<D / 16, true, kCB, true, kCB>(t_s, k_desc, q_desc(g % NQ), idesc_s, 0);
        tc_commit(s_full);
        return true;
      };
      // dP^T(g) = V_j dO_i^T once dO_i has landed and dQ(g-1) has left TMEM
      auto issue_dp = [&](int g) -> bool {
        if (!Cfg::kSepQ && g > 0 && !mbar_wait(dq_empty, (g - 1) & 1, abort_flag, p.status))
          return false;
        if (!mbar_wait(do_full(g % ND), static_cast<uint32_t>(g / ND) & 1, abort_flag, p.status))
          return false;
        tr(7);
        tc_fence_after();
        mma_ss_product<D / 16, true, kCB, true, kCB>(t_dp, v_desc, do_desc(g % ND), idesc_s, 0);
        tc_commit(dp_full);
        return true;
      };

      bool ok = true;
      int g = 0;   // global step
      for (int k = 0; ok; ++k) {
        if (!(ok = mbar_wait(kv_full, k & 1, abort_flag, p.status))) break;
        tr(91);
        const int w = *item_slot;
        if (w >= n_items) break;
#ifdef FA_WAIT_TEST
        // wait-limit test build: nothing completes this phase before the abort
        // path's own commit, so the wait runs out
        if (k == 0 && !(ok = mbar_wait(drain, 0, abort_flag, p.status))) break;
#endif
        tr(9);
        const int N = bwd_item(p, w).n_iter;
        if (!(ok = issue_s(g) && issue_dp(g))) break;
        for (int n = 0; n < N; ++n, ++g) {
          const int st = g % NQ;
          const int sd = g % ND;
          const bool more = n + 1 < N;
          if constexpr (Cfg::kSepQ) {
            // S^T(n+1) as soon as the compute warps have read S^T(n)
            if (more && !(ok = issue_s(g + 1))) break;
            // dV += P^T dO_i (P^T packed in its own columns)
            if (!(ok = mbar_wait(p_full, g & 1, abort_flag, p.status))) break;
            tr(1);
            tc_fence_after();
            mma_ts_product8<false, 0>(t_dv, t_p, do_desc_mn(sd), idesc_kv, n > 0 ? 1u : 0u);
            tc_commit(dv_done);
            tc_commit(do_empty(sd));
            // dS^T(n) written (so dP^T(n) has been read) and dQ(n-1) read out:
            // dQ(n), dP^T(n+1), dK(n)
            if (!(ok = mbar_wait(ds_full, g & 1, abort_flag, p.status))) break;
            tr(3);
            if (g > 0 && !(ok = mbar_wait(dq_empty, (g - 1) & 1, abort_flag, p.status))) break;
            tc_fence_after();
            mma_ss_product<kTileN / 16, false, 0, false, 0>(t_dq, ds_desc_mn, k_desc_mn, idesc_q, 0);
            tc_commit(dq_full);
            if (!more) tc_commit(kv_empty);
            if (more && !(ok = issue_dp(g + 1))) break;
            mma_ss_product<kTileM / 16, true, kCB, false, 0>(t_dk, ds_desc, q_desc_mn(st), idesc_kv,
                                                            n > 0 ? 1u : 0u);
            tc_commit(ds_empty);
            tc_commit(q_empty(st));
            tr(6);
            continue;
          }
          // dV += P^T dO_i  (P^T from TMEM, 16-bit packed: query columns 0-63 in
          // S^T's columns 0-31, columns 64-127 in S^T's columns 96-127)
          if (!(ok = mbar_wait(p_full, g & 1, abort_flag, p.status))) break;
          tr(1);
          tc_fence_after();
          mma_ts_product8<false, 0, 64>(t_dv, t_s, do_desc_mn(sd), idesc_kv, n > 0 ? 1u : 0u);
          tc_commit(dv_done);
          tc_commit(do_empty(sd));
          // dQ (into dP^T's columns: the compute warps have read dP^T(n))
          if (!(ok = mbar_wait(ds_full, g & 1, abort_flag, p.status))) break;
          tr(3);
          tc_fence_after();
          // dQ = dS K_j, both operands MN-major
          mma_ss_product<kTileN / 16, false, 0, false, 0>(t_dq, ds_desc_mn, k_desc_mn, idesc_q, 0);
          tc_commit(dq_full);
          // S^T for the next step of this item; after its last step K and V
          // are free for the next item's
          if (more) {
            if (!(ok = issue_s(g + 1))) break;
          } else {
            tc_commit(kv_empty);
          }
          // dK += dS^T Q_i; then dS^T and stage st (Q_i, dO_i) are free
          mma_ss_product<kTileM / 16, true, kCB, false, 0>(t_dk, ds_desc, q_desc_mn(st), idesc_kv,
                                                          n > 0 ? 1u : 0u);
          tc_commit(ds_empty);
          tc_commit(q_empty(st));
          tr(6);
          // dP^T for the next step, once dQ(n) has left TMEM
          if (more && !(ok = issue_dp(g + 1))) break;
        }
        if (!ok) break;
        tc_commit(kd_done);   // dK, dV of this item are complete in TMEM
        tr(90);
      }
      trace_span(p.trace, 5, clock64());
      if (!ok) {
        tc_commit(drain);
        drain_wait(drain, 0, p.status);
      }
    }
  } else {
    // ============ P^T, dS^T and the dQ read-out (warps 2-9) ============
    // Two warps per TMEM lane quarter, one thread per key row: warps 2-5 take
    // query columns 0-63 of the step (half 0), warps 6-9 columns 64-127
    // (half 1). Each warp writes its packed P^T over score columns it has
    // read itself (half 0: columns 0-31, half 1: 96-127), so the two warps of
    // a quarter never wait for each other; at d = 64 into the P^T buffer's
    // columns [32 half, 32 half + 32) once dV has read the previous P^T.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int c0 = half * 64;                   // first query column of this warp
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + 256;
    const uint32_t t_dp = tmem + lane_off + 384;
    const uint32_t t_dq = Cfg::kSepQ ? tmem + lane_off + 192 : t_dp;
    const uint32_t t_p = Cfg::kSepQ ? tmem + lane_off + 64 : t_s;
    const float c = p.scale_log2;
    // dS^T row r of 64-column chunk `half` of the 128-byte-swizzled tile
    uint8_t* ds_row = smem + Cfg::kOffDS + half * (kTileN * 128) + r * 128;
    Tracer tr((warp == 2 && lane == 0) ? p.trace : nullptr, 2);
    bool ok = true;
    // This warp's dQ staging box (its 32 query rows x 32 fp32). d = 64: the
    // step's 32 columns are one box, staged right after the read-out.
    // d = 128: the step's 64 columns go out as two boxes: the first right after the
    // read-out, the second (held in registers meanwhile) after the next
    // step's dS^T, while the warps would otherwise wait for dQ; by then the
    // first box has long been read, and neither P^T -> dS^T nor the MMA
    // chain waits on the reduce's progress.
    const uint32_t dq_stage = sbase + Cfg::kOffDqS + (warp - 2) * Cfg::kDqStageBytes;
    // row `lane` with the swizzle's row term folded in: unit u is at row_sw ^ (u << 4)
    const uint32_t row_sw = dq_stage + lane * 128 + ((lane & 7) << 4);
    uint32_t dq_pend[32];
    int pend_x = -1, pend_y = 0, pend_bh = 0;
    // stage this lane's 32 values as row `lane` of the box (16-byte unit u at
    // u ^ (lane % 8): the map's 128-byte swizzle), hand the box to the async
    // proxy and let one lane issue the reduce-add
    auto reduce_box = [&](const uint32_t* v, int x, int y, int bh) {
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(row_sw ^ (u << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&p.tm_dq, dq_stage, x, y, bh);
        bulk_commit_group();
      }
    };
    // dQ of step gg (query tile ii, head bhh): TMEM -> fp32 accumulator. This
    // thread holds head-dimension entries [half * D/2, (half + 1) * D/2) of
    // query row r of the tile.
    auto read_dq = [&](int gg, int ii, int bhh) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full, gg & 1, abort_flag, p.status))) return false;
      tr(30);
      tc_fence_after();
      constexpr int kCols = D / 2;
      uint32_t acc[kCols];
#pragma unroll
      for (int cc = 0; cc < kCols / 32; ++cc)
        tmem_ld32(t_dq + half * kCols + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(acc + cc * 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_empty);
      tr(31);
      if constexpr (D == 128) {
        reduce_box(acc, half * 64, ii * kTileM + quarter * 32, bhh);
#pragma unroll
        for (int q = 0; q < 32; ++q) dq_pend[q] = acc[32 + q];
        pend_x = half * 64 + 32;
        pend_y = ii * kTileM + quarter * 32;
        pend_bh = bhh;
      } else {   // d = 64: the step's 32 columns are one box
        reduce_box(acc, half * 32, ii * kTileM + quarter * 32, bhh);
      }
      tr(32);
      return true;
    };
    int prev_i = 0, prev_bh = 0;   // kSepQ: the step whose dQ is still to be read out
    int g = 0;   // global step
    for (int k = 0; ok; ++k) {
      ok = __all_sync(0xffffffffu, mbar_wait(kv_full, k & 1, abort_flag, p.status));
      if (!ok) break;
      const int w = *item_slot;
      if (w >= n_items) break;
      const BwdItem I = bwd_item(p, w);
      const int kv = I.j * kTileN + r;
      for (int it = 0; it < I.n_iter; ++it, ++g) {
        const int st = g % NQ;
        const uint32_t par = static_cast<uint32_t>(g / NQ) & 1;
        const int i = I.i_start + it % I.n_i;
        const float* rowv = reinterpret_cast<const float*>(smem + Cfg::kOffRow + st * 1024);
        const float* l2s = rowv + c0;          // L * log2(e) per query column
        const float* dls = rowv + 128 + c0;    // D per query column
        ok = __all_sync(0xffffffffu, mbar_wait(q_full(st), par, abort_flag, p.status));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, abort_flag, p.status));
        if (!ok) break;
        tr(20);
        if (g == 0 && warp == 2 && lane == 0) trace_span(p.trace, 3, clock64());
        tc_fence_after();
        // Masked entries: key past the sequence end, or (causal) key after the
        // query's position q + kv_offset. Column e of this warp's half is masked
        // iff e < thr; thr <= 0 on every tile that is neither diagonal nor
        // ragged, which skip the selects.
        const int q0 = i * kTileM + c0;
        const int thr = kv >= p.Skv ? 64 : (p.causal ? min(kv - p.kv_offset - q0, 64) : 0);
        const bool any_mask = __any_sync(0xffffffffu, thr > 0);
        uint32_t ppk[32];
        {
          uint32_t raw[64];
          tmem_ld32(t_s + c0, *reinterpret_cast<uint32_t(*)[32]>(raw));
          tmem_ld32(t_s + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
          tmem_wait_ld();
          if constexpr (Cfg::kSepQ) {   // S^T(n+1) may overwrite these scores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
          }
          if (any_mask) {
#pragma unroll
            for (int e = 0; e < 64; ++e) raw[e] = (e < thr) ? __float_as_uint(-INFINITY) : raw[e];
          }
          const uint64_t c2 = f2_pack(c, c);
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float2 l2 = *reinterpret_cast<const float2*>(l2s + e);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[e]), __uint_as_float(raw[e + 1])), c2,
                             f2_pack(-l2.x, -l2.y)), x0, x1);
            ppk[e / 2] = pack2<kBf16>(ex2(x0), ex2(x1));
          }
          if constexpr (Cfg::kSepQ) {
            // dV(n-1) has read the previous P^T: columns [32 half, 32 half + 32)
            // of the P^T buffer take this warp's 64 query columns
            if (g > 0) ok = __all_sync(0xffffffffu, mbar_wait(dv_done, (g - 1) & 1, abort_flag, p.status));
            tc_fence_after();
            tmem_st32(t_p + half * 32, ppk);
          } else {
            tmem_st32(t_s + half * 96, ppk);
          }
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        tr(21);
        if (Cfg::kSepQ && it > 0 && !(ok = read_dq(g - 1, prev_i, prev_bh))) break;

        if (g > 0) ok = __all_sync(0xffffffffu, mbar_wait(ds_empty, (g - 1) & 1, abort_flag, p.status));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(dp_full, g & 1, abort_flag, p.status));
        if (!ok) break;
        tr(22);
        tc_fence_after();
        {
          uint32_t raw[64];
          tmem_ld32(t_dp + c0, *reinterpret_cast<uint32_t(*)[32]>(raw));
          tmem_ld32(t_dp + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
          tmem_wait_ld();
          uint32_t wv[32];
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float2 pp = unpack2<kBf16>(ppk[e / 2]);
            const float2 dd = *reinterpret_cast<const float2*>(dls + e);
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(pp.x, pp.y),
                             f2_sub(f2_pack(__uint_as_float(raw[e]), __uint_as_float(raw[e + 1])),
                                    f2_pack(dd.x, dd.y))), d0, d1);
            wv[e / 2] = pack2<kBf16>(d0, d1);
          }
          // the previous item's dK or dV store reads these rows (below)
          if (it == 0) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          // this warp's 64 query columns = one 128-byte row of chunk `half`;
          // 16-byte unit u of row r sits at unit u ^ (r % 8) (128-byte swizzle)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(ds_row + ((u ^ (r & 7)) << 4)) =
                make_uint4(wv[4 * u], wv[4 * u + 1], wv[4 * u + 2], wv[4 * u + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(ds_full);
          mbar_arrive(q_empty(st));
        }
        tr(23);
        if constexpr (D == 128) {
          if (pend_x >= 0) reduce_box(dq_pend, pend_x, pend_y, pend_bh);
          pend_x = -1;
          tr(34);
        }

        const int bh = I.b * p.Hq + I.g * (p.Hq / p.Hkv) + it / I.n_i;
        if (!Cfg::kSepQ || it + 1 == I.n_iter) {   // else after the next step's P^T
          if (!(ok = read_dq(g, i, bh))) break;
        }
        prev_i = i;
        prev_bh = bh;
      }
      if (!ok) break;
      if (pend_x >= 0) reduce_box(dq_pend, pend_x, pend_y, pend_bh);
      pend_x = -1;
      // ---- epilogue: warps 2-5 write dK = scale * accumulated dS^T Q, warps 6-9 dV ----
      // (the next item's first dV and dK, which overwrite these columns, wait
      // for this CTA's compute warps' P^T arrivals, which follow this read-out)
      // This warp's 32 key rows go out as 128-byte-swizzled boxes of 32 rows x
      // 64 columns through bulk tensor stores (rows past Skv are not written):
      // columns 0-63 staged over its own dS^T rows (free: every product of the
      // item is complete), columns 64-127 (d = 128) in its dQ staging box.
      ok = __all_sync(0xffffffffu, mbar_wait(kd_done, k & 1, abort_flag, p.status));
      if (!ok) break;
      tr(93);
      tc_fence_after();
      {
        const float f = half == 0 ? p.scale : 1.f;
        const uint32_t box0 = sbase + Cfg::kOffDS + half * (kTileN * 128) + quarter * 32 * 128;
        if (lane == 0) bulk_wait_read_all();   // the dQ box's last reduce has read it
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + half * 128 + cc * 32, o);
          tmem_wait_ld();
          const uint32_t row = (cc < 2 ? box0 : dq_stage) + lane * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t u = static_cast<uint32_t>((cc & 1) * 4 + v);   // 16-byte unit of the row
            st_shared_v4(row + ((u ^ (lane & 7)) << 4),
                         pack2<kBf16>(__uint_as_float(o[8 * v]) * f, __uint_as_float(o[8 * v + 1]) * f),
                         pack2<kBf16>(__uint_as_float(o[8 * v + 2]) * f, __uint_as_float(o[8 * v + 3]) * f),
                         pack2<kBf16>(__uint_as_float(o[8 * v + 4]) * f, __uint_as_float(o[8 * v + 5]) * f),
                         pack2<kBf16>(__uint_as_float(o[8 * v + 6]) * f, __uint_as_float(o[8 * v + 7]) * f));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int y = I.j * kTileN + quarter * 32;
        if (lane == 0 && y < p.Skv) {
          const CUtensorMap* tm = half == 0 ? &p.tm_dk : &p.tm_dv;
          tma_store_3d(tm, box0, 0, y, I.bkv);
          if constexpr (D == 128) tma_store_3d(tm, dq_stage, kChunk, y, I.bkv);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      tr(94);
    }
    // the bulk reduces read this warp's staging box until they complete
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (warp == 2 && lane == 0) trace_span(p.trace, 4, clock64());
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_span(p.trace, 6, clock64());
  // the dQ convert kernel (this grid's programmatic dependent) may be
  // scheduled once every CTA got here; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Launch as the programmatic dependent of the kernel before it on the stream:
// the new grid may start before that one completes and synchronizes with it
// through griddepcontrol.wait.
template <typename... Args>
cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D, bool kBf16>
cudaError_t launch_bwd_impl(const BwdParams& p, cudaStream_t stream) {
  constexpr int smem = BwdCfg<D>::kSmemBytes;
  auto kernel = fa_bwd_kernel<D, kBf16>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (the shared and tensor memory of one CTA fill
  // an SM), fewer when there are fewer items
  int dev = 0, n_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long n_items = static_cast<long long>(p.n_kv_tiles) * p.B * p.Hkv;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(n_items, std::max(n_sm, 1)));
  e = launch_dependent(kernel, dim3(grid), dim3(kBwdThreads), smem, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
  // one wave of 8-warp blocks (8 per SM), fewer when the rows run out
  const long long rows = static_cast<long long>(p.BH) * p.Sq_pad;
  const int esize = p.dtype == 0 ? 4 : 2;
  const long long rows_per_block = 8LL * (32 / (p.d * esize / 16));
  const unsigned grid =
      static_cast<unsigned>(std::min<long long>((rows + rows_per_block - 1) / rows_per_block, 152LL * 8));
  if (p.dtype == 0) bwd_pre_kernel<float><<<grid, 256, 0, stream>>>(p);
  else if (p.dtype == 1) bwd_pre_kernel<__half><<<grid, 256, 0, stream>>>(p);
  else bwd_pre_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const BwdParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_bwd_impl<128, true>(p, stream) : launch_bwd_impl<128, false>(p, stream);
  return bf16 ? launch_bwd_impl<64, true>(p, stream) : launch_bwd_impl<64, false>(p, stream);
}

cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(p.BH) * p.Sq * p.d / 8;
  const unsigned grid = static_cast<unsigned>(std::min<long long>((n8 + 255) / 256, 152LL * 16));
  const cudaError_t e =
      p.dtype == 2 ? launch_dependent(dq_convert_kernel<true>, dim3(grid), dim3(256), 0, stream, p)
                   : launch_dependent(dq_convert_kernel<false>, dim3(grid), dim3(256), 0, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace fa
