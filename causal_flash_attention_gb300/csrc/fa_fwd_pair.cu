// Forward pass of causal flash attention on CTA pairs (tcgen05 cta_group::2),
// head dimension 128.
//
// Computes the same O = softmax(mask(Q K^T * scale)) V and LSE as fa_fwd.cu
// ("Phase T14: 融合 Flash-Attention Kernel", section 什么是 flash-attention;
// "Phase 14: Flash Attention 2 for SM120", sections FA2 算法, Causal Mask and
// GQA 支持), with the same online-softmax recurrence, lazy rescale and
// epilogue, but two CTAs on two SMs form one tensor-core unit: the 2-CTA mode
// that "Phase 14", section 硬件约束, lists for the SM100 generation.
//
// A pair owns four 128-row query tiles T0..T3 of one (batch, query head): a
// 512-row block. Slot 0 pairs T0 (leader) with T1 (peer), slot 1 T2 with T3.
// Per key/value tile j the leader's single issuing thread runs, per slot,
//   S = Q K_j^T   M = 256 (128 query rows per CTA), N = 128 keys, K = 128
//   O += P V_j    M = 256, N = 128 head columns, K = 128 keys (P from TMEM)
// Each CTA loads only half of every key/value tile: keys 64r..64r+63 of K_j
// (the N half of S that CTA r holds) and head columns 64r..64r+63 of V_j (its
// N half of O), so a key/value byte crosses into shared memory once per pair.
// Both CTAs of a slot walk the key tiles the later of their two tiles needs;
// the earlier tile's extra (diagonal) tile is masked out entirely by the
// causal mask, about 1/(2n) extra work for a slot of n key tiles.
//
// Warp roles (320 threads per CTA):
//   warp 0      TMA producer: this CTA's two query tiles once, then its halves
//               of K_j and V_j through 4-stage rings; completions land on its
//               own barriers.
//   warp 1      leader: the MMA issuer. Peer: relays each of its own load
//               completions to the matching leader barrier, in load order.
//   warps 2-5   softmax of slot 0 (this CTA's tile), warps 6-9 of slot 1: one
//               thread per query row, as in fa_fwd.cu; P goes back to this
//               CTA's tensor memory and each warp arrives on the leader's
//               "P ready" barrier (the peer's warps remotely).
// Tensor memory per CTA (512 columns, allocated jointly): S_0 [0,128),
// S_1 [128,256), O_0 [256,384), O_1 [384,512).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kPairThreads = 320;
constexpr float kLn2Pair = 0.6931471805599453f;
constexpr float kRescaleThresholdPair = 8.0f;   // as fa_fwd.cu: reference max moves by > 2^8

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kStages = 4;
  static constexpr int kQBytes = kTileM * D * 2;          // one 128-row query tile (2 chunks)
  static constexpr int kQChunk = kTileM * 128;            // 64 columns x 128 rows
  static constexpr int kKHalfBytes = 64 * D * 2;          // 64 keys x 128 columns (2 chunks)
  static constexpr int kKChunk = 64 * 128;                // 64 columns x 64 rows
  static constexpr int kVHalfBytes = kTileN * 64 * 2;     // 128 keys x 64 columns
  static constexpr int kOffQ = 0;                         // [2 slots]
  static constexpr int kOffK = 2 * kQBytes;               // [kStages]
  static constexpr int kOffV = kOffK + kStages * kKHalfBytes;
  static constexpr int kOffBar = kOffV + kStages * kVHalfBytes;
  // q_full, q_peer, k_full[S], k_peer[S], v_full[S], v_peer[S], k_empty[S],
  // v_empty[S], s_full[2], p_full[2], pv_done[2], drain
  static constexpr int kNumBars = 2 + 6 * kStages + 7;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
};

__device__ __forceinline__ void drain_wait_pair(uint32_t bar, uint32_t parity, int* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) {
      atomicOr(status, kStatusWaitTimeout);
      return;
    }
  }
}

template <bool kBf16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = PairCfg;
  constexpr int D = Cfg::D;
  constexpr int NS = Cfg::kStages;
  constexpr uint16_t kBoth = 3;   // multicast mask: both CTAs of the pair
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs: the pair's descriptors address both
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  const uint32_t rank = cluster_ctarank();   // 0: leader
  const bool leader = rank == 0;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  const uint32_t q_full = bar0, q_peer = bar0 + 8;
  auto k_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_peer = [&](int s) { return bar0 + 8 * (2 + NS + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + 2 * NS + s); };
  auto v_peer = [&](int s) { return bar0 + 8 * (2 + 3 * NS + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (2 + 4 * NS + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (2 + 5 * NS + s); };
  auto s_full = [&](int t) { return bar0 + 8 * (2 + 6 * NS + t); };
  auto p_full = [&](int t) { return bar0 + 8 * (4 + 6 * NS + t); };
  auto pv_done = [&](int t) { return bar0 + 8 * (6 + 6 * NS + t); };
  const uint32_t drain = bar0 + 8 * (8 + 6 * NS);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());

  // ---- work: a 512-row query block of one (batch, query head), heaviest first ----
  const int BHq = p.B * p.Hq;
  const int item = static_cast<int>(blockIdx.x) >> 1;
  const int blk = p.n_qblocks - 1 - item / BHq;
  const int bh = item % BHq;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int n_kv_total = (p.Skv + kTileN - 1) / kTileN;
  auto extent = [&](int qt) {   // key tiles query tile qt walks (0 past the sequence end)
    if (qt * kTileM >= p.Sq) return 0;
    return p.causal ? min(qt + p.kv_tiles_ahead, n_kv_total) : n_kv_total;
  };
  int n_s[2], own_qt[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    own_qt[s] = 4 * blk + 2 * s + static_cast<int>(rank);
    n_s[s] = max(extent(4 * blk + 2 * s), extent(4 * blk + 2 * s + 1));
  }
  const int n_load = max(n_s[0], n_s[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_peer, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_peer(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_peer(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 8);   // four softmax warps in each CTA
      mbar_init(pv_done(t), 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ===================== TMA producer (both CTAs) =====================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k_half);
      tma_prefetch_desc(&p.tm_v);
      const uint32_t q_bytes = (n_s[0] > 0 ? Cfg::kQBytes : 0) + (n_s[1] > 0 ? Cfg::kQBytes : 0);
      if (q_bytes) {
        mbar_arrive_expect_tx(q_full, q_bytes);
        for (int s = 0; s < 2; ++s) {
          if (n_s[s] == 0) continue;
          for (int c = 0; c < 2; ++c)
            tma_load_3d(sbase + Cfg::kOffQ + s * Cfg::kQBytes + c * Cfg::kQChunk, &p.tm_q, q_full,
                        c * kChunk, own_qt[s] * kTileM, bh);
        }
      }
      int j = 0;
      for (; j < n_load; ++j) {
        const int st = j % NS;
        const uint32_t use = static_cast<uint32_t>(j / NS);
        if (j >= NS && !mbar_wait_cluster(k_empty(st), (use - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(k_full(st), Cfg::kKHalfBytes);
        for (int c = 0; c < 2; ++c)   // keys 64 rank .. 64 rank + 63 of tile j
          tma_load_3d(sbase + Cfg::kOffK + st * Cfg::kKHalfBytes + c * Cfg::kKChunk, &p.tm_k_half,
                      k_full(st), c * kChunk, j * kTileN + 64 * static_cast<int>(rank), bkv);
        if (j >= NS && !mbar_wait_cluster(v_empty(st), (use - 1) & 1, abort_flag, p.status)) {
          ++j;   // the K load of this iteration is in flight
          break;
        }
        mbar_arrive_expect_tx(v_full(st), Cfg::kVHalfBytes);
        // head columns 64 rank .. 64 rank + 63 of every key of tile j
        tma_load_3d(sbase + Cfg::kOffV + st * Cfg::kVHalfBytes, &p.tm_v, v_full(st),
                    64 * static_cast<int>(rank), j * kTileN, bkv);
      }
      // Before the CTA may leave: in a clean run every stage loaded has been
      // released by the leader's MMAs (so no multicast arrival is still on
      // its way here); otherwise this CTA's own copies are drained.
      bool clean = !*abort_flag;
      for (int jj = max(0, j - NS); clean && jj < j; ++jj) {
        const uint32_t par = static_cast<uint32_t>(jj / NS) & 1;
        clean = mbar_wait_cluster(k_empty(jj % NS), par, abort_flag, p.status) &&
                mbar_wait_cluster(v_empty(jj % NS), par, abort_flag, p.status);
      }
      if (!clean) {
        if (q_bytes) drain_wait_pair(q_full, 0, p.status);
        for (int jj = max(0, j - NS); jj < j; ++jj) {
          const uint32_t par = static_cast<uint32_t>(jj / NS) & 1;
          drain_wait_pair(k_full(jj % NS), par, p.status);
          drain_wait_pair(v_full(jj % NS), par, p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !leader) {
      // ============ peer: relay load completions to the leader ============
      bool ok = true;
      if (n_s[0] > 0 || n_s[1] > 0) {
        ok = mbar_wait(q_full, 0, abort_flag, p.status);
        if (ok) mbar_arrive_remote(map_to_rank(q_peer, 0));
      }
      for (int j = 0; ok && j < n_load; ++j) {
        const int st = j % NS;
        const uint32_t par = static_cast<uint32_t>(j / NS) & 1;
        if (!(ok = mbar_wait(k_full(st), par, abort_flag, p.status))) break;
        mbar_arrive_remote(map_to_rank(k_peer(st), 0));
        if (!(ok = mbar_wait(v_full(st), par, abort_flag, p.status))) break;
        mbar_arrive_remote(map_to_rank(v_peer(st), 0));
      }
    } else if (lane == 0) {
      // ===================== leader: MMA issuer =====================
      constexpr uint32_t idesc_qk = make_idesc(256, kTileN, kBf16, false, false);
      constexpr uint32_t idesc_pv = make_idesc(256, D, kBf16, false, true);
      const uint64_t q_desc0 = make_sdesc(sbase + Cfg::kOffQ, 16, 1024);
      const uint64_t k_desc0 = make_sdesc(sbase + Cfg::kOffK, 16, 1024);
      const uint64_t v_desc0 = make_sdesc(sbase + Cfg::kOffV, kTileN * 128, 1024);
      auto issue_qk = [&](int t, int st) {   // S_t = Q_t K^T over the pair
        mma_pair_ss_product8<true, Cfg::kQChunk, true, Cfg::kKChunk>(
            tmem + t * 128, q_desc0 + t * (Cfg::kQBytes >> 4), k_desc0 + st * (Cfg::kKHalfBytes >> 4),
            idesc_qk, 0);
        tc_commit_pair(s_full(t), kBoth);
      };
      auto issue_pv = [&](int t, int st, bool accumulate) {   // O_t (+)= P_t V over the pair
        mma_pair_ts_product8<false, 0>(tmem + 256 + t * 128, tmem + t * 128,
                                       v_desc0 + st * (Cfg::kVHalfBytes >> 4), idesc_pv,
                                       accumulate ? 1u : 0u);
        tc_commit_pair(pv_done(t), kBoth);
      };
      auto both = [&](uint32_t own, uint32_t peer, uint32_t par) {
        return mbar_wait(own, par, abort_flag, p.status) &&
               mbar_wait_cluster(peer, par, abort_flag, p.status);
      };

      Tracer tr(p.trace, 1);
      bool ok = both(q_full, q_peer, 0);
#ifdef FA_WAIT_TEST
      // wait-limit test build: nothing completes this phase before the abort
      // path's own commit, so the wait runs out
      if (ok) ok = mbar_wait(drain, 0, abort_flag, p.status);
#endif
      if (ok) ok = both(k_full(0), k_peer(0), 0);
      tr(9);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n_s[t] > 0) issue_qk(t, 0);
        tc_commit_pair(k_empty(0), kBoth);
      }
      for (int j = 0; ok && j < n_load; ++j) {
        const int st = j % NS;
        const uint32_t par = static_cast<uint32_t>(j / NS) & 1;
        if (!(ok = both(v_full(st), v_peer(st), par))) break;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= n_s[t]) continue;
          if (!(ok = mbar_wait_cluster(p_full(t), j & 1, abort_flag, p.status))) break;
          tr(50 + t);
          tc_fence_after();
          issue_pv(t, st, j > 0);
          if (j + 1 < n_s[t]) {
            const int st1 = (j + 1) % NS;
            const uint32_t par1 = static_cast<uint32_t>((j + 1) / NS) & 1;
            if (!(ok = both(k_full(st1), k_peer(st1), par1))) break;
            // P_t(j) lives in S_t's columns: wait until P_t(j) V_j has read it.
            if (!(ok = mbar_wait(pv_done(t), j & 1, abort_flag, p.status))) break;
            tr(54 + t);
            tc_fence_after();
            issue_qk(t, st1);
          }
        }
        if (!ok) break;
        tc_commit_pair(v_empty(st), kBoth);
        if (j + 1 < n_load) tc_commit_pair(k_empty((j + 1) % NS), kBoth);
      }
      if (!ok) {
        // every MMA issued so far must finish before either CTA frees its memory
        tc_commit_pair(drain, 1);
        drain_wait_pair(drain, 0, p.status);
      }
    }
  } else {
    // ===================== softmax / correction / epilogue =====================
    const int t = (warp - 2) / 4;               // slot of this warp group
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;          // row within this CTA's tile
    const int q0 = own_qt[t] * kTileM;
    const int row = q0 + r;
    const int n = n_s[t];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + t * 128;
    const uint32_t o_tmem = tmem + lane_off + 256 + t * 128;
    const uint32_t p_ready = leader ? p_full(t) : map_to_rank(p_full(t), 0);
    const float c = p.scale_log2;

    Tracer tr(((warp == 2 || warp == 6) && lane == 0 && leader) ? p.trace : nullptr, 2 + t);
    float m_ref = -INFINITY;   // reference max, scaled log2 domain
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(s_full(t), j & 1, abort_flag, p.status));
      if (!ok) break;
      tr(60);
      tc_fence_after();
      float s[kTileN];
      {
        uint32_t raw[kTileN];
#pragma unroll
        for (int cc = 0; cc < kTileN / 32; ++cc)
          tmem_ld32(s_tmem + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(raw + cc * 32));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kTileN; ++i) s[i] = __uint_as_float(raw[i]);
      }
      const int kv0 = j * kTileN;
      // inline mask (causal and keys past the end); on the pair's extra key
      // tile of the earlier query tile every key is masked and P = 0
      const int lim = p.causal ? row + p.kv_offset : p.Skv - 1;
      if (kv0 + kTileN - 1 > lim) {
#pragma unroll
        for (int i = 0; i < kTileN; ++i)
          if (kv0 + i > lim) s[i] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int i = 4; i < kTileN; i += 4) {
        mx0 = fmaxf(mx0, s[i]);
        mx1 = fmaxf(mx1, s[i + 1]);
        mx2 = fmaxf(mx2, s[i + 2]);
        mx3 = fmaxf(mx3, s[i + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      float m_new = m_ref;
      if (mx > m_ref + kRescaleThresholdPair) m_new = mx;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_ref - m_use);   // 0 when m_ref = -inf
      const bool moved = (m_new != m_ref);
      m_ref = m_new;

      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2(fmaf(s[h * 64 + 2 * i], c, -m_use));
          const float p1 = ex2(fmaf(s[h * 64 + 2 * i + 1], c, -m_use));
          sum[(2 * i) & 3] += p0;
          sum[(2 * i + 1) & 3] += p1;
          pk[i] = pack2<kBf16>(p0, p1);
        }
        tmem_st32(s_tmem + h * 32, pk);
      }
      l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));

      // O <- alpha * O for rows whose reference max moved (not needed for the
      // first tile: its P V overwrites O)
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_cluster(pv_done(t), (j - 1) & 1, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const float a = moved ? alpha : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_tmem + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
          tmem_st32(o_tmem + cc * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(p_ready);
        else mbar_arrive_remote(p_ready);
      }
      tr(61);
    }

    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(pv_done(t), (n - 1) & 1, abort_flag, p.status));
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        using Elem = typename std::conditional<kBf16, __nv_bfloat16, __half>::type;
        Elem* orow = reinterpret_cast<Elem*>(p.out) + (static_cast<size_t>(bh) * p.Sq + row) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_tmem + cc * 32, o);
          tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack2<kBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                __uint_as_float(o[2 * i + 1]) * inv_l);
          if (row < p.Sq) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
        if (row < p.Sq)
          p.lse[static_cast<size_t>(bh) * p.Sq + row] = (m_ref + __log2f(l)) * kLn2Pair;
      }
    }
  }

  // neither CTA leaves (or frees its tensor memory) while the other may still
  // read its shared or tensor memory or arrive on its barriers
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool kBf16>
cudaError_t launch_pair_impl(const FwdParams& p, cudaStream_t stream) {
  constexpr int smem = PairCfg::kSmemBytes;
  auto kernel = fa_fwd_pair_kernel<kBf16>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(2LL * p.B * p.Hq * p.n_qblocks);
  kernel<<<grid, kPairThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pair(const FwdParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? launch_pair_impl<true>(p, stream) : launch_pair_impl<false>(p, stream);
}

}  // namespace fa
