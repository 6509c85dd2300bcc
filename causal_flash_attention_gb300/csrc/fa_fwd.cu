// Forward pass of causal scaled-dot-product flash attention on sm_103a.
//
// Computes, per (batch, query head), O = softmax(mask(Q K^T * scale)) V and the
// natural-log logsumexp LSE_i of each scaled score row, without forming the
// S x S score matrix ("Phase T14: 融合 Flash-Attention Kernel", section
// 什么是 flash-attention; "Phase 14: Flash Attention 2 for SM120", section
// FA2 算法). The online-softmax recurrence keeps a running max m, a running
// sum l and an accumulator O per query row, rescaling O and l by exp(m_old -
// m_new) when the max grows; out = O / l and LSE = m + log l at the end.
//
// A CTA owns T = 1 or 2 consecutive 128-row query tiles of one (batch, query
// head) and walks the key/value tiles up to the causal diagonal (tiles wholly
// above it are never loaded; "Phase 14", section Causal Mask, tile-level
// skip). With Sq queries against Skv >= Sq keys, query row i stands at
// position i + (Skv - Sq), the kv_offset of the same section. Key/value head
// = query head / (Hq / Hkv) ("Phase 14", section GQA 支持).
//
// Warp roles (64 + 128 T threads):
//   warp 0      TMA producer: Q tiles once, then K and V tiles into
//               multi-stage rings (mbarrier full/empty handshakes).
//   warp 1      tcgen05 MMA issuer (one thread) and TMEM owner:
//               S_t = Q_t K_j^T (both operands from shared memory) and
//               O_t += P_t V_j (P_t from tensor memory, V_j from shared memory).
//   warps 2-5   softmax for query tile 0 (T = 2: warps 6-9 for query tile 1):
//               one thread per query row reads its score row from TMEM,
//               applies the causal mask inline, does the online-softmax update
//               with ex2, writes P (bf16/fp16) back to TMEM over its own
//               scores, rescales O in TMEM when the row max grew by more than
//               2^8, and finally writes out = O / l and LSE.
//
// Tensor memory (256 T columns): S_t [128 t, 128 t + 128), O_t [128 T + 128 t,
// ... + d). P_t is packed two 16-bit values per column into the first 64
// columns of S_t, so the next S_t = Q_t K^T may only be issued after the
// P_t V MMA that reads it has completed (tcgen05 MMAs with different
// accumulators are not ordered); the issuer waits for that completion.
// Except at d = 64 with T = 1, where P has its own 64 columns after O (256
// columns in all): there the softmax warps release S as soon as they have
// read it, the issuer starts the next S = Q K^T at once, and the warps wait
// for the previous P V only before writing the new P.
//
// T = 2: the two softmax groups ping-pong inside the CTA: while one works on
// its score tile, the tensor core runs the other tile's P V and Q K^T.
// T = 1: the CTA is small enough (half the tensor memory, one-stage (d = 128)
// or two-stage (d = 64) K and V rings) for two to share an SM, and the two
// CTAs overlap each other's softmax, loads, start-up and write-out the same
// way; the launcher takes it for grids of at least four one-tile CTAs per SM,
// and for every grid at d = 64.
#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
// A row's reference max only moves when the running max exceeds it by more
// than this many powers of two; until then p = 2^(x - m_ref) <= 2^8, which
// fp32 accumulation and 16-bit P both hold without loss of range.
constexpr float kRescaleThreshold = 8.0f;

template <int D, int T>
struct FwdCfg {
  static constexpr int kTiles = T;                          // query tiles per CTA
  static constexpr int kThreads = 64 + 128 * T;
  static constexpr int kTmemCols = 256 * T;
  // d = 64, one tile: P gets its own 64 columns after O (free at that d),
  // so the next S = Q K^T may be issued as soon as S has been read out of
  // TMEM, and runs during the softmax and P V of the current tile
  static constexpr bool kSepP = (D == 64 && T == 1);
  // same form: the softmax in paired fp32 instructions and 3-input max (the
  // registers allow it there; the results are bit-identical to the scalar form)
  static constexpr bool kPaired = kSepP;
  static constexpr int kChunks = D / kChunk;                // 64-col chunks per row
  static constexpr int kTileBytes = kTileM * D * 2;         // one 128 x D tile
  // K ring and V ring depth (one tile per CTA: small enough for two CTAs per SM)
  static constexpr int kStages = T == 2 ? ((D == 128) ? 2 : 3) : ((D == 128) ? 1 : 2);
  static constexpr int kOffQ = 0;                           // T Q tiles
  static constexpr int kOffK = T * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S],
  //           s_full[2], p_full[2], pv_done[2], drain, (kSepP) s_free[2]
  static constexpr int kNumBars = 1 + 4 * kStages + 6 + 1 + (kSepP ? 2 : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
};

struct FwdBars {
  uint32_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, pv_done, drain, s_free;
  int stages;
  __device__ uint32_t kf(int s) const { return k_full + 8 * s; }
  __device__ uint32_t ke(int s) const { return k_empty + 8 * s; }
  __device__ uint32_t vf(int s) const { return v_full + 8 * s; }
  __device__ uint32_t ve(int s) const { return v_empty + 8 * s; }
  __device__ uint32_t sf(int t) const { return s_full + 8 * t; }
  __device__ uint32_t pf(int t) const { return p_full + 8 * t; }
  __device__ uint32_t pv(int t) const { return pv_done + 8 * t; }
  __device__ uint32_t sfr(int t) const { return s_free + 8 * t; }
};

// Bounded wait used on the abort path: only the limit can end it.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) {
      atomicOr(status, kStatusWaitTimeout);
      return;
    }
  }
}

template <int D, bool kBf16, int T>
__global__ void __launch_bounds__(FwdCfg<D, T>::kThreads, 3 - T)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = FwdCfg<D, T>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  FwdBars bars;
  bars.stages = NS;
  bars.q_full = sbase + Cfg::kOffBar;
  bars.k_full = bars.q_full + 8;
  bars.k_empty = bars.k_full + 8 * NS;
  bars.v_full = bars.k_empty + 8 * NS;
  bars.v_empty = bars.v_full + 8 * NS;
  bars.s_full = bars.v_empty + 8 * NS;
  bars.p_full = bars.s_full + 16;
  bars.pv_done = bars.p_full + 16;
  bars.drain = bars.pv_done + 16;
  bars.s_free = bars.drain + 8;

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());

  // ---- work assignment: T consecutive query tiles, heaviest units first (causal) ----
  const int BHq = p.B * p.Hq;
  const int unit = p.n_units - 1 - static_cast<int>(blockIdx.x) / BHq;
  const int bh = static_cast<int>(blockIdx.x) % BHq;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  // key/value tiles each query tile walks (0 past the sequence end). Causal:
  // query tile qt's rows end below q_end = min(128 (qt + 1), Sq) and see keys
  // below q_end + kv_offset <= Skv, i.e. tiles up to qt + kv_tiles_ahead for a
  // full tile and every tile for the last, ragged one.
  const int n_kv_total = (p.Skv + kTileN - 1) / kTileN;
  int n_t[2] = {0, 0};
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const int q0 = unit * T * kTileM + t * kTileM;
    if (q0 >= p.Sq) n_t[t] = 0;
    else n_t[t] = p.causal ? min(q0 / kTileN + p.kv_tiles_ahead, n_kv_total) : n_kv_total;
  }
  const int n_load = max(n_t[0], n_t[1]);
  if (threadIdx.x == 0) {
    trace_span(p.trace, 0, clock64());
    trace_span(p.trace, 1, smid());
    trace_span(p.trace, 2, n_t[0] + n_t[1]);
  }

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.kf(s), 1);
      mbar_init(bars.ke(s), 1);
      mbar_init(bars.vf(s), 1);
      mbar_init(bars.ve(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.sf(t), 1);
      mbar_init(bars.pf(t), 4);   // one arrival per softmax warp
      mbar_init(bars.pv(t), 1);
    }
    if (Cfg::kSepP) mbar_init(bars.sfr(0), 4);   // one arrival per softmax warp
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint32_t q_bytes = (n_t[0] > 0 ? Cfg::kTileBytes : 0) + (n_t[1] > 0 ? Cfg::kTileBytes : 0);
      if (q_bytes) {
        mbar_arrive_expect_tx(bars.q_full, q_bytes);
        for (int t = 0; t < T; ++t) {
          if (n_t[t] == 0) continue;
          const int q0 = unit * T * kTileM + t * kTileM;
          for (int c = 0; c < Cfg::kChunks; ++c)
            tma_load_3d(sbase + Cfg::kOffQ + t * Cfg::kTileBytes + c * (kTileM * 128), &p.tm_q,
                        bars.q_full, c * kChunk, q0, bh);
        }
      }
      int j = 0;
      for (; j < n_load; ++j) {
        const int st = j % NS;
        const uint32_t use = static_cast<uint32_t>(j / NS);
        if (j >= NS && !mbar_wait(bars.ke(st), (use - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(bars.kf(st), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(sbase + Cfg::kOffK + st * Cfg::kTileBytes + c * (kTileN * 128), &p.tm_k,
                      bars.kf(st), c * kChunk, j * kTileN, bkv);
        if (j >= NS && !mbar_wait(bars.ve(st), (use - 1) & 1, abort_flag, p.status)) {
          ++j;   // the K load of this iteration is in flight
          break;
        }
        mbar_arrive_expect_tx(bars.vf(st), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(sbase + Cfg::kOffV + st * Cfg::kTileBytes + c * (kTileN * 128), &p.tm_v,
                      bars.vf(st), c * kChunk, j * kTileN, bkv);
      }
      if (*abort_flag) {
        // let every copy already issued land before the CTA releases its memory
        if (q_bytes) drain_wait(bars.q_full, 0, p.status);
        for (int jj = max(0, j - NS); jj < j; ++jj) {
          const int st = jj % NS;
          const uint32_t par = static_cast<uint32_t>(jj / NS) & 1;
          drain_wait(bars.kf(st), par, p.status);
          drain_wait(bars.vf(st), par, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    if (lane == 0 && n_load > 0) {
      constexpr uint32_t idesc_qk = make_idesc(128, kTileN, kBf16, false, false);
      constexpr uint32_t idesc_pv = make_idesc(128, D, kBf16, false, true);
      bool ok = mbar_wait(bars.q_full, 0, abort_flag, p.status);
#ifdef FA_WAIT_TEST
      // wait-limit test build: nothing completes this phase before the abort
      // path's own commit, so the wait runs out
      if (ok) ok = mbar_wait(bars.drain, 0, abort_flag, p.status);
#endif

      auto issue_qk = [&](int t, int st) {   // S_t = Q_t K^T, both K-major
        const uint64_t qa = make_sdesc(sbase + Cfg::kOffQ + t * Cfg::kTileBytes, 16, 1024);
        const uint64_t kb = make_sdesc(sbase + Cfg::kOffK + st * Cfg::kTileBytes, 16, 1024);
        mma_ss_product<D / 16, true, kTileM * 128, true, kTileN * 128>(tmem + t * 128, qa, kb,
                                                                       idesc_qk, 0);
        tc_commit(bars.sf(t));
      };
      auto issue_pv = [&](int t, int st, bool accumulate) {   // O_t (+)= P_t V
        const uint64_t vb =
            make_sdesc(sbase + Cfg::kOffV + st * Cfg::kTileBytes, kTileN * 128, 1024);
        const uint32_t o_t = tmem + 128 * T + t * 128;
        mma_ts_product8<false, 0>(o_t, Cfg::kSepP ? o_t + D : tmem + t * 128, vb, idesc_pv,
                                  accumulate ? 1u : 0u);
        tc_commit(bars.pv(t));
      };

      Tracer tr(p.trace, 1);
      if (ok) ok = mbar_wait(bars.kf(0), 0, abort_flag, p.status);
      tr(9);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < T; ++t)
          if (n_t[t] > 0) issue_qk(t, 0);
        tc_commit(bars.ke(0));
      }
      for (int j = 0; ok && j < n_load; ++j) {
        const int st = j % NS;
        const uint32_t par = static_cast<uint32_t>(j / NS) & 1;
        bool k_next = false, v_cur = false;   // K_{j+1}, V_j seen landed
        for (int t = 0; t < T && ok; ++t) {
          if constexpr (Cfg::kSepP) {
            if (j + 1 < n_t[t]) {
              const int st1 = (j + 1) % NS;
              const uint32_t par1 = static_cast<uint32_t>((j + 1) / NS) & 1;
              if (!k_next && !(ok = mbar_wait(bars.kf(st1), par1, abort_flag, p.status))) break;
              k_next = true;
              // S_t(j) has been read out of TMEM: S_t(j + 1) may overwrite it
              if (!(ok = mbar_wait(bars.sfr(t), j & 1, abort_flag, p.status))) break;
              tr(54 + t);
              tc_fence_after();
              issue_qk(t, st1);
            }
          }
          if (j >= n_t[t]) continue;
          if (!v_cur && !(ok = mbar_wait(bars.vf(st), par, abort_flag, p.status))) break;
          v_cur = true;
          if (!(ok = mbar_wait(bars.pf(t), j & 1, abort_flag, p.status))) break;
          tr(50 + t);
          tc_fence_after();
          issue_pv(t, st, j > 0);
          if (!Cfg::kSepP && j + 1 < n_t[t]) {
            const int st1 = (j + 1) % NS;
            const uint32_t par1 = static_cast<uint32_t>((j + 1) / NS) & 1;
            if (!(ok = mbar_wait(bars.kf(st1), par1, abort_flag, p.status))) break;
            // P_t(j) lives in S_t's columns: wait until P_t(j) V_j has read it.
            if (!(ok = mbar_wait(bars.pv(t), j & 1, abort_flag, p.status))) break;
            tr(54 + t);
            tc_fence_after();
            issue_qk(t, st1);
          }
        }
        if (!ok) break;
        tc_commit(bars.ve(st));
        if (j + 1 < n_load) tc_commit(bars.ke((j + 1) % NS));
      }
      if (!ok) {
        // every MMA issued so far must finish before the TMEM is released
        tc_commit(bars.drain);
        drain_wait(bars.drain, 0, p.status);
      }
    }
  } else {
    // ===================== softmax / correction / epilogue =====================
    const int t = (warp - 2) / 4;               // query tile of this warp group
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;          // row within the tile
    const int q0 = unit * T * kTileM + t * kTileM;
    const int row = q0 + r;
    const int n = n_t[t];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + t * 128;
    const uint32_t o_tmem = tmem + lane_off + 128 * T + t * 128;
    const uint32_t p_tmem = Cfg::kSepP ? o_tmem + D : s_tmem;
    const float c = p.scale_log2;

    Tracer tr(((warp == 2 || warp == 6) && lane == 0) ? p.trace : nullptr, 2 + t);
    unsigned n_rescale = 0;    // steps that rescaled O (trace builds record it)
    float m_ref = -INFINITY;   // reference max, scaled log2 domain
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.sf(t), j & 1, abort_flag, p.status));
      if (!ok) break;
      tr(60);
      if (j == 0 && warp == 2 && lane == 0) trace_span(p.trace, 3, clock64());
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
      if constexpr (Cfg::kSepP) {   // the issuer may overwrite S_t with the next tile's
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfr(t));
      }
      const int kv0 = j * kTileN;
      // inline mask: causal (key after the query's position) and keys past the
      // sequence end; lim = last visible key of this row (rows past Sq are
      // never stored, so their limit may run past Skv - 1)
      const int lim = p.causal ? row + p.kv_offset : p.Skv - 1;
      if (kv0 + kTileN - 1 > lim) {
#pragma unroll
        for (int i = 0; i < kTileN; ++i)
          if (kv0 + i > lim) s[i] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
      if constexpr (Cfg::kPaired) {
#pragma unroll
        for (int i = 4; i + 8 <= kTileN; i += 8) {
          mx0 = fmax3(mx0, s[i], s[i + 4]);
          mx1 = fmax3(mx1, s[i + 1], s[i + 5]);
          mx2 = fmax3(mx2, s[i + 2], s[i + 6]);
          mx3 = fmax3(mx3, s[i + 3], s[i + 7]);
        }
        mx0 = fmaxf(mx0, s[kTileN - 4]);
        mx1 = fmaxf(mx1, s[kTileN - 3]);
        mx2 = fmaxf(mx2, s[kTileN - 2]);
        mx3 = fmaxf(mx3, s[kTileN - 1]);
      } else {
#pragma unroll
        for (int i = 4; i < kTileN; i += 4) {
          mx0 = fmaxf(mx0, s[i]);
          mx1 = fmaxf(mx1, s[i + 1]);
          mx2 = fmaxf(mx2, s[i + 2]);
          mx3 = fmaxf(mx3, s[i + 3]);
        }
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      float m_new = m_ref;
      if (mx > m_ref + kRescaleThreshold) m_new = mx;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_ref - m_use);   // 0 when m_ref = -inf
      const bool moved = (m_new != m_ref);
      m_ref = m_new;

      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (Cfg::kPaired) {
          // element e adds into sum[e % 4] as in the scalar form: pairs with
          // i even into (sum0, sum1), i odd into (sum2, sum3)
          const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_use, -m_use);
          uint64_t s01 = f2_pack(sum[0], sum[1]), s23 = f2_pack(sum[2], sum[3]);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[h * 64 + 2 * i], s[h * 64 + 2 * i + 1]), c2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            if (i & 1) s23 = f2_add(s23, f2_pack(p0, p1));
            else s01 = f2_add(s01, f2_pack(p0, p1));
            pk[i] = pack2<kBf16>(p0, p1);
          }
          f2_unpack(s01, sum[0], sum[1]);
          f2_unpack(s23, sum[2], sum[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = ex2(fmaf(s[h * 64 + 2 * i], c, -m_use));
            const float p1 = ex2(fmaf(s[h * 64 + 2 * i + 1], c, -m_use));
            sum[(2 * i) & 3] += p0;
            sum[(2 * i + 1) & 3] += p1;
            pk[i] = pack2<kBf16>(p0, p1);
          }
        }
        if (Cfg::kSepP && h == 0 && j > 0) {
          // P_t(j - 1) V_{j-1} has read the P buffer (and O may be rescaled)
          ok = __all_sync(0xffffffffu, mbar_wait(bars.pv(t), (j - 1) & 1, abort_flag, p.status));
          tc_fence_after();
        }
        tmem_st32(p_tmem + h * 32, pk);
      }
      if (!ok) break;
      l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));

      // O <- alpha * O for rows whose reference max moved (not needed for the
      // first tile: its P V overwrites O)
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        ++n_rescale;
        if constexpr (!Cfg::kSepP) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.pv(t), (j - 1) & 1, abort_flag, p.status));
          if (!ok) break;
          tc_fence_after();
        }
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
      if (lane == 0) mbar_arrive(bars.pf(t));
      tr(61);
    }

    if (lane == 0 && quarter == 2) trace_span(p.trace, 5 + 2 * t, n_rescale);
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.pv(t), (n - 1) & 1, abort_flag, p.status));
      if (warp == 2 && lane == 0) trace_span(p.trace, 4, clock64());
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
          p.lse[static_cast<size_t>(bh) * p.Sq + row] = (m_ref + __log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_span(p.trace, 6, clock64());
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int D, bool kBf16, int T>
cudaError_t launch_fwd_impl(const FwdParams& p0, cudaStream_t stream) {
  constexpr int smem = FwdCfg<D, T>::kSmemBytes;
  auto kernel = fa_fwd_kernel<D, kBf16, T>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdParams p = p0;
  p.n_units = (p.Sq + T * kTileM - 1) / (T * kTileM);   // T query tiles per CTA
  const unsigned grid =
      static_cast<unsigned>(static_cast<long long>(p.B) * p.Hq * p.n_units);   // < 2^31
  kernel<<<grid, FwdCfg<D, T>::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// One query tile per CTA when the grid has at least kOneTileWaves one-tile
// CTAs per SM (two co-reside per SM and overlap each other's loads, softmax
// and start-up), else two tiles per CTA (ping-pong inside the CTA, which a
// lone CTA in a grid's last wave still has). d = 64 always takes one tile:
// its separate P buffer lets each CTA overlap the next Q K^T with its own
// softmax, which beats the two-tile form at every grid size. FA_FWD_TILES=1
// or 2 in the environment forces one form for every call; both compute the
// same bits.
constexpr int kOneTileWaves = 4;

template <int D, bool kBf16>
cudaError_t launch_fwd_d(const FwdParams& p, cudaStream_t stream) {
  int tiles = 0;
  const char* env = std::getenv("FA_FWD_TILES");
  if (env && (env[0] == '1' || env[0] == '2') && env[1] == 0) tiles = env[0] - '0';
  if (tiles == 0 && D == 64) tiles = 1;
  if (tiles == 0) {
    int dev = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long one_tile_ctas =
        static_cast<long long>(p.B) * p.Hq * ((p.Sq + kTileM - 1) / kTileM);
    tiles = one_tile_ctas >= static_cast<long long>(kOneTileWaves) * n_sm ? 1 : 2;
  }
  return tiles == 1 ? launch_fwd_impl<D, kBf16, 1>(p, stream) : launch_fwd_impl<D, kBf16, 2>(p, stream);
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_fwd_d<128, true>(p, stream) : launch_fwd_d<128, false>(p, stream);
  return bf16 ? launch_fwd_d<64, true>(p, stream) : launch_fwd_d<64, false>(p, stream);
}

}  // namespace fa
