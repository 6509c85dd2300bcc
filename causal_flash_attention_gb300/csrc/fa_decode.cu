// Split-KV forward for few query rows per head (decode: one or a few new
// tokens against a long key/value cache) on sm_103a.
//
// Same result as the forward kernel: per query row, out = softmax(mask(q K^T *
// scale)) V and LSE, with the causal mask aligned to the last key (query row s
// stands at position s + Skv - Sq; "Phase 14: Flash Attention 2 for SM120",
// section Causal Mask, kv_offset = kv_len - q_len, introduced for a KV cache
// longer than Q). The work is laid out for that shape instead of one CTA per
// 256 query rows, which would leave most of the GPU idle and stream each
// key/value head once per query head:
//
//   - the G query heads that share a key/value head are packed into one
//     128-row query tile (row r = gq * Sq + s, R = G * Sq <= 128 real rows), so
//     each key/value tile is read once for all of them;
//   - the key/value sequence of a head is cut into `n_splits` ranges of whole
//     128-key tiles, one CTA each, so that B * Hkv * n_splits CTAs stream the
//     cache in parallel ("Phase 14", section 已知局限与后续优化方向, item 1:
//     a dedicated decode kernel that reduces in parallel along the key/value
//     dimension);
//   - each CTA runs the online-softmax recurrence over its range and writes
//     its partial result out_s = O / l and lse2_s = m + log2 l (base 2, scaled
//     scores); a merge kernel combines the ranges with the same rescaling the
//     recurrence uses when its running max grows ("FlashAttention 与 SDPA
//     Backend", section Online softmax 的三个状态):
//       M = max_s lse2_s,  w_s = 2^(lse2_s - M),  out = sum_s w_s out_s / sum_s w_s,
//       LSE = (M + log2 sum_s w_s) * ln 2.
//     With one range the CTA writes the final out and LSE itself.
//
// The tile loop is HBM-bound (the query tile is mostly padding rows, so the
// tensor-core work per key tile is small next to its 2 * 128 * d * 2 bytes),
// which sets the design: K and V tiles stream through 3-deep TMA rings, the
// score tile is double-buffered in tensor memory (S_0, S_1) so that the next
// Q K^T runs while the softmax works on the current one, and O accumulates in
// tensor memory.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 one thread per query-tile row (they also stage the query
// rows into shared memory at the start).
//
// Tensor memory: S_0 [0,128), S_1 [128,256), O [256, 256+d).
#include <algorithm>
#include <type_traits>

#include "fa_decode.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 192;
constexpr float kLn2D = 0.6931471805599453f;
constexpr float kRescaleThresholdD = 8.0f;   // same lazy-rescale rule as the forward

template <int D>
struct DecCfg {
  static constexpr int kChunks = D / kChunk;
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // q_ready, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2],
  // p_full[2], pv_done[2], drain
  static constexpr int kNumBars = 1 + 4 * kStages + 6 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
};

__device__ __forceinline__ void drain_wait_d(uint32_t bar, uint32_t parity, int* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) {
      atomicOr(status, kStatusWaitTimeout);
      return;
    }
  }
}

template <int D, bool kBf16>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_kernel(const __grid_constant__ DecodeParams p) {
  using Cfg = DecCfg<D>;
  constexpr int NS = Cfg::kStages;
  using Elem = typename std::conditional<kBf16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  const uint32_t bar0 = sbase + Cfg::kOffBar;
  const uint32_t q_ready = bar0;
  auto k_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (1 + NS + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (1 + 2 * NS + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (1 + 3 * NS + s); };
  auto s_full = [&](int b) { return bar0 + 8 * (1 + 4 * NS + b); };
  auto p_full = [&](int b) { return bar0 + 8 * (3 + 4 * NS + b); };
  auto pv_done = [&](int b) { return bar0 + 8 * (5 + 4 * NS + b); };
  const uint32_t drain = bar0 + 8 * (7 + 4 * NS);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());

  // ---- work: key-tile range `split` of (batch, key/value head) ----
  const int split = static_cast<int>(blockIdx.x) % p.n_splits;
  const int bkv = static_cast<int>(blockIdx.x) / p.n_splits;
  const int b = bkv / p.Hkv, kvh = bkv % p.Hkv;
  const int t_begin = split * p.tiles_per_split;
  const int n = min(t_begin + p.tiles_per_split, p.n_kv_tiles) - t_begin;   // >= 1
  const int k_end = min((t_begin + n) * kTileN, p.Skv);                      // one past the last key

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 4);   // one arrival per row warp
    for (int s = 0; s < NS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(s_full(bb), 1);
      mbar_init(p_full(bb), 4);
      mbar_init(pv_done(bb), 1);
    }
    mbar_init(drain, 1);
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
  // the merge kernel (when there is one) may be scheduled now; it waits for
  // this grid's completion before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ===================== TMA producer =====================
    // Lane 0 waits for a free slot and posts the expected bytes. Contiguous:
    // lane 0 then issues the tile's one box per 64-column chunk. Paged: each
    // lane i < 128 / box_rows reads the block-table entry of box i and issues
    // that box itself, so that the boxes of a tile are issued in parallel and
    // no copy waits on a dependent table load.
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    const int n_blocks = p.block_table ? (p.Skv + p.block_size - 1) / p.block_size : 0;
    const int n_boxes = p.block_table ? kTileN / p.box_rows : 1;
    // This lane's part of one 128-key tile into `dst` (chunk c at dst + c *
    // 16 KB). Paged: a block past the sequence, or a table entry outside
    // [0, num_blocks), is loaded from an out-of-range row, which the copy
    // fills with zeros.
    auto load_part = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int tile, int pb) {
      if (!p.block_table) {
        if (lane == 0)
          for (int c = 0; c < Cfg::kChunks; ++c)
            tma_load_3d(dst + c * (kTileN * 128), tm, bar, c * kChunk, tile * kTileN, bkv);
        return;
      }
      if (lane >= n_boxes) return;
      const int key = tile * kTileN + lane * p.box_rows;
      const bool in_range = pb >= 0 && pb < p.num_blocks;
      const int y = in_range ? key % p.block_size : p.block_size;   // out of range: zeros
      const int z = in_range ? pb * p.Hkv + kvh : 0;
      for (int c = 0; c < Cfg::kChunks; ++c)
        tma_load_3d(dst + c * (kTileN * 128) + lane * p.box_rows * 128, tm, bar, c * kChunk, y, z);
    };
    int j = 0;
    for (; j < n; ++j) {
      const int tile = t_begin + j;
      const int st = j % NS;
      const uint32_t use = static_cast<uint32_t>(j / NS);
      int pb = -1;
      if (p.block_table && lane < n_boxes) {
        const int lb = (tile * kTileN + lane * p.box_rows) / p.block_size;
        if (lb < n_blocks) pb = p.block_table[static_cast<size_t>(b) * p.max_blocks + lb];
      }
      int stop = 0;
      if (lane == 0) {
        if (j >= NS && !mbar_wait(k_empty(st), (use - 1) & 1, abort_flag, p.status)) stop = 1;
        else mbar_arrive_expect_tx(k_full(st), Cfg::kTileBytes);
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
      load_part(&p.tm_k, sbase + Cfg::kOffK + st * Cfg::kTileBytes, k_full(st), tile, pb);
      if (lane == 0) {
        if (j >= NS && !mbar_wait(v_empty(st), (use - 1) & 1, abort_flag, p.status)) stop = 1;
        else mbar_arrive_expect_tx(v_full(st), Cfg::kTileBytes);
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) {
        ++j;   // this iteration's K load is in flight
        break;
      }
      load_part(&p.tm_v, sbase + Cfg::kOffV + st * Cfg::kTileBytes, v_full(st), tile, pb);
    }
    if (lane == 0 && *abort_flag) {
      // let every copy already issued land before the CTA releases its memory
      for (int jj = max(0, j - NS); jj < j; ++jj) {
        const uint32_t par = static_cast<uint32_t>(jj / NS) & 1;
        drain_wait_d(k_full(jj % NS), par, p.status);
        drain_wait_d(v_full(jj % NS), par, p.status);
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(128, kTileN, kBf16, false, false);
      constexpr uint32_t idesc_pv = make_idesc(128, D, kBf16, false, true);
      const uint64_t qa = make_sdesc(sbase + Cfg::kOffQ, 16, 1024);
      auto issue_qk = [&](int j) {   // S_(j%2) = Q K_j^T
        const int st = j % NS;
        const uint64_t kb = make_sdesc(sbase + Cfg::kOffK + st * Cfg::kTileBytes, 16, 1024);
        mma_ss_product<D / 16, true, kTileM * 128, true, kTileN * 128>(tmem + (j & 1) * 128, qa, kb,
                                                                       idesc_qk, 0);
        tc_commit(s_full(j & 1));
        tc_commit(k_empty(st));
      };
      bool ok = mbar_wait(q_ready, 0, abort_flag, p.status) &&
                mbar_wait(k_full(0), 0, abort_flag, p.status);
#ifdef FA_WAIT_TEST
      // wait-limit test build: nothing completes this phase before the abort
      // path's own commit, so the wait runs out
      if (ok) ok = mbar_wait(drain, 0, abort_flag, p.status);
#endif
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % NS;
        if (j + 1 < n) {
          // S_((j+1)%2) held P_(j-1), which P_(j-1) V_(j-1) must have read
          const int st1 = (j + 1) % NS;
          if (!(ok = mbar_wait(k_full(st1), static_cast<uint32_t>((j + 1) / NS) & 1, abort_flag,
                               p.status)))
            break;
          if (j >= 1 && !(ok = mbar_wait(pv_done((j - 1) & 1), static_cast<uint32_t>((j - 1) >> 1) & 1,
                                         abort_flag, p.status)))
            break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        if (!(ok = mbar_wait(p_full(j & 1), static_cast<uint32_t>(j >> 1) & 1, abort_flag, p.status)))
          break;
        if (!(ok = mbar_wait(v_full(st), static_cast<uint32_t>(j / NS) & 1, abort_flag, p.status)))
          break;
        tc_fence_after();
        const uint64_t vb = make_sdesc(sbase + Cfg::kOffV + st * Cfg::kTileBytes, kTileN * 128, 1024);
        mma_ts_product8<false, 0>(tmem + 256, tmem + (j & 1) * 128, vb, idesc_pv, j > 0 ? 1u : 0u);
        tc_commit(pv_done(j & 1));
        tc_commit(v_empty(st));
      }
      if (!ok) {
        // every MMA issued so far must finish before the TMEM is released
        tc_commit(drain);
        drain_wait_d(drain, 0, p.status);
      }
    }
  } else {
    // ===== row warps: stage Q, then softmax per key tile, then the epilogue =====
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;          // query-tile row
    const bool real = r < p.R;
    const int gq = real ? r / p.Sq : 0;
    const int s = real ? r % p.Sq : 0;
    const size_t qrow = (static_cast<size_t>(b) * p.Hq + kvh * p.G + gq) * p.Sq + s;
    // Stage the query row into the 128-byte-swizzled K-major query tile
    // (16-byte unit u of a 128-byte row sits at unit u ^ (r % 8)); rows past R
    // are zero.
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.q) + qrow * D);
#pragma unroll
      for (int c = 0; c < Cfg::kChunks; ++c) {
        uint8_t* dst_row = smem + Cfg::kOffQ + c * (kTileM * 128) + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = real ? src[c * 8 + u] : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dst_row + ((u ^ (r & 7)) << 4)) = v;
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);

    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + lane_off + 256;
    const float c = p.scale_log2;
    float m_ref = -INFINITY;   // reference max, scaled log2 domain
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t s_tmem = tmem + lane_off + (j & 1) * 128;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full(j & 1), static_cast<uint32_t>(j >> 1) & 1,
                                             abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      float sc[kTileN];
      {
        uint32_t raw[kTileN];
#pragma unroll
        for (int cc = 0; cc < kTileN / 32; ++cc)
          tmem_ld32(s_tmem + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(raw + cc * 32));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kTileN; ++i) sc[i] = __uint_as_float(raw[i]);
      }
      // Mask: keys past this split's range (they belong to the next split or
      // lie past Skv) and, causal, keys after the row's position s + kv_offset.
      // Rows past R are never stored, so their limit is the range end.
      const int kv0 = (t_begin + j) * kTileN;
      const int lim = (p.causal && real) ? min(s + p.kv_offset, k_end - 1) : k_end - 1;
      if (kv0 + kTileN - 1 > lim) {
#pragma unroll
        for (int i = 0; i < kTileN; ++i)
          if (kv0 + i > lim) sc[i] = -INFINITY;
      }
      float mx0 = sc[0], mx1 = sc[1], mx2 = sc[2], mx3 = sc[3];
#pragma unroll
      for (int i = 4; i < kTileN; i += 4) {
        mx0 = fmaxf(mx0, sc[i]);
        mx1 = fmaxf(mx1, sc[i + 1]);
        mx2 = fmaxf(mx2, sc[i + 2]);
        mx3 = fmaxf(mx3, sc[i + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      float m_new = m_ref;
      if (mx > m_ref + kRescaleThresholdD) m_new = mx;
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
          const float p0 = ex2(fmaf(sc[h * 64 + 2 * i], c, -m_use));
          const float p1 = ex2(fmaf(sc[h * 64 + 2 * i + 1], c, -m_use));
          sum[(2 * i) & 3] += p0;
          sum[(2 * i + 1) & 3] += p1;
          pk[i] = pack2<kBf16>(p0, p1);
        }
        tmem_st32(s_tmem + h * 32, pk);
      }
      l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));

      // O <- alpha * O for rows whose reference max moved (the first tile's
      // P V overwrites O)
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done((j - 1) & 1),
                                               static_cast<uint32_t>((j - 1) >> 1) & 1, abort_flag,
                                               p.status));
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
      if (lane == 0) mbar_arrive(p_full(j & 1));
    }

    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(pv_done((n - 1) & 1),
                                             static_cast<uint32_t>((n - 1) >> 1) & 1, abort_flag,
                                             p.status));
      if (ok) {
        tc_fence_after();
        // a row that sees no key of this range contributes weight 0 to the merge
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse2 = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
        if (p.n_splits == 1) {
          Elem* orow = static_cast<Elem*>(p.out) + qrow * D;
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
            if (real) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
          if (real) p.lse[qrow] = lse2 * kLn2D;
        } else {
          const size_t prow = (static_cast<size_t>(bkv) * p.n_splits + split) * p.R + r;
          float* orow = p.part_out + prow * D;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(o_tmem + cc * 32, o);
            tmem_wait_ld();
            if (real) {
              float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                     __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
            }
          }
          if (real) p.part_lse2[prow] = lse2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ merge --
// One warp per output row (b, hq, s); each lane owns d / 32 columns. The
// merge is latency-bound (a few KB per row), so the loads are batched: the
// first batch of up to kMergeBatch ranges' partial rows and their lse2 values
// is issued before the maximum over all ranges' lse2 is reduced (lane i reads
// ranges i, i + 32, ...), and every lane forms the same weights
// 2^(lse2 - M) from broadcast reads, so the row sum needs no reduction.
constexpr int kMergeBatch = 16;

template <int PER>
struct alignas(4 * PER) MergeVec { float x[PER]; };

template <typename T, int PER>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeMergeParams p) {
  // Launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partial results are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;   // (b * Hq + hq) * Sq + s
  if (row >= static_cast<long long>(p.B) * p.Hq * p.Sq) return;
  const int s = static_cast<int>(row % p.Sq);
  const long long bh = row / p.Sq;
  const int hq = static_cast<int>(bh % p.Hq), b = static_cast<int>(bh / p.Hq);
  const int bkv = b * p.Hkv + hq / p.G;
  const int r = (hq % p.G) * p.Sq + s;
  const size_t base = static_cast<size_t>(bkv) * p.n_splits;
  const int n = p.n_splits;
  using V = MergeVec<PER>;
  auto part = [&](int sp) {
    return reinterpret_cast<const V*>(p.part_out + ((base + sp) * p.R + r) * p.d)[lane];
  };
  auto lse2_of = [&](int sp) { return p.part_lse2[(base + sp) * p.R + r]; };

  V v[kMergeBatch];
  float lv[kMergeBatch];
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k)
    if (k < n) {
      v[k] = part(k);
      lv[k] = lse2_of(k);
    }
  float M = -INFINITY;
  for (int sp = lane; sp < n; sp += 32) M = fmaxf(M, lse2_of(sp));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int sp0 = 0; sp0 < n; sp0 += kMergeBatch) {
    if (sp0 > 0) {
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k)
        if (sp0 + k < n) {
          v[k] = part(sp0 + k);
          lv[k] = lse2_of(sp0 + k);
        }
    }
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k)
      if (sp0 + k < n) {
        const float w = M != -INFINITY ? ex2(lv[k] - M) : 0.f;   // an empty range has lse2 = -inf
        L += w;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[k].x[e], acc[e]);
      }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  T* dst = static_cast<T*>(p.out) + row * p.d + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[e] = static_cast<T>(acc[e] * inv);
  if (lane == 0) p.lse[row] = L > 0.f ? (M + __log2f(L)) * kLn2D : -INFINITY;
}

template <int D, bool kBf16>
cudaError_t launch_decode_impl(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = DecCfg<D>::kSmemBytes;
  auto kernel = fa_decode_kernel<D, kBf16>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.n_splits * p.B * p.Hkv);
  kernel<<<grid, kDecThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128)
    return bf16 ? launch_decode_impl<128, true>(p, stream) : launch_decode_impl<128, false>(p, stream);
  return bf16 ? launch_decode_impl<64, true>(p, stream) : launch_decode_impl<64, false>(p, stream);
}

// The merge runs as a programmatic dependent launch of the split kernel on the
// same stream, so that its launch overlaps the split kernel's tail.
cudaError_t launch_decode_merge(const DecodeMergeParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dtype == 2)
    return p.d == 128 ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<__nv_bfloat16, 4>, p)
                      : cudaLaunchKernelEx(&cfg, decode_merge_kernel<__nv_bfloat16, 2>, p);
  return p.d == 128 ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<__half, 4>, p)
                    : cudaLaunchKernelEx(&cfg, decode_merge_kernel<__half, 2>, p);
}

}  // namespace fa
