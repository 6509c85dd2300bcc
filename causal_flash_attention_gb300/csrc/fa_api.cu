// C-ABI entry points of libfa (declared in include/fa.h): argument checks,
// TMA descriptor construction and kernel launches. No device memory is
// allocated here; the only device-resident state is the status word below.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/fa.h"
#include "fa_decode.h"
#include "fa_internal.h"

namespace fa {

// Sticky device status word: kernels OR kStatus* bits into it when they give
// up a wait instead of hanging.
__device__ int g_status;

namespace {

constexpr float kLog2e = 1.4426950408889634f;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Device address of g_status on the current device, looked up once per
// device (the lookup is a runtime call worth microseconds of host time).
constexpr int kMaxDevices = 128;
std::atomic<int*> g_status_ptr[kMaxDevices];

int* status_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status) != cudaSuccess) return nullptr;
  g_status_ptr[dev].store(p, std::memory_order_release);
  return p;
}

// 3-D view [rows = BH][S][d] of a contiguous 16-bit tensor; box = 64 columns
// (128 bytes, one swizzle span) x 128 sequence rows x 1 head.
bool make_tmap(CUtensorMap* m, const void* base, int BH, int S, int d, bool bf16,
               int box_rows = kTileM) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(S) * d * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view [BH][S_pad][d] of the fp32 dQ accumulator for bulk reduce-adds;
// box = 32 columns (128 bytes) x 32 rows x 1 head, 128-byte swizzle.
bool make_tmap_acc(CUtensorMap* m, float* base, int BH, int S_pad, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(S_pad),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(S_pad) * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sq query rows against Skv key/value rows. Under the causal mask query row i
// stands at position i + (Skv - Sq), so every row sees at least one key only
// when Skv >= Sq; fewer keys than queries is a shape error.
int check_common(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, float scale,
                 int dtype) {
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1 || Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_SHAPE;
  if (causal && Skv < Sq) return FA_ERR_SHAPE;
  // grid and index ranges: up to B*Hq*ceil(Sq/128) forward CTAs; B*Hkv*ceil(Skv/128)
  // backward work items, claimed from a 32-bit counter that runs past the
  // last item by at most one claim per CTA (so the bound keeps 2^16 of
  // headroom); element offsets in 64 bits
  const long long bh = static_cast<long long>(B) * Hq;
  const long long bhkv = static_cast<long long>(B) * Hkv;
  if (bh > (1LL << 30) || Sq > (1 << 30) || Skv > (1 << 30) ||
      bh * ((Sq + 127) / 128) > 0x7fffffffLL ||
      bhkv * ((Skv + 127) / 128) > 0x7fffffffLL - 0xffffLL)
    return FA_ERR_SHAPE;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_SCALE;
  return FA_OK;
}

inline long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

// Forward kernel for 16-bit inputs at d = 128: the CTA-pair kernel
// (fa_fwd_pair.cu, tcgen05 cta_group::2) or the single-CTA one (fa_fwd.cu).
// Both compute the same function. FA_FWD_CTA_PAIR=1 (or 0) in the environment
// selects one for every call; otherwise kPairForwardDefault does.
constexpr bool kPairForwardDefault = false;

bool use_pair_forward(int d) {
  if (d != 128) return false;
  const char* e = std::getenv("FA_FWD_CTA_PAIR");
  if (e && e[0] == '1') return true;
  if (e && e[0] == '0') return false;
  return kPairForwardDefault;
}

struct WsLayout {
  size_t dq_acc, delta, lse2, work, total;
};

WsLayout ws_layout(int B, int Hq, int Sq, int d) {
  const long long bh = static_cast<long long>(B) * Hq;
  const long long s_pad = round_up(Sq, kTileM);
  WsLayout w;
  w.dq_acc = 0;
  w.delta = static_cast<size_t>(round_up(bh * s_pad * d * 4, 256));
  w.lse2 = w.delta + static_cast<size_t>(round_up(bh * s_pad * 4, 256));
  w.work = w.lse2 + static_cast<size_t>(round_up(bh * s_pad * 4, 256));
  w.total = w.work + 256;   // the backward's work-item counter
  return w;
}

// Split-KV plan of fa_fwd_splitkv: key tiles per CTA, CTA count per (batch,
// key/value head) and the partial-result workspace. One CTA fits on an SM at a
// time and each CTA pays a start-up (barriers, tensor memory, query staging,
// first-load latency), so the automatic choice is the largest range count that
// keeps every CTA in one wave on the 152 SMs (one range when the (batch,
// key/value head) pairs alone fill the GPU), never an empty range.
constexpr int kDecodeWaveCtas = 152;
constexpr int kDecodeMaxRows = 128;   // G * Sq rows must fit one query tile

struct SplitPlan {
  int n_splits, tiles_per_split, R;
  size_t part_out, part_lse2, total;
};

SplitPlan split_plan(int B, int Hq, int Hkv, int Sq, int Skv, int d, int n_splits_req) {
  SplitPlan sp;
  const int n_tiles = (Skv + kTileN - 1) / kTileN;
  const long long bhkv = static_cast<long long>(B) * Hkv;
  long long want = n_splits_req > 0 ? n_splits_req : kDecodeWaveCtas / bhkv;
  want = std::max(1LL, std::min<long long>(want, n_tiles));
  sp.tiles_per_split = static_cast<int>((n_tiles + want - 1) / want);
  sp.n_splits = (n_tiles + sp.tiles_per_split - 1) / sp.tiles_per_split;
  sp.R = (Hq / Hkv) * Sq;
  sp.part_out = 0;
  if (sp.n_splits == 1) {
    sp.part_lse2 = sp.total = 0;
  } else {
    const long long rows = bhkv * sp.n_splits * sp.R;
    sp.part_lse2 = static_cast<size_t>(round_up(rows * d * 4, 256));
    sp.total = sp.part_lse2 + static_cast<size_t>(round_up(rows * 4, 256));
  }
  return sp;
}

}  // namespace

int check_bwd_args(const void* q, const void* k, const void* v, const void* out,
                   const void* dout, const float* lse, const void* dq, const void* dk,
                   const void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                   float scale, int dtype) {
  int rc = check_common(B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype);
  if (rc != FA_OK) return rc;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGN;
  return FA_OK;
}

}  // namespace fa

using namespace fa;

#ifdef FA_TRACE
// Trace builds only: the device buffer kernels record their timelines into
// (kTraceCtas x kTraceRoles x kTraceSlots 64-bit entries), or null.
static unsigned long long* g_trace_buf = nullptr;
extern "C" void fa_trace_set(void* buf) { g_trace_buf = static_cast<unsigned long long*>(buf); }
#define FA_TRACE_PTR g_trace_buf
#else
#define FA_TRACE_PTR nullptr
#endif

extern "C" {

int fa_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_SHAPE:
      return "invalid shape (B, Hq, Hkv, S >= 1, Hq % Hkv == 0, d in {64, 128}, causal Skv >= Sq)";
    case FA_ERR_DTYPE: return "unsupported dtype (FA_F32, FA_F16 or FA_BF16)";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_bwd_workspace_bytes()";
    case FA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_TMA: return "the driver rejected a tensor-memory-access descriptor";
    case FA_ERR_NOALLOC_LIMIT:
      return "sizes need more scratch than fa_bwd_noalloc's fixed FA_NOALLOC_SCRATCH_BYTES";
    default: return "unknown error code";
  }
}

int fa_fwd_kv(const void* q, const void* k, const void* v, void* out, float* lse, int B,
              int Hq, int Hkv, int Sq, int Skv, int d, int causal, float scale, int dtype,
              fa_stream_t stream) {
  int rc = check_common(B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype);
  if (rc != FA_OK) return rc;
  if (!q || !k || !v || !out || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int kv_offset = causal ? Skv - Sq : 0;

  if (dtype == FA_F32) {
    SimtParams p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.o_out = static_cast<float*>(out);
    p.lse_out = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.kv_offset = kv_offset; p.d = d;
    p.causal = causal != 0;
    p.scale = scale;
    return launch_fwd_simt(p, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  const bool bf16 = dtype == FA_BF16;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_tmap(&p.tm_q, q, B * Hq, Sq, d, bf16) || !make_tmap(&p.tm_k, k, B * Hkv, Skv, d, bf16) ||
      !make_tmap(&p.tm_v, v, B * Hkv, Skv, d, bf16))
    return FA_ERR_TMA;
  p.out = out;
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.kv_offset = kv_offset;
  p.causal = causal != 0;
  p.scale_log2 = scale * kLog2e;
  p.kv_tiles_ahead = 1 + (kv_offset + kTileN - 1) / kTileN;
  p.trace = FA_TRACE_PTR;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  if (use_pair_forward(d)) {
    if (!make_tmap(&p.tm_k_half, k, B * Hkv, Skv, d, bf16, kTileN / 2)) return FA_ERR_TMA;
    p.n_qblocks = (Sq + 4 * kTileM - 1) / (4 * kTileM);
    return launch_fwd_pair(p, bf16, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  return launch_fwd_tc(p, d, bf16, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
           int Hkv, int S, int d, int causal, float scale, int dtype, fa_stream_t stream) {
  return fa_fwd_kv(q, k, v, out, lse, B, Hq, Hkv, S, S, d, causal, scale, dtype, stream);
}

size_t fa_bwd_kv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d) {
  // the causal constraint is checked by fa_bwd_kv itself
  if (check_common(B, Hq, Hkv, Sq, Skv, d, 0, 1.f, FA_BF16) != FA_OK) return 0;
  return ws_layout(B, Hq, Sq, d).total;
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int S, int d) {
  return fa_bwd_kv_workspace_bytes(B, Hq, Hkv, S, S, d);
}

int fa_bwd_kv(const void* q, const void* k, const void* v, const void* out, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
              int Skv, int d, int causal, float scale, int dtype, void* workspace,
              size_t workspace_bytes, fa_stream_t stream) {
  int rc = check_bwd_args(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Skv, d, causal,
                          scale, dtype);
  if (rc != FA_OK) return rc;
  const WsLayout ws = ws_layout(B, Hq, Sq, d);
  if (!workspace || workspace_bytes < ws.total) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  const int BH = B * Hq;
  const int Sq_pad = static_cast<int>(round_up(Sq, kTileM));
  const int kv_offset = causal ? Skv - Sq : 0;

  float* delta = reinterpret_cast<float*>(wsb + ws.delta);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  float* dq_acc = dtype == FA_F32 ? nullptr : reinterpret_cast<float*>(wsb + ws.dq_acc);
  int* status = status_ptr();
  if (!status) return FA_ERR_CUDA;

  // Everything that can fail on the host (descriptor encoding, the status
  // lookup) happens before the first kernel is enqueued.
  const bool bf16 = dtype == FA_BF16;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (dtype != FA_F32 &&
      (!make_tmap(&p.tm_q, q, BH, Sq, d, bf16) || !make_tmap(&p.tm_k, k, B * Hkv, Skv, d, bf16) ||
       !make_tmap(&p.tm_v, v, B * Hkv, Skv, d, bf16) ||
       !make_tmap(&p.tm_do, dout, BH, Sq, d, bf16) ||
       !make_tmap_acc(&p.tm_dq, dq_acc, BH, Sq_pad, d) ||
       !make_tmap(&p.tm_dk, dk, B * Hkv, Skv, d, bf16, 32) ||
       !make_tmap(&p.tm_dv, dv, B * Hkv, Skv, d, bf16, 32)))
    return FA_ERR_TMA;

  BwdPreParams pre;
  pre.out = out;
  pre.dout = dout;
  pre.lse = lse;
  pre.delta = delta;
  pre.lse2 = lse2;
  pre.dq_acc = dq_acc;
  pre.work = dtype == FA_F32 ? nullptr : reinterpret_cast<int*>(wsb + ws.work);
  pre.BH = BH; pre.Sq = Sq; pre.Sq_pad = Sq_pad; pre.d = d;
  pre.dtype = dtype;
  if (launch_bwd_pre(pre, st) != cudaSuccess) return FA_ERR_CUDA;

  if (dtype == FA_F32) {
    SimtParams sp{};
    sp.q = static_cast<const float*>(q);
    sp.k = static_cast<const float*>(k);
    sp.v = static_cast<const float*>(v);
    sp.dout = static_cast<const float*>(dout);
    sp.lse = lse;
    sp.delta = delta;
    sp.dq = static_cast<float*>(dq);
    sp.dk = static_cast<float*>(dk);
    sp.dv = static_cast<float*>(dv);
    sp.B = B; sp.Hq = Hq; sp.Hkv = Hkv; sp.Sq = Sq; sp.Skv = Skv; sp.kv_offset = kv_offset;
    sp.d = d;
    sp.causal = causal != 0;
    sp.scale = scale;
    return launch_bwd_simt(sp, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  p.delta = delta;
  p.lse2 = lse2;
  p.dq_acc = dq_acc;
  p.work = reinterpret_cast<int*>(wsb + ws.work);
  p.dk = dk;
  p.dv = dv;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.Sq_pad = Sq_pad;
  p.kv_offset = kv_offset;
  p.causal = causal != 0;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.n_kv_tiles = (Skv + kTileN - 1) / kTileN;
  p.n_q_tiles = (Sq + kTileM - 1) / kTileM;
  p.trace = FA_TRACE_PTR;
  p.status = status;
  if (launch_bwd_tc(p, d, bf16, st) != cudaSuccess) return FA_ERR_CUDA;

  DqConvertParams cv;
  cv.dq_acc = dq_acc;
  cv.dq = dq;
  cv.BH = BH; cv.Sq = Sq; cv.Sq_pad = Sq_pad; cv.d = d;
  cv.scale = scale;
  cv.dtype = dtype;
  return launch_dq_convert(cv, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int d,
           int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
           fa_stream_t stream) {
  return fa_bwd_kv(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, S, S, d, causal, scale, dtype,
                   workspace, workspace_bytes, stream);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                      int n_splits) {
  if (check_common(B, Hq, Hkv, Sq, Skv, d, 0, 1.f, FA_BF16) != FA_OK || n_splits < 0 ||
      (Hq / Hkv) * Sq > kDecodeMaxRows)
    return 0;
  return split_plan(B, Hq, Hkv, Sq, Skv, d, n_splits).total;
}

}  // extern "C"

namespace {

// Shared body of fa_fwd_splitkv and fa_fwd_splitkv_paged (block_table null:
// contiguous K/V).
int splitkv_impl(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                 int Hkv, int Sq, int Skv, int d, int causal, float scale, int dtype, int n_splits,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream,
                 const int* block_table, int block_size, int max_blocks, int num_blocks) {
  const bool paged = block_table != nullptr;
  const SplitPlan sp = split_plan(B, Hq, Hkv, Sq, Skv, d, n_splits);
  if (sp.total > 0 && (!workspace || workspace_bytes < sp.total)) return FA_ERR_WORKSPACE;
  if (sp.total > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == FA_BF16;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  if (paged) {
    p.box_rows = std::min(block_size, kTileN);
    if (!make_tmap(&p.tm_k, k, num_blocks * Hkv, block_size, d, bf16, p.box_rows) ||
        !make_tmap(&p.tm_v, v, num_blocks * Hkv, block_size, d, bf16, p.box_rows))
      return FA_ERR_TMA;
    p.block_table = block_table;
    p.block_size = block_size;
    p.max_blocks = max_blocks;
    p.num_blocks = num_blocks;
  } else if (!make_tmap(&p.tm_k, k, B * Hkv, Skv, d, bf16) ||
             !make_tmap(&p.tm_v, v, B * Hkv, Skv, d, bf16)) {
    return FA_ERR_TMA;
  }
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.part_out = sp.total ? reinterpret_cast<float*>(wsb + sp.part_out) : nullptr;
  p.part_lse2 = sp.total ? reinterpret_cast<float*>(wsb + sp.part_lse2) : nullptr;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv;
  p.kv_offset = causal ? Skv - Sq : 0;
  p.causal = causal != 0;
  p.G = Hq / Hkv;
  p.R = sp.R;
  p.n_kv_tiles = (Skv + kTileN - 1) / kTileN;
  p.tiles_per_split = sp.tiles_per_split;
  p.n_splits = sp.n_splits;
  p.scale_log2 = scale * kLog2e;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  if (launch_decode(p, d, bf16, st) != cudaSuccess) return FA_ERR_CUDA;
  if (sp.n_splits == 1) return FA_OK;

  DecodeMergeParams m;
  m.part_out = p.part_out;
  m.part_lse2 = p.part_lse2;
  m.out = out;
  m.lse = lse;
  m.B = B; m.Hq = Hq; m.Hkv = Hkv; m.Sq = Sq; m.G = p.G; m.R = p.R; m.d = d;
  m.n_splits = sp.n_splits;
  m.dtype = dtype;
  return launch_decode_merge(m, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                   int Hq, int Hkv, int Sq, int Skv, int d, int causal, float scale, int dtype,
                   int n_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  int rc = check_common(B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype);
  if (rc != FA_OK) return rc;
  if (n_splits < 0 || (Hq / Hkv) * Sq > kDecodeMaxRows) return FA_ERR_SHAPE;
  if (!q || !k || !v || !out || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if (dtype == FA_F32)   // plain fp32 arithmetic: one warp per query row, no split
    return fa_fwd_kv(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype, stream);
  return splitkv_impl(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype, n_splits,
                      workspace, workspace_bytes, stream, nullptr, 0, 0, 0);
}

int fa_fwd_splitkv_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int* block_table, void* out, float* lse, int B, int Hq, int Hkv,
                         int Sq, int Skv, int d, int block_size, int num_blocks, int max_blocks,
                         int causal, float scale, int dtype, int n_splits, void* workspace,
                         size_t workspace_bytes, fa_stream_t stream) {
  int rc = check_common(B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype);
  if (rc != FA_OK) return rc;
  if (dtype == FA_F32) return FA_ERR_DTYPE;   // the paged path runs on the tensor cores only
  if (n_splits < 0 || (Hq / Hkv) * Sq > kDecodeMaxRows) return FA_ERR_SHAPE;
  if (block_size < 16 || block_size > 1024 || (block_size & (block_size - 1)) != 0 ||
      num_blocks < 1 || static_cast<long long>(num_blocks) * Hkv > (1LL << 30) ||
      max_blocks < (Skv + block_size - 1) / block_size)
    return FA_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !block_table || !out || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(lse) || (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
    return FA_ERR_ALIGN;
  return splitkv_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype,
                      n_splits, workspace, workspace_bytes, stream, block_table, block_size,
                      max_blocks, num_blocks);
}

int fa_last_device_status(fa_stream_t stream, int* status) {
  if (!status) return FA_ERR_NULL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int value = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbolAsync(&value, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FA_ERR_CUDA;
  *status = value;
  return FA_OK;
}

}  // extern "C"
