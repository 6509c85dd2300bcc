// Internal interface between the C-ABI entry points (fa_api.cu) and the
// kernel launchers (fa_fwd.cu, fa_bwd.cu, fa_simt.cu). Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Tile geometry shared by the tensor-core kernels: 128 query rows per tile,
// 128 key/value rows per tile, 64-element (128-byte) column chunks.
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kChunk = 64;

// Sequence lengths: Sq query rows, Skv key/value rows (equal for
// self-attention). Under the causal mask query row i stands at position
// i + kv_offset, kv_offset = Skv - Sq >= 0 (0 without the mask).
struct FwdParams {
  CUtensorMap tm_q;   // [B*Hq][Sq][d], box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;   // [B*Hkv][Skv][d]
  CUtensorMap tm_v;   // [B*Hkv][Skv][d]
  void* out;          // [B*Hq][Sq][d], same dtype as q
  float* lse;         // [B*Hq][Sq], natural log
  int B, Hq, Hkv, Sq, Skv, kv_offset;
  int causal;
  float scale_log2;   // softmax scale * log2(e)
  int n_units;        // CTAs per (batch, query head): ceil(Sq / (128 T)) for T query
                      // tiles per CTA (set by the forward's launcher)
  int kv_tiles_ahead; // 1 + ceil(kv_offset / 128): key tiles a full causal
                      // query tile qt walks is qt + kv_tiles_ahead
  int* status;        // device status word (wait timeouts)
  unsigned long long* trace;   // timeline buffer of trace builds (FA_TRACE); else null
  // CTA-pair forward (d = 128) only:
  CUtensorMap tm_k_half;   // k as tm_k with a box of 64 rows: each CTA of a pair loads half a tile
  int n_qblocks;           // ceil(Sq / 512): CTA pairs per (batch, query head)
};

struct BwdPreParams {
  const void* out;    // [B*Hq][Sq][d]
  const void* dout;   // [B*Hq][Sq][d]
  const float* lse;   // [B*Hq][Sq]
  float* delta;       // [B*Hq][Sq_pad]   D_i = <dO_i, O_i>, 0 on padding rows
  float* lse2;        // [B*Hq][Sq_pad]   LSE_i * log2(e), +inf on padding rows
  float* dq_acc;      // [B*Hq][Sq_pad][d] fp32, zeroed here
  int* work;          // the main kernel's work-item counter, zeroed here (null: none)
  int BH, Sq, Sq_pad, d;
  int dtype;
};

struct BwdParams {
  CUtensorMap tm_q;   // [B*Hq][Sq][d]
  CUtensorMap tm_k;   // [B*Hkv][Skv][d]
  CUtensorMap tm_v;   // [B*Hkv][Skv][d]
  CUtensorMap tm_do;  // [B*Hq][Sq][d]
  CUtensorMap tm_dq;  // dq_acc as fp32 [B*Hq][Sq_pad][d], box (32, 32, 1), 128B swizzle
  CUtensorMap tm_dk;  // dk [B*Hkv][Skv][d], box (64, 32, 1), 128B swizzle (stores)
  CUtensorMap tm_dv;  // dv, as tm_dk
  const float* delta; // [B*Hq][Sq_pad]
  const float* lse2;  // [B*Hq][Sq_pad]
  float* dq_acc;      // [B*Hq][Sq_pad][d]
  void* dk;           // [B*Hkv][Skv][d]
  void* dv;           // [B*Hkv][Skv][d]
  int* work;          // work-item counter, zeroed by the pre-pass
  int B, Hq, Hkv, Sq, Skv, Sq_pad, kv_offset;
  int causal;
  float scale;        // softmax scale
  float scale_log2;   // softmax scale * log2(e)
  int n_kv_tiles;     // ceil(Skv / 128): work items per (batch, key/value head)
  int n_q_tiles;      // ceil(Sq / 128)
  int* status;
  unsigned long long* trace;   // timeline buffer of trace builds (FA_TRACE); else null
};

struct DqConvertParams {
  const float* dq_acc;  // [B*Hq][Sq_pad][d]
  void* dq;             // [B*Hq][Sq][d]
  int BH, Sq, Sq_pad, d;
  float scale;
  int dtype;
};

// Plain fp32 (SIMT) kernels for fp32 inputs.
struct SimtParams {
  const float *q, *k, *v, *out, *dout, *lse;
  float *o_out, *lse_out, *dq, *dk, *dv;
  const float* delta;   // [B*Hq][Sq_pad]
  int B, Hq, Hkv, Sq, Skv, kv_offset, d;
  int causal;
  float scale;
};

// Host-side argument checks of the backward entry points (shapes, dtype,
// scale, null and 16-byte alignment of every pointer); FA_OK or an FA_ERR_*
// code. Defined in fa_api.cu.
int check_bwd_args(const void* q, const void* k, const void* v, const void* out,
                   const void* dout, const float* lse, const void* dq, const void* dk,
                   const void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                   float scale, int dtype);

// Launchers; each returns a cudaError_t from the launch.
cudaError_t launch_fwd_tc(const FwdParams& p, int d, bool bf16, cudaStream_t stream);
cudaError_t launch_fwd_pair(const FwdParams& p, bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_tc(const BwdParams& p, int d, bool bf16, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream);
cudaError_t launch_fwd_simt(const SimtParams& p, cudaStream_t stream);
cudaError_t launch_bwd_simt(const SimtParams& p, cudaStream_t stream);

}  // namespace fa
