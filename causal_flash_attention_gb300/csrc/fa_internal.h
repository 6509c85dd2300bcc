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

struct FwdParams {
  CUtensorMap tm_q;   // [B*Hq][S][d], box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;   // [B*Hkv][S][d]
  CUtensorMap tm_v;   // [B*Hkv][S][d]
  void* out;          // [B*Hq][S][d], same dtype as q
  float* lse;         // [B*Hq][S], natural log
  int B, Hq, Hkv, S;
  int causal;
  float scale_log2;   // softmax scale * log2(e)
  int n_qpairs;       // ceil(S / 256): CTAs per (batch, query head)
  int* status;        // device status word (wait timeouts)
  unsigned long long* trace;   // timeline buffer of trace builds (FA_TRACE); else null
};

struct BwdPreParams {
  const void* out;    // [B*Hq][S][d]
  const void* dout;   // [B*Hq][S][d]
  const float* lse;   // [B*Hq][S]
  float* delta;       // [B*Hq][S_pad]   D_i = <dO_i, O_i>, 0 on padding rows
  float* lse2;        // [B*Hq][S_pad]   LSE_i * log2(e), +inf on padding rows
  float* dq_acc;      // [B*Hq][S_pad][d] fp32, zeroed here
  int BH, S, S_pad, d;
  int dtype;
};

struct BwdParams {
  CUtensorMap tm_q;   // [B*Hq][S][d]
  CUtensorMap tm_k;   // [B*Hkv][S][d]
  CUtensorMap tm_v;   // [B*Hkv][S][d]
  CUtensorMap tm_do;  // [B*Hq][S][d]
  const float* delta; // [B*Hq][S_pad]
  const float* lse2;  // [B*Hq][S_pad]
  float* dq_acc;      // [B*Hq][S_pad][d]
  void* dk;           // [B*Hkv][S][d]
  void* dv;           // [B*Hkv][S][d]
  int B, Hq, Hkv, S, S_pad;
  int causal;
  float scale;        // softmax scale
  float scale_log2;   // softmax scale * log2(e)
  int n_kv_tiles;     // ceil(S / 128)
  int* status;
  unsigned long long* trace;   // timeline buffer of trace builds (FA_TRACE); else null
};

struct DqConvertParams {
  const float* dq_acc;  // [B*Hq][S_pad][d]
  void* dq;             // [B*Hq][S][d]
  int BH, S, S_pad, d;
  float scale;
  int dtype;
};

// Plain fp32 (SIMT) kernels for fp32 inputs.
struct SimtParams {
  const float *q, *k, *v, *out, *dout, *lse;
  float *o_out, *lse_out, *dq, *dk, *dv;
  const float* delta;
  int B, Hq, Hkv, S, d;
  int causal;
  float scale;
};

// Launchers; each returns a cudaError_t from the launch.
cudaError_t launch_fwd_tc(const FwdParams& p, int d, bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_tc(const BwdParams& p, int d, bool bf16, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream);
cudaError_t launch_fwd_simt(const SimtParams& p, cudaStream_t stream);
cudaError_t launch_bwd_simt(const SimtParams& p, cudaStream_t stream);

}  // namespace fa
