// Internal interface of the split-KV forward for few query rows per head
// (decode): parameters shared by the C-ABI entry point (fa_api.cu) and the
// kernels (fa_decode.cu). Not installed.
#pragma once

#include "fa_internal.h"

namespace fa {

// One CTA per (key-tile range `split`, batch, key/value head); its 128-row
// query tile packs the R = G * Sq query rows of the head's G query heads
// (row r = gq * Sq + s for query head kvh * G + gq and query row s).
struct DecodeParams {
  CUtensorMap tm_k;   // [B*Hkv][Skv][d], box (64, 128, 1), 128B swizzle
  CUtensorMap tm_v;
  const void* q;      // [B*Hq][Sq][d]
  void* out;          // [B*Hq][Sq][d]   written when n_splits == 1
  float* lse;         // [B*Hq][Sq]      written when n_splits == 1
  float* part_out;    // [B*Hkv][n_splits][R][d] fp32 per-split out = O / l
  float* part_lse2;   // [B*Hkv][n_splits][R]    per-split log2-sum-exp2 of scaled scores
  int B, Hq, Hkv, Sq, Skv, kv_offset, causal;
  int G, R;
  int n_kv_tiles;     // ceil(Skv / 128)
  int tiles_per_split, n_splits;
  float scale_log2;   // softmax scale * log2(e)
  int* status;
};

struct DecodeMergeParams {
  const float* part_out;
  const float* part_lse2;
  void* out;          // [B*Hq][Sq][d]
  float* lse;         // [B*Hq][Sq], natural log
  int B, Hq, Hkv, Sq, G, R, d, n_splits, dtype;
};

cudaError_t launch_decode(const DecodeParams& p, int d, bool bf16, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecodeMergeParams& p, cudaStream_t stream);

}  // namespace fa
