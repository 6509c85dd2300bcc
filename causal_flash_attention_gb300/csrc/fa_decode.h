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
  CUtensorMap tm_k;   // contiguous: [B*Hkv][Skv][d], box (64, 128, 1), 128B swizzle;
  CUtensorMap tm_v;   // paged: [num_blocks*Hkv][block_size][d], box (64, box_rows, 1)
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
  // Paged key/value cache (block_table != nullptr): key position t of batch b
  // is row t % block_size of physical block block_table[b * max_blocks +
  // t / block_size]; a 128-key tile is loaded as 128 / box_rows boxes
  // (box_rows = min(block_size, 128)).
  const int* block_table;
  int block_size, box_rows, max_blocks, num_blocks;
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
