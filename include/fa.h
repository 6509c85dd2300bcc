/*
 * fa.h — C ABI of libfa: causal scaled-dot-product flash attention, forward
 * and backward, on one NVIDIA GB300 (sm_103a).
 *
 * What is computed. For every batch b and query head h (key/value head
 * g = h / (Hq / Hkv), grouped-query attention as in "Phase 14: Flash
 * Attention 2 for SM120", section GQA 支持):
 *
 *   s_ij   = scale * <Q[b,h,i,:], K[b,g,j,:]>,  s_ij = -inf for j > i if causal
 *   P_ij   = exp(s_ij - LSE_i),   LSE_i = log(sum_j exp(s_ij))   (natural log)
 *   out_i  = sum_j P_ij V[b,g,j,:]
 *
 * ("Phase T14: 融合 Flash-Attention Kernel", section 什么是 flash-attention,
 * and its Key Design Decisions item 2: the forward keeps only LSE per row).
 * The backward recomputes P from Q, K, V and LSE, forms D_i = <dO_i, out_i>
 * (item 3 of the same section) and
 *
 *   dP_ij = <dO_i, V_j>,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij K_j,  dK_j = scale * sum_i dS_ij Q_i,
 *   dV_j  = sum_i P_ij dO_i
 *
 * with dK, dV of a key/value head summed over its Hq/Hkv query heads. No S x S
 * matrix is ever stored.
 *
 * Layout. Every tensor is a dense, contiguous array in device memory:
 *   q, out, dout, dq : [B][Hq][S][d]      k, v, dk, dv : [B][Hkv][S][d]
 *   lse              : [B][Hq][S]  float32
 * Element type of q/k/v/out/dout/dq/dk/dv is `dtype` (FA_F32, FA_F16 or
 * FA_BF16). d must be 64 or 128. Every pointer must be 16-byte aligned.
 *
 * Precision. FA_BF16 / FA_F16 run on the tensor cores with fp32 accumulation;
 * P is rounded to the input type before it multiplies V (and dS before it
 * multiplies Q and K). FA_F32 runs on plain fp32 arithmetic.
 *
 * Ownership and execution. The caller owns every buffer; the library keeps no
 * pointer after a call returns and allocates no device memory. Calls are
 * asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream) and
 * run on the current CUDA device, which must be the stream's device. Outputs
 * are overwritten, never accumulated into. Calls that share output or
 * workspace buffers must be ordered by the caller.
 *
 * Errors. Functions return FA_OK (0) or a negative FA_ERR_* code. Argument
 * errors are detected on the host before anything is enqueued, so a call that
 * returns an argument error has written nothing. FA_ERR_CUDA means a CUDA
 * runtime call or a kernel launch failed (the CUDA error is left for
 * cudaGetLastError to report). A kernel that gives up an internal wait (it
 * never should) sets a device status word instead of hanging; read it with
 * fa_last_device_status.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

enum {
  FA_OK = 0,
  FA_ERR_SHAPE = -1,        /* B, Hq, Hkv, S < 1, Hq % Hkv != 0, d not 64/128, causal with
                               Skv < Sq (fa_*_kv), or too large */
  FA_ERR_DTYPE = -2,        /* dtype not one of fa_dtype */
  FA_ERR_NULL = -3,         /* a required pointer is NULL */
  FA_ERR_ALIGN = -4,        /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = -5,    /* workspace NULL or smaller than fa_bwd_workspace_bytes */
  FA_ERR_CUDA = -6,         /* a CUDA runtime call or kernel launch failed */
  FA_ERR_SCALE = -7,        /* scale not finite and > 0 */
  FA_ERR_TMA = -8,          /* the driver rejected a tensor-memory-access descriptor */
  FA_ERR_NOALLOC_LIMIT = -9 /* fa_bwd_noalloc: sizes need more than FA_NOALLOC_SCRATCH_BYTES */
};

/*
 * Forward pass. Writes out[B][Hq][S][d] (dtype) and lse[B][Hq][S] (float32,
 * natural-log logsumexp of the scaled, masked score row). causal != 0 masks
 * key positions j > i. scale is usually 1/sqrt(d).
 *
 * For FA_BF16 / FA_F16 at d = 128 the forward (here and in fa_fwd_kv) runs
 * either a single-CTA kernel (the default) or a CTA-pair kernel on the
 * tensor cores' 2-CTA mode ("Phase 14: Flash Attention 2 for SM120", section
 * 硬件约束); both write the same bits. The environment variable
 * FA_FWD_CTA_PAIR, read at every call, selects the pair kernel when it is "1"
 * and the single-CTA kernel when it is "0". The single-CTA kernel gives each
 * CTA one 128-row query tile (two CTAs share an SM) at d = 64 and, at
 * d = 128, when the grid has at least four such CTAs per SM, else two tiles;
 * FA_FWD_TILES ("1" or "2", read at every call) forces one form. All forms
 * write the same bits.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
           int B, int Hq, int Hkv, int S, int d, int causal, float scale,
           int dtype, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes (the same for every
 * dtype): an fp32 dQ accumulator [B][Hq][S128][d], D and LSE*log2(e) rows
 * [B][Hq][S128] each, where S128 = S rounded up to a multiple of 128, each
 * region starting on a 256-byte boundary, then 256 bytes holding the
 * counter from which the main kernel's CTAs claim work items. Returns 0 for
 * invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int S, int d);

/*
 * Backward pass. Inputs: q, k, v, out and lse from fa_fwd with the same
 * arguments, dout = dL/dout. Writes dq [B][Hq][S][d], dk and dv [B][Hkv][S][d]
 * (dtype). `workspace` is caller-owned device memory of at least
 * fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) bytes, 256-byte aligned; its
 * contents on entry do not matter and are clobbered.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* out,
           const void* dout, const float* lse, void* dq, void* dk, void* dv,
           int B, int Hq, int Hkv, int S, int d, int causal, float scale,
           int dtype, void* workspace, size_t workspace_bytes,
           fa_stream_t stream);

/*
 * Separate query and key/value lengths: Sq query rows against Skv key/value
 * rows, for a chunk of queries at the end of a longer context (chunked
 * prefill, a few new tokens against a KV cache) or, without the mask, any two
 * lengths. Layout:
 *   q, out, dout, dq : [B][Hq][Sq][d]     k, v, dk, dv : [B][Hkv][Skv][d]
 *   lse              : [B][Hq][Sq]  float32
 * With causal != 0, query row i stands at sequence position i + kv_offset,
 * kv_offset = Skv - Sq, and key j is masked when j > i + kv_offset ("Phase 14:
 * Flash Attention 2 for SM120", section Causal Mask: kv_offset = kv_len -
 * q_len, for a KV cache longer than Q). Causal calls need Skv >= Sq, else
 * FA_ERR_SHAPE (rows with no visible key have no softmax). Everything else
 * (dtypes, d, alignment, ownership, errors, asynchrony) is as for fa_fwd and
 * fa_bwd, which are these calls with Sq = Skv = S.
 */
int fa_fwd_kv(const void* q, const void* k, const void* v, void* out, float* lse,
              int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
              float scale, int dtype, fa_stream_t stream);

/* Workspace bytes of fa_bwd_kv: as fa_bwd_workspace_bytes, sized by Sq (the
 * dQ accumulator and the per-row D and LSE have one row per query). Returns 0
 * for invalid sizes. */
size_t fa_bwd_kv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d);

int fa_bwd_kv(const void* q, const void* k, const void* v, const void* out,
              const void* dout, const float* lse, void* dq, void* dk, void* dv,
              int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
              float scale, int dtype, void* workspace, size_t workspace_bytes,
              fa_stream_t stream);

/*
 * Split-KV forward for few query rows per head: decode (one or a few new
 * tokens, Sq small, against a long key/value cache Skv). Same arguments,
 * layouts, mask (kv_offset = Skv - Sq under causal) and results as fa_fwd_kv;
 * only the work layout differs. The G = Hq / Hkv query heads of a key/value
 * head are packed into one 128-row tile, so G * Sq must be at most 128
 * (else FA_ERR_SHAPE); the key/value sequence of each (batch, key/value head)
 * is cut into n_splits ranges of whole 128-key tiles processed in parallel,
 * each producing a partial out and log-sum-exp, which a second kernel merges
 * ("Phase 14: Flash Attention 2 for SM120", section 已知局限与后续优化方向,
 * item 1: a dedicated decode kernel that reduces in parallel along the
 * key/value dimension).
 *
 * n_splits: 0 = automatic (the largest count that keeps all B * Hkv * n_splits
 * CTAs in one wave on the GPU's 152 SMs, at least 1); otherwise the requested
 * number of ranges, reduced so that no range is empty (at most ceil(Skv/128)).
 * workspace: caller-owned device memory of at least
 * fa_fwd_splitkv_workspace_bytes(...) bytes, 256-byte aligned, for the
 * per-range partial results (fp32); it may be NULL when that size is 0 (one
 * range). FA_F32 inputs take the fa_fwd_kv path (no split, no workspace).
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* out, float* lse,
                   int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                   float scale, int dtype, int n_splits, void* workspace,
                   size_t workspace_bytes, fa_stream_t stream);

/* Workspace bytes of fa_fwd_splitkv for these sizes and n_splits (0 =
 * automatic): B * Hkv * ranges * G * Sq rows of d + 1 floats, each region
 * 256-byte aligned; 0 when one range suffices, and 0 for invalid sizes (the
 * call reports those). */
size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                      int n_splits);

/*
 * fa_fwd_splitkv over a paged key/value cache: the keys and values of all
 * sequences live in fixed-size blocks of a shared pool, and a block table maps
 * each sequence's logical blocks to physical ones ("FlashAttention 与 SDPA
 * Backend", section 与 PagedAttention、KV Cache 的组合: a paged decode kernel
 * looks up the block table while it loads the K/V tiles and runs the online
 * softmax). Layouts:
 *   k_cache, v_cache : [num_blocks][Hkv][block_size][d]   (dtype)
 *   block_table      : [B][max_blocks] int32; key position t of sequence b is
 *                      row t % block_size of block block_table[b][t / block_size]
 * block_size: a power of two from 16 to 1024. Only the first
 * ceil(Skv / block_size) entries of a row are read (max_blocks must be at
 * least that); an entry outside [0, num_blocks) reads as zeros instead of
 * faulting. Every sequence has the same Skv. q, out, lse, the mask, the
 * results, n_splits and the workspace (fa_fwd_splitkv_workspace_bytes) are as
 * for fa_fwd_splitkv. FA_BF16 and FA_F16 only (FA_F32 gives FA_ERR_DTYPE).
 */
int fa_fwd_splitkv_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int* block_table, void* out, float* lse,
                         int B, int Hq, int Hkv, int Sq, int Skv, int d,
                         int block_size, int num_blocks, int max_blocks, int causal,
                         float scale, int dtype, int n_splits, void* workspace,
                         size_t workspace_bytes, fa_stream_t stream);

/*
 * Size of the fixed device scratch array behind fa_bwd_noalloc (32 MiB). A
 * call fits when fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) is at most this,
 * e.g. B*Hq = 96 heads at S = 1024, d = 64 (about 25.9 MB). The limit uses
 * that one size for every dtype, although FA_F32 calls use only the D and
 * LSE rows of it.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * Backward pass for callers that cannot allocate device memory (for example
 * code inside a framework or plugin callback that owns every device
 * allocation, or latency-critical code that must not call cudaMalloc/cudaFree
 * because they can synchronize the device). Same arguments and results as
 * fa_bwd, without the workspace: the scratch is a fixed
 * FA_NOALLOC_SCRATCH_BYTES array in the library's device memory, held on every
 * GPU that loads the library until the process exits. The call allocates
 * nothing. This entry point has no counterpart in the method's description;
 * it is a deployment aid.
 *
 * Errors: first fa_bwd's argument errors (FA_ERR_SHAPE, FA_ERR_DTYPE,
 * FA_ERR_SCALE, FA_ERR_NULL, FA_ERR_ALIGN), then FA_ERR_NOALLOC_LIMIT when
 * the sizes need more scratch than FA_NOALLOC_SCRATCH_BYTES; either way
 * nothing is enqueued and the scratch array is not looked up.
 *
 * Device and set-up: the array used is the current device's, so the current
 * device must be the one that owns `stream` and every pointer. The first call
 * that passes the checks with a given device current looks up the array's
 * device address on that device; make that first call before any stream
 * capture.
 *
 * Sharing: every call shares the one array and it keeps the last call's
 * contents (each call rewrites all of it that it reads, so results do not
 * depend on them). Calls whose work overlaps on the GPU (unordered streams,
 * concurrent host threads) race on the array: the caller must order them.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv,
                   int B, int Hq, int Hkv, int S, int d, int causal, float scale,
                   int dtype, fa_stream_t stream);

/* Static description of an FA_* code. */
const char* fa_strerror(int code);

/*
 * Waits for `stream`, then reads and clears the device status word of the
 * current device: 0 when no kernel has given up a wait since the last read,
 * else a bit mask (1 = an mbarrier wait ran past its limit). Returns FA_OK or
 * FA_ERR_CUDA.
 */
int fa_last_device_status(fa_stream_t stream, int* status);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
