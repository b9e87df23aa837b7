/*
 * fa.h -- C-ABI of libfa.so: exact scaled-dot-product attention on one
 * GB300 (sm_103a): forward and backward, dense, causal, key-padded,
 * block-sparse and with fused dropout.
 *
 * What is computed (per batch b and head h; Q, K, V, dO in R^{N x d}):
 *   S = scale * Q K^T + M,  P = softmax(S) row-wise,  O = P V,
 *   LSE_i = ln sum_j exp(S_ij)  (natural log, scale included).
 * This is standard attention as stated in the condensed FlashAttention paper
 * (sample_paper.md, section 2 "Background"; shapes "Q: N x d, K^T: d x N,
 * QK^T: N x N, sm(QK^T)V: N x d" in the aggregator page's figure captions).
 * The kernels tile Q, K, V through on-chip memory and rescale the softmax
 * incrementally, so S and P never reach HBM (sample_paper.md section 3,
 * "Tiling" and "Softmax rescaling / recomputation"; Figure 1 of the Medium
 * article "No More Quadratic Complexity for Transformers"). The result is
 * exact up to floating-point rounding.
 *
 * Conventions common to every entry point
 *   - Tensors are DEVICE pointers, row-major [B, H, N, d] with d fastest and
 *     no padding between rows or heads. q, k, v, o, dout, dq, dk, dv are bf16
 *     (passed as void*); lse is fp32 [B, H, N].
 *   - Base addresses must be 16-byte aligned. d must be 64 or 128. Any N >= 1.
 *   - The mask M_ij is 0 or -inf: causal keeps j <= i; kv_len (optional) keeps
 *     j < kv_len[b] for every query row of batch b; a block mask keeps whole
 *     128 x 128 blocks. A query row that sees no key gets O = 0 and
 *     LSE = -inf (and zero gradients).
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Outputs are valid once the stream is synchronised. Inputs are only read.
 *   - Ownership: the caller owns every buffer. The library never allocates or
 *     frees device memory; the backward pass takes a caller-provided
 *     workspace whose size is linear in N (fa_bwd_workspace_bytes).
 *   - Errors: arguments are validated before anything is launched and
 *     nothing is written on error. FA_ERR_INVALID_ARG: a NULL pointer, B, H
 *     or N < 1, non-finite scale, a misaligned base address, an output that
 *     shares an element with an input or with another output, or a workspace
 *     that is too small. [B, H, N, d] tensors of one call are compared element
 *     by element, so views that interleave in one buffer without sharing an
 *     element (q, k, v or dq, dk, dv of a packed [B, N, 3, H, d] tensor) are
 *     accepted; lse and workspaces by address range. FA_ERR_UNSUPPORTED:
 *     d not in {64, 128}, block_size != 128, or a device that is not sm_103.
 *     FA_ERR_CUDA: a CUDA call or launch failed. FA_ERR_DEVICE_TIMEOUT is
 *     reported by fa_device_status() when a bounded device-side wait expired.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_DEVICE_TIMEOUT = 4,
  FA_ERR_DEVICE_CHECK = 5  /* checked builds only: a device-side bounds / alignment check failed */
} fa_status;

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

/* Forward pass: O = softmax(scale * Q K^T [+ causal mask]) V and the per-row
 * logsumexp LSE that the backward pass recomputes P from (sample_paper.md
 * section 3: tiling, online softmax rescaling, "stored statistics").
 *   q, k, v : bf16 [B,H,N,d] inputs;  o : bf16 [B,H,N,d] output;
 *   lse     : fp32 [B,H,N] output;    causal : 0 or 1;  scale : finite. */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, struct CUstream_st* stream);

/* Forward pass with key padding: as fa_fwd, and keys j >= kv_len[b] are
 * masked for every query row of batch b. kv_len is a DEVICE int32 [B]
 * (values are clamped to [0, N] on the device) or NULL for no padding. */
int fa_fwd_kpad(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, int causal, float scale, const int32_t* kv_len,
                struct CUstream_st* stream);

/* Forward pass that may spread its last wave of work over every SM. The
 * forward's work items are pairs of 128-row Q tiles; when their number is
 * not a multiple of the SM count, the last round keeps only part of the GPU
 * busy. Given a workspace, the items of that last round are cut into equal
 * runs of K/V tiles, one run per SM (a stream-K schedule); each cut item's
 * parts leave their unnormalised O and per-row running maximum and sum in
 * the workspace, and a second kernel merges them with the same rescaling the
 * online softmax applies from one K/V block to the next (condensed paper
 * sample_paper.md section 3, "Softmax rescaling"). The pages themselves do
 * not split the key range; this is a scheduling choice for small B*H or
 * short sequences on a 152-SM GPU, and the result is the same attention.
 *   fa_fwd_workspace_bytes: bytes of workspace with which fa_fwd_split (and
 *     fa_attention_fwd_split) split these sizes on the current device; 0
 *     when a split would not shorten the pass (then no workspace is needed).
 *     Also 0 for invalid sizes.
 *   fa_fwd_split: as fa_fwd_kpad, plus `workspace` (DEVICE, 16-byte aligned,
 *     at least fa_fwd_workspace_bytes bytes, contents ignored; NULL with
 *     workspace_bytes = 0 allowed). With a smaller or NULL workspace, with
 *     kv_len != NULL, or when the split would not help, it runs exactly as
 *     fa_fwd_kpad. The workspace must not overlap any tensor of the call.
 *     Two calls that share a workspace must be ordered on the GPU. */
size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal);
int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, const int32_t* kv_len, void* workspace,
                 size_t workspace_bytes, struct CUstream_st* stream);

/* Bytes of workspace fa_bwd needs: an fp32 dQ accumulator plus two fp32
 * per-row vectors (log2-scaled LSE and D = rowsum(dO * O)), each padded to a
 * multiple of 128 rows per head. Linear in N (sample_paper.md section 4:
 * memory linear in sequence length). Returns 0 for invalid sizes. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/* Bytes of backward workspace with which the backward calls (fa_bwd,
 * fa_bwd_main, fa_dropout_bwd, fa_attention_bwd) spread their last wave of
 * work over every SM, as fa_fwd_split does for the forward: the key-tile
 * items of the last round are cut into equal runs of Q tiles, each part
 * adds its dQ into the accumulator as usual and leaves its dK, dV in the
 * workspace, and a short kernel after the main kernel sums the parts. It is
 * fa_bwd_workspace_bytes plus the parts' area when these sizes gain from the
 * split on the current device, else fa_bwd_workspace_bytes. A workspace of
 * at least this size enables the split; one of at least
 * fa_bwd_workspace_bytes still works, without it. No split with kv_len or a
 * block mask. 0 for invalid sizes. */
size_t fa_bwd_split_workspace_bytes(int B, int H, int N, int d, int causal);

/* Backward pass: gradients of L = sum(dO * O) with respect to Q, K, V. P is
 * recomputed on chip from Q, K and the forward's LSE instead of being read
 * from HBM (sample_paper.md section 3, "in the backward pass, the attention
 * matrix is recomputed on-chip from stored statistics").
 *   q, k, v, o, dout : bf16 [B,H,N,d] (o and lse from fa_fwd / fa_fwd_kpad
 *                      with the same causal, scale and kv_len);
 *   lse              : fp32 [B,H,N];
 *   dq, dk, dv       : bf16 [B,H,N,d] outputs;
 *   kv_len           : DEVICE int32 [B] or NULL (as in fa_fwd_kpad);
 *   workspace        : DEVICE scratch of at least fa_bwd_workspace_bytes,
 *                      16-byte aligned; its contents on entry are ignored.
 *                      With fa_bwd_split_workspace_bytes or more, the last
 *                      wave of work is split over every SM (see there). */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
           float scale, const int32_t* kv_len, void* workspace, size_t workspace_bytes,
           struct CUstream_st* stream);

/* The three stages of fa_bwd as separate calls, for callers that schedule
 * or time them individually. fa_bwd(...) is exactly fa_bwd_preprocess,
 * fa_bwd_main, fa_bwd_dq_convert on the same stream with the same sizes and
 * workspace. Arguments mean what they mean for fa_bwd; a stage reads only the
 * pointers it takes.
 *   fa_bwd_preprocess: D = rowsum(dO * O), LSE in log2 units, and a zeroed
 *     fp32 dQ accumulator, all written into the workspace.
 *   fa_bwd_main: recomputes P tile by tile and writes dK, dV; adds dQ into
 *     the workspace accumulator. Needs the workspace prepared by
 *     fa_bwd_preprocess for the same (B, H, N, d) and LSE.
 *   fa_bwd_dq_convert: dq (bf16) = the workspace accumulator. */
int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int N,
                      int d, void* workspace, size_t workspace_bytes, struct CUstream_st* stream);
int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                int B, int H, int N, int d, int causal, float scale, const int32_t* kv_len,
                void* workspace, size_t workspace_bytes, struct CUstream_st* stream);
int fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, void* workspace,
                      size_t workspace_bytes, struct CUstream_st* stream);

/* Backward pass for callers that cannot allocate device memory. There is no
 * counterpart of this call in the method's papers: it exists because some
 * callers of a kernel library may not call cudaMalloc -- a CUDA-graph
 * capture that must not allocate, a framework that routes every allocation
 * through its own pool, a plugin that receives tensors but no allocator --
 * and fa_bwd needs a workspace.
 *
 * Same arguments and results as fa_bwd, minus the workspace: the library
 * uses its own static device buffer of FA_NOALLOC_SCRATCH_BYTES (64 MiB),
 * which every GPU that loads libfa.so holds until the process exits. The
 * caller still passes every input and output. Nothing is allocated or freed.
 *   - Limit: the call returns FA_ERR_INVALID_ARG, without launching, when
 *     fa_bwd_workspace_bytes(B, H, N, d) > FA_NOALLOC_SCRATCH_BYTES, i.e.
 *     when B*H*Npad (Npad = N rounded up to a multiple of 128) exceeds
 *     254,080 rows at d = 64 or 129,024 rows at d = 128. NULL tensors are
 *     rejected the same way, before the device is touched.
 *   - Set-up: the first call on each device, with that device current, looks
 *     up the buffer's device address (cudaGetSymbolAddress). Make that first
 *     call before any stream capture on that device.
 *   - Sharing: all calls on a device share the one buffer, and it keeps the
 *     last call's contents; each call re-initialises what it reads. Calls
 *     whose kernels overlap on the GPU (different streams without ordering
 *     between them) race on the buffer and give wrong results. */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, const int32_t* kv_len, struct CUstream_st* stream);

/* Block-sparse forward: fa_fwd (non-causal) where query block r attends only
 * to key blocks c with block_mask[r * nb + c] != 0, nb = ceil(N / 128); the
 * masked blocks are -inf and are skipped entirely, so IO and work fall in
 * proportion to the sparsity (FlashAttention abstract, "block-sparse
 * attention"; aggregator page, "IO complexity smaller ... proportional to the
 * sparsity"). block_mask is a DEVICE uint8 [nb, nb] shared by all (b, h);
 * block_size must be 128. */
int fa_blocksparse_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, const uint8_t* block_mask, int block_size,
                       struct CUstream_st* stream);

/* Backward pass of the block-sparse forward (fa_blocksparse_fwd): dQ, dK, dV
 * of L = sum(dO * O) when attention is restricted to the kept 128 x 128
 * blocks. Masked blocks contribute nothing, so the recomputation and the five
 * products run only over kept blocks (condensed paper sample_paper.md,
 * section 4: block-sparse FlashAttention, IO proportional to the sparsity).
 *   q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes : as fa_bwd
 *                 (o and lse from fa_blocksparse_fwd with the same mask and scale);
 *   block_mask  : as fa_blocksparse_fwd (DEVICE uint8 [nb][nb], nonzero = kept);
 *   block_size  : must be 128 (else FA_ERR_UNSUPPORTED).
 * Key tiles kept by no query tile get dK = dV = 0; query rows of a tile that
 * keeps no key tile get dQ = 0. Errors as fa_bwd. */
int fa_blocksparse_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, const uint8_t* block_mask, int block_size,
                       void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/* Attention with fused dropout on P (inverted dropout): O = (P * Z / (1 - p')) V
 * with Z_ij in {0, 1}, LSE that of the undropped scores. Dropout is one of the
 * stages that the method fuses into its single kernel, at no extra memory
 * (FlashAttention aggregator page, GPT-2 time-breakdown figure); the keep
 * decisions are drawn on chip and never stored, and the backward pass draws
 * them again from the same indices.
 *   Draws: Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as
 *   1, 2, 3", SC'11) with key (seed mod 2^32, seed div 2^32). Element
 *   (b, h, i, j) uses byte j mod 16 (byte j mod 4 of word (j mod 16) / 4,
 *   little-endian) of the block at counter (j / 16, i, b*H + h, offset), and
 *   is kept iff that byte >= t, t = round(256 * dropout_p) capped at 255, so
 *   the drop probability is p' = t / 256 and kept entries are scaled by
 *   256 / (256 - t). Use a new (seed, offset) pair for every call whose mask
 *   must be independent of earlier ones.
 *   dropout_p : in [0, 1) (else FA_ERR_INVALID_ARG); 0 gives fa_fwd's result.
 * Other arguments, layouts and errors: as fa_fwd_kpad (kv_len may be NULL). */
int fa_dropout_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, int causal, float scale, const int32_t* kv_len,
                   float dropout_p, uint64_t seed, uint32_t offset, struct CUstream_st* stream);

/* Backward pass of fa_dropout_fwd: gradients of L = sum(dO * O) with the same
 * (dropout_p, seed, offset) -- dV = Pd^T dO with Pd = P * Z / (1 - p'), and
 * dS = P * (Z * dPd / (1 - p') - D), dPd = dO V^T, D = rowsum(dO * O).
 * Arguments, workspace and errors: as fa_bwd (o and lse from fa_dropout_fwd
 * with the same causal, scale, kv_len, dropout_p, seed and offset). */
int fa_dropout_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, const int32_t* kv_len, float dropout_p, uint64_t seed,
                   uint32_t offset, void* workspace, size_t workspace_bytes,
                   struct CUstream_st* stream);

/* The keep decisions Z of fa_dropout_fwd / fa_dropout_bwd for the same
 * (B, H, N, dropout_p, seed, offset): keep is a DEVICE uint8 [B, H, N, N]
 * (query row i, key j), 1 where the element is kept, 0 where it is dropped.
 * For inspection and tests; the attention calls never materialise it.
 * Errors: FA_ERR_INVALID_ARG for B, H or N < 1, a NULL keep or dropout_p
 * outside [0, 1). */
int fa_dropout_mask(int B, int H, int N, float dropout_p, uint64_t seed, uint32_t offset,
                    uint8_t* keep, struct CUstream_st* stream);

/* Options of fa_attention_fwd / fa_attention_bwd, the general entry points:
 * every combination of layout, causal mask, key padding, block mask and
 * dropout in one call. Zero-initialise, then set scale and what is needed.
 *   stride_b, stride_h, stride_n : element strides of the batch, head and row
 *       axes, shared by every bf16 [B, H, N, d] tensor of the call (q, k, v,
 *       o; dout, dq, dk, dv); the d axis is contiguous. All three 0 means
 *       row-major [B, H, N, d]. [B, N, H, d] storage is {N*H*d, d, H*d}.
 *       Each must be >= 0, a multiple of 8 (16 bytes) and < 2^36, and rows
 *       must not overlap: sorted by stride (axes of extent 1 excluded), the
 *       smallest is >= d and each next is >= the previous stride times that
 *       axis' extent. lse stays fp32 [B, H, N] row-major.
 *   causal       : 0 or 1 (keeps j <= i).
 *   scale        : finite, > 0.
 *   kv_len       : DEVICE int32 [B] or NULL (as fa_fwd_kpad).
 *   block_mask, block_size : as fa_blocksparse_fwd, or NULL / ignored. With
 *       causal = 1 a block is visited only if kept and not above the diagonal.
 *   dropout_p, dropout_seed, dropout_offset : as fa_dropout_fwd; dropout_p = 0
 *       means no dropout.
 * Every mask applies together (an element is kept if it passes all of them). */
typedef struct fa_attention_options {
  int64_t stride_b, stride_h, stride_n;
  int causal;
  float scale;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int block_size;
  float dropout_p;
  uint64_t dropout_seed;
  uint32_t dropout_offset;
} fa_attention_options;

/* Forward pass with options: O and LSE as fa_fwd / fa_fwd_kpad /
 * fa_blocksparse_fwd / fa_dropout_fwd, which are this call with the
 * corresponding options. Errors as those calls, plus FA_ERR_INVALID_ARG for a
 * NULL opt or strides that break the rules above. */
int fa_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, const fa_attention_options* opt,
                     struct CUstream_st* stream);

/* fa_attention_fwd with a workspace for the split of the last wave, as
 * fa_fwd_split (fa_fwd_workspace_bytes gives its size). No split with kv_len
 * or a block mask; then, or with too small a workspace, exactly
 * fa_attention_fwd. */
int fa_attention_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, const fa_attention_options* opt,
                           void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/* Backward pass of fa_attention_fwd with the same options (o and lse from
 * that call): dq, dk, dv in the same strides. Workspace and errors as fa_bwd. */
int fa_attention_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                     int H, int N, int d, const fa_attention_options* opt, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream);

/* Device-side status of the current device: FA_OK, or FA_ERR_DEVICE_TIMEOUT
 * if a bounded wait inside a kernel gave up since the last call, or (in a
 * library built with FA_CHECKS=1) FA_ERR_DEVICE_CHECK if a TMA copy failed
 * its coordinate or alignment check and was skipped. Reading
 * clears it. Call only after synchronising the streams that ran the
 * kernels. Returns FA_ERR_CUDA if the status word cannot be read. */
int fa_device_status(void);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(int status);

/* Self-test of the device watchdog: launches one CTA that waits on an
 * mbarrier nothing ever arrives on, with a budget of `limit_cycles` SM
 * cycles. The wait gives up, the kernel records FA_ERR_DEVICE_TIMEOUT and
 * returns; fa_device_status() then reports it. Nothing traps or hangs. */
int fa_selftest_wait_timeout(long long limit_cycles, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
