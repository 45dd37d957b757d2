/*
 * fa.h - exact, IO-aware attention (FlashAttention forward and recompute backward) for GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no C++ or framework types.
 *
 * The operation.  For every batch b and head h, with q_i, k_j, v_j the rows of one [N, d]
 * slice of Q, K, V:
 *     s_ij = scale * (q_i . k_j)  if allowed(i, j), else -inf
 *     O_i  = sum_j softmax_j(s_ij) v_j,     LSE_i = ln sum_j exp(s_ij)
 * ("FlashAttention：让精确注意力服从内存层次", opening formula softmax(QK^T/sqrt(d))V; the method computes the same function as standard attention,
 * "FlashAttention: Exact Attention with Less GPU Memory", section "Why the word 'exact' is in
 * the title").  The N x N score and probability matrices are computed tile by tile on chip
 * with an online softmax and never written to device memory ("FlashAttention paper story",
 * tiling and online-softmax paragraphs).  The forward keeps one statistic per row, the
 * log-sum-exp, from which the backward recomputes P ("FlashAttention paper story", backward
 * paragraph: only the softmax statistics are stored and P is rebuilt on chip).
 *
 *     allowed(i, j) = (!causal || j <= i)                      causal mask, top-left aligned
 *                  && (kv_lens == NULL || j < kv_lens[b])       key padding
 *                  && (block_mask == NULL ||
 *                      block_mask[(i / 128) * T + (j / 128)] != 0)   block-sparse tile mask
 *     with T = ceil(N / 128).  A tile whose mask entry is 0 is skipped: its K/V rows are not
 *     loaded ("FlashAttention paper story", block-sparse paragraph).
 *     A query row with no allowed key gets O_i = 0 and LSE_i = -inf; its gradients are 0.
 *
 * Layout and ownership (all calls).
 *   - Q, K, V, O, dO, dQ, dK, dV: contiguous [B, H, N, d] row-major (d innermost), in the
 *     dtype given; device memory owned by the caller; base addresses 16-byte aligned.
 *   - LSE: float32 [B, H, N], natural log.  kv_lens: int32 [B].  block_mask: uint8 [T, T],
 *     row-major, one mask for every (b, h).  All device pointers.
 *   - d must be 64 or 128.  N >= 1 (B, H or N equal to 0 is a no-op returning FA_OK).
 *   - The library allocates no device memory.  The backward's scratch (the per-row
 *     D = rowsum(dO * O), and for fa_backward_fused also an fp32 dQ accumulator) is the
 *     caller's workspace.
 *   - No call depends on process-wide state set by another call, except the two test hooks at
 *     the end of this header.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).  A
 *     return of FA_OK means the kernels were launched.  Argument errors are detected on the
 *     host before anything is launched.  No call aborts or throws.
 *   - Device-side failures (a bounded wait that ran out inside a kernel) are recorded in a
 *     per-device error word and reported by fa_check_device_status().
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
  FA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer, scale <= 0 */
  FA_ERR_UNSUPPORTED = 2,   /* head dim other than 64/128, unknown dtype, size limits */
  FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_TIMEOUT = 4        /* a kernel's bounded wait ran out (see fa_check_device_status) */
} fa_status;

typedef enum {
  FA_BF16 = 0,              /* bf16 inputs and outputs, fp32 accumulation (tcgen05 path) */
  FA_FP32 = 1,              /* fp32 inputs and outputs, fp32 CUDA-core arithmetic */
  FA_FP16 = 2               /* fp16 inputs and outputs, fp32 accumulation (tcgen05 path); P and
                               dS enter the tensor cores as fp16, so |dS| must stay < 65504 */
} fa_dtype;

/*
 * Forward pass.  Writes O [B,H,N,d] (dtype) and LSE [B,H,N] (fp32).
 *   q, k, v    : inputs, [B,H,N,d] in `dtype`
 *   o          : output, [B,H,N,d] in `dtype` (must not alias q/k/v)
 *   lse        : output, [B,H,N] fp32, ln of the softmax normaliser of each query row
 *   scale      : multiplies q.k before the softmax (1/sqrt(d) for standard attention); finite
 *                and > 0
 *   causal     : nonzero = mask keys j > i
 *   block_mask : nullable; [T,T] uint8 tile mask (0 = tile skipped); with a mask, N <= 786432
 *   kv_lens    : nullable; [B] int32 valid key count per sequence (keys j >= kv_lens[b]
 *                are masked for every query; values are clamped to [0, N])
 *   stream     : cudaStream_t to launch on
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N, int d, float scale, int causal,
                     const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                     void* stream);

/*
 * fa_forward_gqa for tile masks whose query rows have very unequal numbers of live key tiles (the
 * global rows of a local + global pattern, "FlashAttention paper story", block-sparse paragraph,
 * attend to every key tile while the others see a few).  With one CTA per 256-row pair of query
 * tiles such a pair is a chain of hundreds of tiles that outlasts all the other work.  Here a
 * plan computed on the device from the mask cuts every pair whose live key tiles exceed a target
 * length into ranges run by separate CTAs (at most 16 extra CTAs per (b, h) slice), and the range
 * that finishes last merges the ranges' partial results with the merge law of the online-softmax
 * statistics ("FlashAttention：让精确注意力服从内存层次", section "Online softmax").  The plan
 * depends only on the mask: results are the same bits on every call (they can differ from
 * fa_forward's in the last bits, the sums being grouped differently).
 *   workspace : >= fa_forward_blocksparse_workspace_size(B, H, N, d) bytes, 256-byte aligned,
 *               caller-owned, contents on entry irrelevant; calls in flight at once need their own
 *               (it holds the plan, the pairs' live-tile bitmaps, the counter from which the
 *               d = 64 kernel's persistent CTAs claim their work, and the partial results: about
 *               B*H * 32 * 256 * (d+1) * 4 bytes)
 * Without a block mask, or with fp32 inputs, this is fa_forward_gqa (the workspace is not used).
 * Other arguments, errors and ownership as in fa_forward_gqa.
 */
size_t fa_forward_blocksparse_workspace_size(int B, int H, int N, int d);
fa_status fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int N, int d, float scale, int causal,
                                 const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped-query attention (the pages list "GQA head mapping" among the semantics production use
 * needs: "FlashAttention：让精确注意力服从内存层次", list after the CPU reference): H query heads
 * share Hkv key/value heads, query head h reading key/value head h / (H / Hkv).  K and V (and, in
 * the backward, dK and dV) are [B, Hkv, N, d]; Q, O, dO, dQ are [B, H, N, d]; LSE is [B, H, N].
 * dK and dV of a key/value head sum the contributions of all query heads of its group.
 * Hkv must divide H; bf16 or fp16 only (FA_ERR_UNSUPPORTED otherwise).  Hkv = H is fa_forward /
 * fa_backward.  The backward's workspace is fa_backward_workspace_size(B, H, N, d).
 */
fa_status fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Hkv, int N, int d, float scale, int causal,
                         const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                         void* stream);
fa_status fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv,
                          int B, int H, int Hkv, int N, int d, float scale, int causal,
                          const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deterministic backward: the same gradients as fa_backward_gqa (Hkv = H for plain multi-head
 * attention), reproducible to the bit from run to run on the same GPU and inputs.  The
 * recompute-based backward ("FlashAttention paper story", backward paragraph) is split into a
 * pass over key tiles that writes dK and dV, and a pass over query tiles that recomputes S and
 * dP and accumulates each dQ row in one place in a fixed key order; no partial sums are added
 * from several CTAs.  It costs two extra matrix products per tile pair.  bf16 or fp16 only
 * (FA_ERR_UNSUPPORTED for fp32).  workspace: at least
 * fa_backward_deterministic_workspace_size(B, H, N) bytes, 256-byte aligned, caller-owned,
 * contents on entry irrelevant.  Other arguments, errors and ownership as in fa_backward.
 */
size_t fa_backward_deterministic_workspace_size(int B, int H, int N);
fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                    int B, int H, int Hkv, int N, int d, float scale, int causal,
                                    const uint8_t* block_mask, fa_dtype dtype,
                                    const int32_t* kv_lens, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Dropout on the attention probabilities (the "dropout RNG" of the pages' list of production
 * semantics, replayed in the backward).  Element (i, j) of slice (b, h) is kept with probability
 * k8 / 256, k8 = round((1 - p) * 256), and kept probabilities are scaled by 256 / k8:
 *     O = (P * M * 256/k8) V,  LSE as without dropout.
 * M is regenerated, never stored: Philox4x32-10 (Salmon et al., SC 2011) with key = seed and
 * counter (j / 4, i / 4, b*H + h, offset); byte (j mod 4) of output word (i mod 4) is the
 * element's 8-bit uniform, kept iff below k8.  The backward with the same seed and offset
 * replays the same mask.  p must lie in [0, 1]; p = 0 is plain attention.
 */
typedef struct {
  float p;          /* dropout probability */
  uint64_t seed;    /* generator key */
  uint32_t offset;  /* counter word 3: distinct offsets give independent masks for one seed */
} fa_dropout;

/* fa_forward_gqa with dropout (bf16/fp16; no packed sequences, no split-KV). */
fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int Hkv, int N, int d, float scale, int causal,
                             const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                             const fa_dropout* dropout, void* stream);
/* The matching backward (two-pass; workspace fa_backward_deterministic_workspace_size(B, H, N)). */
fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int N, int d, float scale, int causal,
                              const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                              const fa_dropout* dropout, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Packed sequences ("ragged offsets" and the "document mask" in the pages' list of production
 * semantics, "FlashAttention：让精确注意力服从内存层次", list after the CPU reference).  n_seqs
 * sequences of different lengths are stored back to back along each head's token axis:
 *   q, o, dO, dq : [H, total, d];  k, v, dk, dv : [Hkv, total, d];  lse : fp32 [H, total]
 *   cu_seqlens   : device int32 [n_seqs + 1], 0 = cu[0] <= cu[1] <= ... <= cu[n_seqs] <= total;
 *                  sequence s is rows [cu[s], cu[s+1]) of every head
 *   max_seqlen   : an upper bound of every cu[s+1] - cu[s] (sizes the grid; host value)
 * A query attends only to keys of its own sequence (and, with causal, to those at or before it
 * within the sequence); rows outside every sequence are neither read into a result nor written.
 * Grouped heads as in fa_forward_gqa.  bf16 or fp16 only.  The backward is the two-pass
 * backward of fa_backward_deterministic; its workspace is
 * fa_backward_deterministic_workspace_size(1, H, total) bytes.  The offsets live on the device,
 * so they are checked there: a sequence whose offsets break the rules above is skipped and
 * fa_check_device_status then returns FA_ERR_INVALID_ARG.
 */
fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens, int n_seqs, int max_seqlen, int total,
                            int H, int Hkv, int d, float scale, int causal, fa_dtype dtype,
                            void* stream);
fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             const int32_t* cu_seqlens, int n_seqs, int max_seqlen, int total,
                             int H, int Hkv, int d, float scale, int causal, fa_dtype dtype,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-KV forward for decode-shaped problems (few queries against a long key sequence) and for
 * problems with too few (b, h) slices to fill the GPU: the key tiles of every query tile are cut
 * into n_splits ranges processed by separate CTAs, each producing its own (O_s, LSE_s); a merge
 * kernel then combines them with the merge law of the online-softmax statistics (m, l, u)
 * ("FlashAttention：让精确注意力服从内存层次", section "Online softmax": statistics of two tiles
 * combine as m = max(m_a, m_b), l = e^{m_a-m} l_a + e^{m_b-m} l_b, u = e^{m_a-m} u_a + e^{m_b-m} u_b).
 * The result is the same function as fa_forward for Nq = Nk.
 *   q          : [B, H, Nq, d]; k, v: [B, H, Nk, d]; o: [B, H, Nq, d]; lse: [B, H, Nq] fp32
 *   kv_lens    : nullable; [B] valid keys per sequence (clamped to [0, Nk]); no causal or tile mask
 *   dtype      : FA_BF16 or FA_FP16 (FA_FP32: FA_ERR_UNSUPPORTED)
 *   n_splits   : key-tile ranges per query tile, >= 0 (0 = fa_forward_splitkv_auto_splits);
 *                values above ceil(Nk / 128) are reduced to it
 *   workspace  : >= fa_forward_splitkv_workspace_size(B, H, Nq, d, n_splits) bytes (with the
 *                n_splits actually used), 256-byte aligned, caller-owned, overwritten
 */
fa_status fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int Nq, int Nk, int d, float scale,
                             const int32_t* kv_lens, fa_dtype dtype, int n_splits,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_forward_splitkv for grouped-query attention (decode with H query heads on Hkv key/value
 * heads; k, v are [B, Hkv, Nk, d]).  The G = H / Hkv query heads of a group are consecutive in
 * [B, H, Nq, d], so their G * Nq queries form one block of rows that is attended against the
 * group's key/value head in one pass: each K/V tile is read once per group instead of once per
 * query head, and short query blocks fill the 128-row tiles.  Equivalent to
 * fa_forward_splitkv(q, k, v, o, lse, B, Hkv, G * Nq, Nk, ...); n_splits = 0 therefore uses
 * fa_forward_splitkv_auto_splits(B, Hkv, G * Nq, Nk), and the workspace is
 * fa_forward_splitkv_workspace_size(B, H, Nq, d, n_splits) (the same number of rows).
 */
fa_status fa_forward_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                 const int32_t* kv_lens, fa_dtype dtype, int n_splits,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of fa_forward_splitkv (fp32 partial O and LSE of every range). */
size_t fa_forward_splitkv_workspace_size(int B, int H, int Nq, int d, int n_splits);

/* The number of ranges fa_forward_splitkv uses for n_splits = 0: at least about two CTAs per SM
 * of the current device, then the fewest ranges whose CTAs fill their last wave (one CTA per SM)
 * to 95 %; at least two key tiles per range, at most 64 ranges. */
int fa_forward_splitkv_auto_splits(int B, int H, int Nq, int Nk);

/* Bytes of workspace fa_backward, fa_backward_gqa and fa_backward_noalloc's path need for these
 * sizes: one fp32 per query row for D (B*H*N*4), then the order of the work units used under a
 * tile mask (2 ints per 128-row tile and slice, about 1/64 of D), each rounded up to a multiple
 * of 256.  d is not used; it is kept so that the size is asked for with the problem's own sizes. */
size_t fa_backward_workspace_size(int B, int H, int N, int d);

/*
 * Recompute-based backward.  Given the forward's inputs, its O and LSE, and dO, writes
 * dQ, dK, dV ([B,H,N,d], dtype).  P is rebuilt from LSE tile by tile; the N x N matrices are
 * never stored ("FlashAttention paper story", backward paragraph).  Gradients:
 *     dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i * O_i),  dS = P * (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 *   o, lse      : the forward's outputs for the same inputs and mask settings
 *   dO          : incoming gradient of O
 *   dq, dk, dv  : outputs (must not alias any input)
 *   workspace   : device scratch of at least fa_backward_workspace_size(B,H,N,d) bytes,
 *                 256-byte aligned, owned by the caller; its contents on entry do not matter
 *                 and are overwritten.  Two calls in flight at once need two workspaces.
 * Other arguments as in fa_forward.  bf16 and fp16 run the two-pass backward of
 * fa_backward_deterministic (dK/dV over key tiles, dQ over query tiles, no cross-block sums):
 * the same bits on every run.  fp32 runs on the CUDA cores and adds dQ from several blocks
 * into the fp32 dq output (which doubles as its accumulator), in an order that varies in the
 * last bits.
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const void* dO, const float* lse, void* dq, void* dk, void* dv,
                      int B, int H, int N, int d, float scale, int causal,
                      const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_backward without a caller workspace, for callers that cannot allocate device memory:
 * plugin interfaces that pass only input and output pointers, hosts whose device memory is all
 * reserved by their own allocator, and latency-critical paths where cudaMalloc (which
 * synchronises the device) is not allowed.  The pages have no counterpart of this call.
 * The scratch comes from a fixed array of fa_backward_noalloc_max_workspace() bytes (32 MiB)
 * built into the library; every GPU that loads the library holds it until the process exits.
 * Arguments and results are those of fa_backward (the same path: two-pass for bf16/fp16,
 * CUDA cores for fp32).  Returns FA_ERR_UNSUPPORTED, launching nothing, when
 * fa_backward_workspace_size(B, H, N, d) exceeds that size (above about 8.2 million query rows
 * B*H*N).  The first call in a CUDA context looks up the array's device address and caches it
 * for that context; make it before any stream capture.  Not supported after cudaDeviceReset on
 * the device (the cached address can be stale).  All calls share the array: calls that overlap
 * on the GPU race on it and must be serialised.  Nothing carries over between calls: every call
 * rewrites D for each row before reading it.
 */
fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal,
                              const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                              void* stream);

/* Size in bytes of fa_backward_noalloc's built-in scratch array (no counterpart in the pages). */
size_t fa_backward_noalloc_max_workspace(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.  Returns
 * FA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last check, FA_ERR_INVALID_ARG
 * if a kernel found packed-sequence offsets outside their contract, FA_ERR_CUDA if the
 * synchronisation reported a CUDA error, FA_OK otherwise.
 */
fa_status fa_check_device_status(void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/*
 * Test hooks for the failure-detection path (no fault is involved); not for production use.
 * mode 1 makes the next launches of the tensor-core forward skip issuing their first K/V tile
 * load, so the consumers' bounded waits run out; the kernel then records FA_ERR_TIMEOUT and
 * returns normally.  wait_limit_ms sets the bound of every such wait (default 2000 ms; 0
 * restores it).  Both settings are process-wide and change every later launch from every host
 * thread: a test that sets them must restore them (mode 0, limit 0) before other work runs.
 */
void fa_debug_set_fault_injection(int mode);
void fa_debug_set_wait_limit_ms(uint32_t wait_limit_ms);

/*
 * The backward as one key-stationary kernel that computes dK, dV and dQ together, the work
 * partition of the pages' single-pass backward ("FlashAttention paper story", backward
 * paragraph): each key tile's share of dQ is added into an fp32 accumulator in the workspace by
 * the TMA unit (bulk tensor reduce-add), then scaled and converted.  Five matrix products per
 * tile pair instead of the two-pass kernel's seven, but the additions from several CTAs land in
 * an order that varies in the last bits of dQ, and on GB300 it measures slower than the two-pass
 * backward on most shapes.  bf16 or fp16 (FA_ERR_UNSUPPORTED for fp32); grouped heads as in
 * fa_backward_gqa.  workspace: at least fa_backward_fused_workspace_size(B, H, N, d) bytes
 * (fp32 dQ accumulator [B,H,N,d], then D), 256-byte aligned, caller-owned, contents on entry
 * irrelevant.  Other arguments, errors and ownership as in fa_backward.
 */
size_t fa_backward_fused_workspace_size(int B, int H, int N, int d);
fa_status fa_backward_fused(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ABI version of this header: major * 100 + minor. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
