/* Paged Multi-head Latent Attention (MLA) decode for one GB300 (sm_103a).
 *
 * C ABI of libmla_decode.so. Plain pointers and sizes only; every pointer
 * named "device" is caller-owned device memory (for example a torch tensor's
 * data_ptr()). The calls below never allocate device memory and never
 * synchronise the stream, except mla_get_error, which is a diagnostic.
 * `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *
 * The operation, as the pages state it:
 *  - Each token of a DeepSeek-V2/V3-style MLA layer is cached as one latent
 *    row: kv_lora_rank 512 (c_kv) plus qk_rope_head_dim 64, with no per-head
 *    K or V (SGLang PR #32972 "Let Kimi-Linear use the paged MLA attention
 *    backends", Validation). With the query absorbed into latent space
 *    (q_nope * W_UK || q_rope, 576-d), every head attends over the same
 *    576-d keys, and the first 512 dims of each row are the shared value.
 *  - The pool is paged; a request's pages are listed in a block table or in
 *    CSR kv_indices (same page, "What this does").
 *  - The pool has a leading layer dimension so layers never alias slots
 *    (MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention shim (MLA)",
 *    Root causes 5).
 *  - The new token's latent row is written through slot_mapping on every
 *    decode step (same page, Root causes 2); context_length excludes that
 *    just-generated token (Root causes 4), so the new token sits at position
 *    L = context_lens[b] and is attended.
 *  - The MLA softmax scale is passed explicitly (same page, Changes).
 *  - Optional sliding window over the most recent tokens (FastDeploy PR #8049
 *    "Support MLA_SWA functionality", Motivation): window W > 0 attends
 *    positions [max(0, L + 1 - W), L]; W = 0 attends [0, L].
 *  - Optional fp8_e4m3 cache (SGLang PR #32972, Validation table,
 *    tokenspeed_mla row), dequantised inside the kernel, never materialised
 *    as bf16 (same page, Pre-existing issues 2).
 *
 * Error behaviour: every call returns 0 or a negative MLA_ERR_* code after
 * checking its host-visible arguments. Conditions only the device can see
 * (a page id outside [0, num_pages), a slot outside the layer, a plan that
 * does not match the decode call, a bounded wait that ran out) set bits in a
 * sticky status word inside the workspace and the offending load or store is
 * skipped; no kernel traps. Read the word with mla_get_error.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_OK 0
#define MLA_ERR_ARG (-1)          /* bad host argument (null, size, range) */
#define MLA_ERR_UNSUPPORTED (-2)  /* shape or dtype this library does not build */
#define MLA_ERR_WORKSPACE (-3)    /* workspace too small or misaligned */
#define MLA_ERR_CUDA (-4)         /* a CUDA runtime call failed */

/* Bits of the device status word (mla_get_error). */
#define MLA_STATUS_BAD_PAGE 0x1     /* page id outside [0, num_pages): load skipped */
#define MLA_STATUS_BAD_SLOT 0x2     /* slot_mapping entry >= num_pages*page_size: write skipped */
#define MLA_STATUS_PLAN_MISMATCH 0x4 /* decode arguments differ from the plan's */
#define MLA_STATUS_TIMEOUT 0x8      /* a bounded wait inside a kernel ran out */
#define MLA_STATUS_BAD_LENGTH 0x10  /* context_lens[b] < 0 or beyond the block table */

#define MLA_DTYPE_BF16 0
#define MLA_DTYPE_FP8_E4M3 1

#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_LATENT_DIM 576 /* MLA_KV_LORA_RANK + MLA_ROPE_DIM */
#define MLA_V_HEAD_DIM 128 /* output width of mla_uv_project */

/* A paged latent pool: data is [num_layers][num_pages][page_size][576]
 * row-major, element type bf16 or e4m3 (one byte). data must be 16-byte
 * aligned. page_size is 16, 32, 64 or 128. kv_scale (fp8 only, > 0): the
 * stored code is e4m3(x / kv_scale) and the value read is code * kv_scale. */
typedef struct {
  void* data;
  int num_layers;
  int num_pages;
  int page_size;
  int dtype;
  float kv_scale;
} mla_kv_pool;

/* Latent write (the per-step KV persistence of MoE-Infinity PR #195, Root
 * causes 2 and Changes; pad-row rule of SGLang PR #32972, Cuda-graph safety).
 * For i < n: if slot_mapping[i] >= 0, row `new_rows[i]` is stored at
 * pool[layer][slot / page_size][slot % page_size]; negative slots are pad rows
 * and write nothing. fp8 pools store e4m3 with round-to-nearest-even and
 * saturation to +-448 of (float(x) / kv_scale), computed in IEEE fp32.
 *   new_rows:     device, [n][576] bf16, 16-byte aligned rows.
 *   slot_mapping: device, [n] int64, slot within the layer.
 *   workspace:    device decode workspace whose status word records slots
 *                 beyond the layer (write skipped), or NULL to skip silently.
 * Returns MLA_ERR_ARG for a null pool/rows/slots with n > 0 or a layer out of
 * range. */
int mla_kv_write(const mla_kv_pool* pool, int layer, const void* new_rows,
                 const int64_t* slot_mapping, int n, void* workspace,
                 void* stream);

/* Bytes of decode workspace for `batch` requests of `num_heads` heads on the
 * current device (room for the widest schedule, mla_decode_num_clusters()).
 * 0 on bad arguments or when the device cannot run the decode kernel. The
 * workspace must be 256-byte aligned and zeroed once before its first use
 * (its status word starts at 0); later calls keep it consistent. */
size_t mla_decode_workspace_size(int batch, int num_heads);

/* Number of two-CTA clusters of the decode kernel that fit on the current
 * device at once (the default schedule width), or a negative error. */
int mla_decode_num_clusters(void);

/* Split-KV schedule (the plan/run split of FlashInfer's plan(), described in
 * SGLang PR #32972, Correction: the plan writes into a buffer the caller
 * keeps, so a captured decode reads what the last plan wrote).
 * Reads context_lens (device, [batch] int32, tokens cached before this step),
 * splits the attended tokens of all requests into 64-token blocks, and
 * deals the blocks to `num_clusters` clusters. Either the concatenated block
 * sequence is cut into equal contiguous ranges, one per cluster, or (batches
 * of up to 1024 requests, when it is estimated cheaper) only requests
 * heavier than a cluster's share are split into near-equal pieces and the
 * pieces are dealt largest first, at most two per cluster. A request split
 * over several clusters has its partial results merged by mla_decode. The
 * schedule depends only on the lengths and is the same on every call with
 * the same arguments. Must be re-run whenever context_lens,
 * batch, num_heads, page_size or window change, before mla_decode.
 *   num_clusters: 0 = mla_decode_num_clusters(); 1 = no split at all;
 *                 values above mla_decode_num_clusters() are clamped to it.
 *   window:       0 = full attention, else the sliding-window width.
 * Returns MLA_ERR_WORKSPACE if workspace_bytes is below
 * mla_decode_workspace_size(batch, num_heads). */
int mla_decode_plan(const int32_t* context_lens, int batch, int num_heads,
                    int page_size, int window, int num_clusters,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Absorbed paged MLA decode, q_len = 1. For each request b and head h:
 *   s_t = softmax_scale * q[b,h,:] . K_t over t in [start_b, L_b],
 *   out[b,h,:] = sum_t softmax(s)_t * K_t[0:512],
 *   lse[b,h]   = log(sum_t exp(s_t))  (natural log),
 * with K_t the 576-d latent row of position t of request b in `layer`, and
 * start_b = 0 or max(0, L_b + 1 - window). Positions live in block
 * t / page_size of the request's page list: page_indptr != NULL selects the
 * CSR form (page_ids[page_indptr[b] + j]); otherwise page_ids is a block
 * table [batch][max_blocks]. Only the blocks that hold attended positions are
 * read (the bounded-prefix rule of SGLang PR #32972, Correction); a page id
 * outside [0, num_pages) sets MLA_STATUS_BAD_PAGE and its rows read as zero.
 *   q:   device, [batch][num_heads][576] bf16 (absorbed nope 512 || rope 64).
 *   out: device, [batch][num_heads][512] bf16, 32-byte aligned (the kernel
 *        writes whole 32-byte sectors). lse: device [batch][num_heads] fp32
 *        or NULL. q must be 16-byte aligned; MLA_ERR_ARG otherwise.
 *   workspace: the one last given to mla_decode_plan with the same batch,
 *        num_heads, page_size and window.
 * num_heads must be 16, 32, 64 or 128 (MLA_ERR_UNSUPPORTED otherwise). The
 * latent width is fixed at 576/512. Arithmetic: fp32 accumulation; the two
 * CTAs that share a work unit exchange their half-dimension partial scores,
 * scaled to log2 units and rounded to fp16 (relative error at most 2^-11 of
 * a partial; magnitudes beyond 65504 saturate). fp8 pools are dequantised in the kernel, tile by tile: the codes
 * are exact in f16, q is converted to f16 (exact for |q| in [2^-14, 65504],
 * saturating beyond) and kv_scale multiplies the scores and the output.
 * Launches the split kernel and the merge kernel (which returns at once when
 * the plan split no request) on `stream`. */
int mla_decode(const mla_kv_pool* pool, int layer, const void* q,
               const int32_t* page_indptr, const int32_t* page_ids,
               int max_blocks, const int32_t* context_lens, int batch,
               int num_heads, float softmax_scale, int window,
               void* workspace, void* out, float* lse, void* stream);

/* Several query positions per request: multi-token decode (speculative or
 * multi-token-prediction steps, LightLLM PR #1593 "Support dsv4 model",
 * Summary and Validation) and, with longer runs of positions, the absorbed
 * form of chunked prefill over the paged latent (vLLM #12639 "[Attention]
 * MLA with chunked prefill", Future work). Request b holds L_b =
 * context_lens[b] cached tokens before this step; its q_len new tokens sit
 * at positions L_b .. L_b + q_len - 1 (their latent rows written beforehand
 * with mla_kv_write, q_len slots per request), and query position i attends
 * positions [start_i, L_b + i] with start_i = 0, or max(0, L_b + i + 1 -
 * window): causal within the step. q_len = 1 is mla_decode exactly.
 *   q:   device [batch][q_len][num_heads][576] bf16, 16-byte aligned.
 *   out: device [batch][q_len][num_heads][512] bf16, 32-byte aligned;
 *   lse: device [batch][q_len][num_heads] fp32 or NULL.
 * The q_len x num_heads rows of a request run in groups of 128 (one
 * tensor-core tile of rows); each group reads the request's pages once.
 * batch x q_len x num_heads must stay below 2^31 (MLA_ERR_ARG).
 * Workspace and plan: mla_decode_workspace_size_q and mla_decode_plan_q with
 * the same batch, q_len and num_heads (a plan made for another q_len sets
 * MLA_STATUS_PLAN_MISMATCH). Everything else as for mla_decode. */
size_t mla_decode_workspace_size_q(int batch, int q_len, int num_heads);
int mla_decode_plan_q(const int32_t* context_lens, int batch, int q_len,
                      int num_heads, int page_size, int window,
                      int num_clusters, void* workspace,
                      size_t workspace_bytes, void* stream);
int mla_decode_q(const mla_kv_pool* pool, int layer, const void* q,
                 const int32_t* page_indptr, const int32_t* page_ids,
                 int max_blocks, const int32_t* context_lens, int batch,
                 int q_len, int num_heads, float softmax_scale, int window,
                 void* workspace, void* out, float* lse, void* stream);

/* W_UV projection after attention: y[b,h,:] = attn_out[b,h,:] @ w_uv[h],
 * v_head_dim 128 (MoE-Infinity PR #195, Root causes 3).
 *   attn_out: device [batch][num_heads][512] bf16; w_uv: device
 *   [num_heads][512][128] bf16; y: device [batch][num_heads][128] bf16; all
 *   16-byte aligned (MLA_ERR_ARG otherwise).
 *   workspace: a decode workspace (256-byte aligned) whose status word
 *   records MLA_STATUS_TIMEOUT if a bounded wait inside the kernel runs out,
 *   or NULL. Either way the rows such a wait leaves unfinished are written
 *   as NaN, never left stale.
 * fp32 accumulation. */
int mla_uv_project(const void* attn_out, const void* w_uv, void* y, int batch,
                   int num_heads, void* workspace, void* stream);

/* Reads the status word of `workspace` into *code (MLA_STATUS_* bits) and, if
 * `clear` is nonzero, resets it. Synchronises `stream`: diagnostics only. */
int mla_get_error(void* workspace, int* code, int clear, void* stream);

/* Self-test of the bounded wait that every kernel of this library uses on
 * its mbarriers (the published method has no counterpart of this call): one
 * thread waits for the first phase of a fresh mbarrier, limited to limit_us
 * microseconds of global time. With arrive == 0 nothing ever completes the
 * phase, the wait runs out and MLA_STATUS_TIMEOUT is OR-ed into *status (a
 * device int32); with arrive != 0 the thread arrives first and *status is
 * left unchanged. Either way the kernel returns and the context stays
 * usable. Returns MLA_ERR_ARG for a null status or limit_us outside
 * [1, 1000000]. Asynchronous on `stream`. */
int mla_selftest_bounded_wait(int arrive, unsigned int limit_us, int32_t* status, void* stream);

/* Allocation-free decode, for callers that cannot allocate device memory at
 * all: code running inside a memory pool or arena that it does not own,
 * plugins whose host forbids cudaMalloc while a graph or a tight memory
 * budget is active, or embedded runtimes that only hand out fixed buffers.
 * The published method has no counterpart of this call; it is the same operation as
 * mla_decode_plan followed by mla_decode (same arguments, same results),
 * with the schedule and the split partials kept in a scratch array that the
 * library declares at file scope (MLA_NOALLOC_SCRATCH_BYTES of device
 * memory, held by every GPU that loads the library until the process ends).
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - A call needs mla_decode_workspace_size(batch, num_heads) bytes of that
 *     scratch: on a 152-SM GPU about 38 MiB of split partials at 128 heads
 *     plus 64 bytes per request, so up to about 150,000 requests fit; a
 *     larger call returns MLA_ERR_WORKSPACE without launching anything.
 *   - The first call on a device looks up the scratch array's device
 *     address; make that first call before any stream capture.
 *   - Every call shares the one scratch array: calls whose work overlaps on
 *     the GPU (different streams, no ordering between them) race. Order them
 *     on one stream.
 *   - The scratch keeps the last call's contents; each call resets its
 *     status word first. status (device int32 or NULL) receives the
 *     MLA_STATUS_* bits of this call when the decode has finished.
 *   - num_clusters as in mla_decode_plan (0 = full width). */
#define MLA_NOALLOC_SCRATCH_BYTES (48u << 20)
int mla_decode_noalloc(const mla_kv_pool* pool, int layer, const void* q,
                       const int32_t* page_indptr, const int32_t* page_ids,
                       int max_blocks, const int32_t* context_lens, int batch,
                       int num_heads, float softmax_scale, int window,
                       int num_clusters, void* out, float* lse,
                       int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
