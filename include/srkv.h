/*
 * srkv.h -- C ABI of libsrkv: block-sparse retrieval decode attention over a paged
 * KV cache, for one GB300 GPU (sm_103a).
 *
 * The method (openGauss 7.0.0 DataVec, "KV Cache Query-Based Computation Inference
 * Acceleration"):
 *   - "Feature Description": at prefill, one representation vector is extracted for
 *     every KV block;
 *   - "Overall Solution": the cache of a sequence is split into initial_tokens, the
 *     sliding_window and the offload_tokens between them; at each decode step the
 *     current query is scored by inner product against the representation vector of
 *     every offload block, the topK blocks are kept, and attention runs over the
 *     initial tokens, the kept blocks and the window together;
 *   - "Configuration Parameters": INIT_TOKENS_NUM (1024), LOCAL_TOKENS_NUM (7192),
 *     TOPK_PERCENT (0.2), block size 128, DENSE_BOUNDARY (32K: a prompt shorter than
 *     this is attended densely).
 * Attention itself is softmax(q K^T / sqrt(d)) V (rkmt.cn ATB KV-cache reuse article,
 * §1.1), read through a page table of physical pages (same article, §2.2); a group of
 * query heads shares one K/V head (KV-cache survey "大模型推理百倍加速之KV cache篇",
 * section "Share--KV cache共享").
 *
 * Definitions used by every entry point (S = block_size = 128 tokens per page):
 *   L      = seq_lens[r], the tokens in request r's cache, the current token included;
 *   W      = L - local_tokens, the first token of the sliding window;
 *   candidate blocks of r = logical blocks b whose tokens [bS, bS+S) meet [init_tokens, W);
 *   rep[p][h][:] = fp32 mean of the keys of physical page p, kv head h, over its valid
 *            tokens (the representation vector);
 *   score of block b for (r, h) = (sum of the query vectors of h's group) . rep[bt[r][b]][h];
 *   k = min(n, ceil(topk_percent * n - 1e-9)) of n candidates (0 if n = 0), or n when
 *       prompt_lens[r] < dense_boundary;
 *   selection = the k candidates of highest score, ties to the lower block index;
 *   attended tokens = [0, init_tokens) u (selected blocks n [init_tokens, W)) u [W, L),
 *       as a set; out = softmax over them of q.K/sqrt(d), times V; L = 0 gives 0.
 *
 * Layouts (all row-major, all device memory unless stated):
 *   q, out          [B][Hq][d]        dtype of the config (bf16 or fp32)
 *   k_cache,v_cache [P][Hkv][S][d]    dtype of the config; one (page, kv head) slab of
 *                                     S*d elements is contiguous
 *   reps            [P][Hkv][d]       fp32
 *   block_table     [B][max_blocks]   int32 physical page of logical block b; entries for
 *                                     b >= ceil(L/S) are never read
 *   seq_lens, prompt_lens [B]         int32
 *   sel             [B][Hkv][kmax]    int32 selected logical blocks, ascending
 *   nsel            [B][Hkv]          int32
 * Ownership: the caller owns every buffer.  The library allocates nothing, frees
 * nothing and synchronises only in srkv_retrieval_decode_host (which returns its output in
 * host memory); every other call is asynchronous on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and returns after launching.
 * Errors: the return value reports host-side argument checks and launch failures.
 * Problems only visible on the device (a page id outside [0, num_pages), a sequence
 * longer than max_blocks*S, a malformed selection, a bounded wait that ran out) make
 * the kernels skip the offending work, never fault, and set SRKV_EFLAG_* bits in the
 * optional device word `error_flags` (may be NULL; the caller clears it).
 * No C++ exception crosses this interface.
 */
#ifndef SRKV_H
#define SRKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* srkv_stream; /* identical to cudaStream_t */

typedef enum {
  SRKV_OK = 0,
  SRKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad alignment, bad config value */
  SRKV_ERR_UNSUPPORTED = 2, /* a valid configuration that this build does not implement */
  SRKV_ERR_WORKSPACE = 3,   /* workspace missing or smaller than srkv_decode_workspace_size */
  SRKV_ERR_CUDA = 4         /* a CUDA call or kernel launch failed */
} srkv_status;

typedef enum { SRKV_BF16 = 0, SRKV_F32 = 1 } srkv_dtype;

/* Device-side error bits, OR-ed into *error_flags. */
#define SRKV_EFLAG_PAGE_RANGE 1u /* a block-table entry outside [0, num_pages) was skipped */
#define SRKV_EFLAG_SEQ_LEN 2u    /* seq_len < 0 or > max_blocks*S; clamped into range */
#define SRKV_EFLAG_SELECTION 4u  /* nsel outside [0, kmax], or a sel entry that is not a
                                    candidate or not ascending; such entries were skipped */
#define SRKV_EFLAG_TIMEOUT 8u    /* a bounded on-chip wait ran out; the kernel returned early */
#define SRKV_EFLAG_PREFIX 16u    /* a request maps a block of the declared shared prefix to
                                    another page than the batch's other requests (the
                                    shared-prefix calls read one page for all of them) */

/* Configuration: the method's knobs ("Configuration Parameters") and the head layout. */
typedef struct {
  int32_t num_q_heads;    /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;   /* Hkv */
  int32_t head_dim;       /* d: 64 or 128 */
  int32_t block_size;     /* S: must be 128 (the pages' recommended block size) */
  int32_t init_tokens;    /* INIT_TOKENS_NUM, >= 0, default 1024 */
  int32_t local_tokens;   /* LOCAL_TOKENS_NUM, >= 0, default 7192 */
  double topk_percent;    /* TOPK_PERCENT in [0, 1], default 0.2 */
  int32_t dense_boundary; /* DENSE_BOUNDARY, >= 0, default 32768; 0 disables dense mode */
  int32_t dtype;          /* srkv_dtype of q, caches and out */
} srkv_config;

/* Fills the pages' defaults: Hq 32, Hkv 8, d 128, S 128, 1024 / 7192 / 0.2 / 32768, bf16. */
void srkv_default_config(srkv_config* cfg);

/* Human-readable name of a status; never NULL. */
const char* srkv_status_string(srkv_status status);

/* k for n candidates at ratio p (definition above); 0 for n <= 0. */
int64_t srkv_topk_count(int64_t n_candidates, double topk_percent);

/* Number of candidate blocks of a sequence of seq_len tokens under cfg; 0 if cfg is NULL. */
int64_t srkv_num_candidates(const srkv_config* cfg, int64_t seq_len);

/* The sel capacity (kmax) that srkv_score_topk needs for any request of at most
 * max_blocks*S tokens: all candidates when dense mode can occur, else k of them. */
int32_t srkv_kmax_bound(const srkv_config* cfg, int32_t max_blocks);

/*
 * Representation vectors ("Feature Description": extracted block by block at prefill).
 * For i < n_pages: reps[page_ids[i]][h][:] = mean over t < page_valid_tokens[i] of
 * k_cache[page_ids[i]][h][t][:], accumulated in fp32, for every kv head h.  Pages not
 * listed are left untouched.  page_valid_tokens[i] = 0 writes zeros.
 *   k_cache: [num_pages][Hkv][S][d], 16-byte aligned.   reps: [num_pages][Hkv][d] fp32.
 *   page_ids, page_valid_tokens: device int32 [n_pages]; an id outside [0, num_pages) or a
 *   count outside [0, S] is skipped and flagged (SRKV_EFLAG_PAGE_RANGE).
 */
srkv_status srkv_build_block_reps(const srkv_config* cfg, const void* k_cache,
                                  int64_t num_pages, const int32_t* page_ids,
                                  const int32_t* page_valid_tokens, int32_t n_pages,
                                  float* reps, int32_t* error_flags, srkv_stream stream);

/*
 * Decode-time maintenance of the cache and of the vector store (openGauss page, "Feature
 * Description": the representation vectors are extracted block by block, and "Overall
 * Solution": decode keeps adding tokens to the cache).  For every request r and kv head h,
 * the new token's key and value k_new[r][h][:], v_new[r][h][:] are written at position
 * L = seq_lens[r] of the request, i.e. row L % S of page block_table[r][L / S], and that
 * page's representation vector reps[page][h][:] is recomputed over its rows [0, L % S] -- the
 * same value srkv_build_block_reps gives for the page with L % S + 1 valid tokens.
 *   k_new, v_new: [B][Hkv][d] in the cache dtype, 16-byte aligned; k_cache, v_cache,
 *   num_pages, block_table, max_blocks, reps: as for the other calls (written in place).
 *   seq_lens: device int32 [B], read only: the caller advances the lengths (seq_lens[r] += 1)
 *   after the call, and must give request r a page of its own at block L / S (a page shared
 *   with other requests would change for them too).
 *   A length outside [0, max_blocks * S) (SRKV_EFLAG_SEQ_LEN) or a page id outside
 *   [0, num_pages) (SRKV_EFLAG_PAGE_RANGE) skips that request and is flagged.
 * Asynchronous on `stream`; one kernel.
 */
srkv_status srkv_append_kv(const srkv_config* cfg, const void* k_new, const void* v_new,
                           void* k_cache, void* v_cache, int64_t num_pages,
                           const int32_t* block_table, int32_t max_blocks,
                           const int32_t* seq_lens, int32_t batch, float* reps,
                           int32_t* error_flags, srkv_stream stream);

/*
 * Compressed pages (KV-cache survey "大模型推理百倍加速之KV cache篇": quantising the cache is
 * one of the ways to shrink it).  Writes the listed pages of a bf16 cache as E4M3 codes (the
 * 8-bit floating point format "E4M3" of the OCP 8-bit floating point specification: 4
 * exponent bits, 3 mantissa bits, largest finite value 448) with one fp32 scale per
 * (page, kv head, token) row:
 *   scale = max over the row of |x| / 448   (1 for an all-zero row),
 *   code  = E4M3(x / scale), the quotient in fp32, rounded to nearest, ties to even,
 *           finite values past 448 saturated,
 * so a value is code x scale.  Per row rather than per page, so that a later token needs no
 * re-quantisation of its page.
 *   cfg->dtype must be SRKV_BF16 (the source); k_cache, v_cache: [num_pages][Hkv][S][d] bf16;
 *   k_fp8, v_fp8: [num_pages][Hkv][S][d] bytes; k_scale, v_scale: [num_pages][Hkv][S] fp32;
 *   every pointer 16-byte aligned.  Page page_ids[i] of the source is written to the same
 *   page of the destination; other pages are untouched.  An id outside [0, num_pages) is
 *   skipped and flags SRKV_EFLAG_PAGE_RANGE.
 */
srkv_status srkv_quantize_kv_fp8(const srkv_config* cfg, const void* k_cache,
                                 const void* v_cache, int64_t num_pages,
                                 const int32_t* page_ids, int32_t n_pages, void* k_fp8,
                                 void* v_fp8, float* k_scale, float* v_scale,
                                 int32_t* error_flags, srkv_stream stream);

/*
 * Scoring and top-k ("Overall Solution": inner product of the current query with each
 * representation vector, keep the topK closest).  For every request r and kv head h:
 * sel[r][h][0..nsel[r][h]) = the selected candidate blocks of (r, h), ascending; dense
 * requests (prompt_lens[r] < dense_boundary) select every candidate.
 *   q: [B][Hq][d] (cfg dtype, 16-byte aligned); reps: [num_pages][Hkv][d] fp32 as written
 *   by srkv_build_block_reps for every page a candidate block maps to;
 *   prompt_lens may be NULL (then prompt = seq_len);
 *   kmax >= srkv_kmax_bound(cfg, max_blocks), else SRKV_ERR_INVALID_ARG;
 *   max_blocks <= 25600 (3 276 800 tokens: the key and page of every candidate are held
 *   on chip while a unit is selected), else SRKV_ERR_UNSUPPORTED.
 * The selection is a function of the inputs alone: bitwise the same on every call.
 */
srkv_status srkv_score_topk(const srkv_config* cfg, const void* q, const float* reps,
                            int64_t num_pages, const int32_t* block_table, int32_t max_blocks,
                            const int32_t* seq_lens, const int32_t* prompt_lens, int32_t batch,
                            int32_t* sel, int32_t kmax, int32_t* nsel, int32_t* error_flags,
                            srkv_stream stream);

/* Bytes of device workspace srkv_sparse_paged_decode needs for `batch` requests on the
 * current device; 0 if cfg is invalid. */
size_t srkv_decode_workspace_size(const srkv_config* cfg, int32_t batch);

/*
 * Sparse paged decode attention ("Overall Solution": the kept blocks are concatenated
 * with the initial and window KV and take part in attention; flash-decoding split and
 * merge as in the survey's "Share--KV cache共享" section).  For every request r and query
 * head j of kv head h = j / G:
 *   out[r][j][:] = softmax over the attended tokens of q[r][j].K_t / sqrt(d), times V_t,
 * with the attended set built from sel/nsel (as written by srkv_score_topk, or any
 * ascending list of candidate blocks).  Accumulation is fp32; out has the cfg dtype.
 *   k_cache, v_cache: [num_pages][Hkv][S][d], 16-byte aligned;
 *   workspace: >= srkv_decode_workspace_size(cfg, batch) bytes, 256-byte aligned, contents
 *   need not be initialised; it is scratch owned by this call until the stream reaches
 *   the end of the call.
 */
srkv_status srkv_sparse_paged_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                                     const void* v_cache, int64_t num_pages,
                                     const int32_t* block_table, int32_t max_blocks,
                                     const int32_t* seq_lens, int32_t batch,
                                     const int32_t* sel, int32_t kmax, const int32_t* nsel,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     int32_t* error_flags, srkv_stream stream);

/*
 * One whole decode step: the result of srkv_score_topk followed by srkv_sparse_paged_decode
 * on the same stream, with the selection written to the caller's sel/nsel buffers (openGauss
 * page, "Overall Solution": score, keep the topK blocks, attend them with the initial tokens
 * and the window).  Arguments as for those two calls; prompt_lens may be NULL (the prompt
 * is then the sequence length).
 *   How: a batch small enough for one thread-block cluster per (request, kv head) unit to be
 *   resident (at most 15 units with clusters of 8 to 16 CTAs, or, for bf16 pages with d 128
 *   and a top-k ratio <= 0.3, at most 36 units with clusters of 4 to 7; the largest cluster
 *   size whose clusters are all resident is taken; <= 1024 candidate blocks per request,
 *   bf16, d 64 or 128, group <= 8) runs as one kernel; otherwise the scoring
 *   kernel, the split decode (which
 *   streams the initial and window pages while the scoring runs) and the combine.  The first
 *   call for a configuration on a device queries the device (cluster residency); make it
 *   before any stream capture.  max_blocks <= 25600 as for srkv_score_topk.
 *   Reproducibility: sel and nsel are bitwise the same on every call.  On the three-kernel
 *   path (and in srkv_sparse_paged_decode) out is too.  On the one-kernel path each
 *   streaming CTA of a unit's cluster gets its first 16 kept blocks assigned by the
 *   selection (round robin); out is bitwise the same on every call when no unit keeps more
 *   than 16 blocks per streaming CTA (with clusters of 12 CTAs, 11 streaming: up to 176 kept
 *   blocks); beyond that the CTAs take the remaining kept blocks from a shared pool as their
 *   pages arrive, the partial sums split at pages that vary from call to call, and out may
 *   differ in its last bits.
 */
srkv_status srkv_retrieval_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                                  const void* v_cache, const float* reps, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_blocks,
                                  const int32_t* seq_lens, const int32_t* prompt_lens,
                                  int32_t batch, int32_t* sel, int32_t kmax, int32_t* nsel,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  int32_t* error_flags, srkv_stream stream);

/*
 * srkv_retrieval_decode with host buffers for the per-step inputs and the output, as a
 * serving loop on the host calls it: q_host ([batch][Hq][d] in the cfg dtype), seq_lens_host
 * and prompt_lens_host ([batch] int32; prompt_lens_host may be NULL) are copied into
 * `staging`, the decode runs on them, out is copied into out_host ([batch][Hq][d] in the cfg
 * dtype), and the call returns once out_host holds it (it synchronises `stream`).  Host
 * buffers in page-locked memory copy asynchronously; pageable ones work too, more slowly.
 *   staging: device memory of at least srkv_host_staging_size(cfg, batch) bytes, 256-byte
 *     aligned, owned by the caller; its contents on entry do not matter.  It holds q, then
 *     seq_lens, then prompt_lens, each at a 256-byte boundary; host inputs that sit in one
 *     buffer at those same offsets go in one copy, others in one copy each.
 *   Every other argument, its layout and its errors: srkv_retrieval_decode (out is still a
 *   device buffer, the one the decode writes).  SRKV_ERR_INVALID_ARG for a NULL host
 *   pointer or staging, a small or unaligned staging; SRKV_ERR_CUDA if a copy or the
 *   synchronisation fails (out_host is then undefined).
 */
size_t srkv_host_staging_size(const srkv_config* cfg, int32_t batch);
srkv_status srkv_retrieval_decode_host(const srkv_config* cfg, const void* q_host,
                                       const int32_t* seq_lens_host,
                                       const int32_t* prompt_lens_host, void* out_host,
                                       void* staging, size_t staging_bytes,
                                       const void* k_cache, const void* v_cache,
                                       const float* reps, int64_t num_pages,
                                       const int32_t* block_table, int32_t max_blocks,
                                       int32_t batch, int32_t* sel, int32_t kmax, int32_t* nsel,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       int32_t* error_flags, srkv_stream stream);

/*
 * srkv_retrieval_decode with an offload tier (openGauss page, "Overall Solution" and
 * "Feature Description": KV blocks past the offload boundary live off the accelerator's
 * memory, their representation vectors stay resident, and only the topK blocks the query
 * selects are fetched each step).  Page ids in [0, num_pages) name pages of the device pool
 * k_cache/v_cache; ids in [num_pages, num_pages + num_host_pages) name page
 * (id - num_pages) of a second pool k_host/v_host with the same [page][Hkv][S][d] layout.
 * The decode reads host pages in place, over the chip-to-chip link, straight into the shared
 * memory stages the device pages go through (no staging copy in HBM); which pages live where
 * is the caller's choice (typically the candidate blocks go to the host pool and the initial
 * and window pages stay on the device).  Results equal srkv_retrieval_decode's on the same
 * page contents.
 *   k_host, v_host: pinned (page-locked, e.g. cudaHostAlloc) or managed host memory, or
 *     device memory; 16-byte aligned; pageable memory is rejected (SRKV_ERR_INVALID_ARG).
 *     May be NULL when num_host_pages = 0 (the call is then srkv_retrieval_decode).
 *   reps: [num_pages + num_host_pages][Hkv][d] fp32 in device memory (computed while the
 *     pages were on the device, e.g. by srkv_build_block_reps before they are moved).
 *   A host pool needs the tensor-core decode (bf16, d 64 or 128, group <= 8), else
 *     SRKV_ERR_UNSUPPORTED.  Other arguments, ownership and errors: srkv_retrieval_decode.
 *     The host pool must not be written while the call runs.
 */
srkv_status srkv_retrieval_decode_tiered(const srkv_config* cfg, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         int64_t num_pages, const void* k_host,
                                         const void* v_host, int64_t num_host_pages,
                                         const float* reps, const int32_t* block_table,
                                         int32_t max_blocks, const int32_t* seq_lens,
                                         const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                                         int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                         size_t workspace_bytes, int32_t* error_flags,
                                         srkv_stream stream);

/*
 * srkv_retrieval_decode over compressed pages (srkv_quantize_kv_fp8): the attended K and V
 * values are code x scale of the E4M3 caches, widened to fp16 (exactly) for the tensor-core
 * products, with fp32 accumulation as in the bf16 decode.  The selection comes from `reps`,
 * the representation vectors of the full-precision keys (built by srkv_build_block_reps
 * before the pages are compressed), so it is the selection the bf16 call makes.
 *   cfg->dtype = SRKV_BF16 (the query and the output), head_dim 128, group <= 8, else
 *   SRKV_ERR_UNSUPPORTED.  k_fp8, v_fp8: [num_pages][Hkv][S][d] bytes; k_scale, v_scale:
 *   [num_pages][Hkv][S] fp32; all 16-byte aligned.  Other arguments, ownership, paths (one
 *   kernel for small batches, else three) and errors: srkv_retrieval_decode.
 */
srkv_status srkv_retrieval_decode_fp8(const srkv_config* cfg, const void* q, const void* k_fp8,
                                      const void* v_fp8, const float* k_scale,
                                      const float* v_scale, const float* reps,
                                      int64_t num_pages, const int32_t* block_table,
                                      int32_t max_blocks, const int32_t* seq_lens,
                                      const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                                      int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t* error_flags,
                                      srkv_stream stream);

/*
 * Shared-prefix decode (KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV
 * cache共享": FlashInfer's cascade inference and Hydragen attend a prefix shared by a batch's
 * requests once, as a matrix-matrix product over all their queries, and merge it with each
 * request's own part like Flash-Decoding partials; the ATB reuse article, §2.1 and §3.3, keeps
 * such prefix pages once and references them from every request).  The results are those of
 * srkv_sparse_paged_decode / srkv_retrieval_decode on the same inputs: only the way the work
 * is split changes.  The first prefix_blocks logical blocks of EVERY request must map to the
 * same physical pages (block_table[r][b] == block_table[0][b] for b < prefix_blocks); the
 * whole pages of that prefix a request's length covers are attended for all requests at once,
 * one (page, kv head) slab read per group of up to 128 query rows, with each request's own
 * rows of it (initial tokens, window, its selected blocks) masked in; the rest of each request
 * goes through the split decode.  A request whose table breaks the contract inside its
 * prefix flags SRKV_EFLAG_PREFIX (its result is then not the definition's).
 *   prefix_blocks: 0 <= prefix_blocks <= max_blocks, at most 2048 (else
 *     SRKV_ERR_UNSUPPORTED); 0 gives the plain call.
 *   cfg: bf16, head_dim 128, group 1, 2, 4 or 8 (else SRKV_ERR_UNSUPPORTED).
 *   workspace: >= srkv_prefix_decode_workspace_size(cfg, batch) bytes, 256-byte aligned.
 *   Other arguments, ownership and errors: srkv_sparse_paged_decode / srkv_retrieval_decode.
 *   Both calls always take the kernels of the split path (no one-kernel path); their output
 *   is bitwise the same on every call.
 */
size_t srkv_prefix_decode_workspace_size(const srkv_config* cfg, int32_t batch);

srkv_status srkv_sparse_paged_decode_prefix(const srkv_config* cfg, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            int64_t num_pages, const int32_t* block_table,
                                            int32_t max_blocks, const int32_t* seq_lens,
                                            int32_t batch, int32_t prefix_blocks,
                                            const int32_t* sel, int32_t kmax,
                                            const int32_t* nsel, void* out, void* workspace,
                                            size_t workspace_bytes, int32_t* error_flags,
                                            srkv_stream stream);

srkv_status srkv_retrieval_decode_prefix(const srkv_config* cfg, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         const float* reps, int64_t num_pages,
                                         const int32_t* block_table, int32_t max_blocks,
                                         const int32_t* seq_lens, const int32_t* prompt_lens,
                                         int32_t batch, int32_t prefix_blocks, int32_t* sel,
                                         int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                         size_t workspace_bytes, int32_t* error_flags,
                                         srkv_stream stream);

/*
 * Number of kernels one srkv_retrieval_decode call with these arguments launches on the
 * current device (1 for the one-kernel small-batch path, else 3); 0 if cfg is invalid.
 * Host only; queries the device like the first call does.
 */
int32_t srkv_retrieval_decode_launches(const srkv_config* cfg, int32_t batch, int32_t max_blocks);

/*
 * For callers that cannot allocate device memory: srkv_sparse_paged_decode without a
 * workspace argument.  (The method's pages have no counterpart of this; it is a service of
 * this library.)  Some callers cannot call cudaMalloc on the decode path: code running under
 * stream capture for a CUDA graph (plain cudaMalloc is not a capturable operation), serving
 * loops that forbid allocator calls so that every step costs the same, plugins handed only
 * their input and output buffers by a host framework that owns all device memory, and
 * processes whose device memory is fully reserved up front.  They pass only inputs and
 * outputs; the scratch space is a file-scope device array of SRKV_NOALLOC_WORKSPACE_BYTES
 * in this library, which every GPU that loads the library holds until the process exits.
 *   - Arguments, layouts and results are those of srkv_sparse_paged_decode.
 *   - A batch whose decode needs more scratch than SRKV_NOALLOC_WORKSPACE_BYTES
 *     (srkv_decode_workspace_size) is rejected with SRKV_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and keeps it for the current CUDA context; a call made in another context of
 *     the device (one the caller created, or the primary context brought up again after
 *     cudaDeviceReset) looks it up again.  Make the first call in each context before any
 *     stream capture.
 *   - Every call on a device shares the one array, and each call leaves its contents behind
 *     (nothing in it needs to start at zero: a call writes every value it reads).  Calls
 *     whose kernels overlap on the GPU (on different streams, without ordering between
 *     them) race on it: order them.
 *   - No allocation, free or allocating library routine is called.
 */
#define SRKV_NOALLOC_WORKSPACE_BYTES ((size_t)16 << 20)

srkv_status srkv_sparse_paged_decode_noalloc(const srkv_config* cfg, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             int64_t num_pages, const int32_t* block_table,
                                             int32_t max_blocks, const int32_t* seq_lens,
                                             int32_t batch, const int32_t* sel, int32_t kmax,
                                             const int32_t* nsel, void* out,
                                             int32_t* error_flags, srkv_stream stream);

/*
 * Self-test of the bounded on-chip waits (no counterpart on the pages; a service of this
 * library).  Every wait of the decode kernels gives up after a limit of 2 s, sets
 * SRKV_EFLAG_TIMEOUT and lets its kernel finish instead of hanging.  This call launches one
 * kernel (a cluster of 2 CTAs) whose waits, one on a CTA-scope and one on a cluster-scope
 * mbarrier, have no arrival at all: both run to their limit, OR SRKV_EFLAG_TIMEOUT into
 * *error_flags (device memory) and return, about 4 s after the kernel starts.  Nothing else
 * is read or written, nothing faults, and the context stays usable.
 */
srkv_status srkv_selftest_wait_timeout(int32_t* error_flags, srkv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SRKV_H */
