// srkv_api.cu -- the extern "C" entry points of libsrkv: argument checks and dispatch.
//
// Nothing here allocates, frees or synchronises: every entry point validates its
// arguments on the host, launches on the caller's stream and returns.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "srkv_internal.cuh"

namespace srkv {
namespace {

// Upper bound on the split grid of any kernel on any device this library targets; the
// workspace is sized for it so that its size does not depend on the device.
constexpr int32_t kMaxCtas = 1024;
constexpr int32_t kMaxBlocks = 16777215;  // max_blocks * 128 must fit in int32

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool config_ok(const srkv_config* c) {
  if (!c) return false;
  if (c->num_kv_heads <= 0 || c->num_q_heads <= 0 || c->num_q_heads % c->num_kv_heads) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->block_size != kBlock) return false;
  if (c->init_tokens < 0 || c->local_tokens < 0 || c->dense_boundary < 0) return false;
  if (!(c->topk_percent >= 0.0 && c->topk_percent <= 1.0)) return false;
  if (c->dtype != SRKV_BF16 && c->dtype != SRKV_F32) return false;
  return true;
}

int32_t sm_count() {
  static int32_t cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

srkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SRKV_OK : SRKV_ERR_CUDA; }

int64_t host_topk_count(int64_t n, double p) {
  if (n <= 0) return 0;
  volatile double prod = p * (double)n;  // rounded on its own, as on the device
  const double x = ceil(prod - 1e-9);
  if (!(x > 0.0)) return 0;
  if (x > (double)n) return n;
  return (int64_t)x;
}

int64_t host_num_candidates(const srkv_config& c, int64_t L) {
  const int64_t W = L - c.local_tokens;
  if (W <= c.init_tokens) return 0;
  return (W + kBlock - 1) / kBlock - c.init_tokens / kBlock;
}

int32_t host_kmax_bound(const srkv_config& c, int32_t max_blocks) {
  const int64_t n = host_num_candidates(c, (int64_t)max_blocks * kBlock);
  return (int32_t)(c.dense_boundary > 0 ? n : host_topk_count(n, c.topk_percent));
}

// ranges: partial slots per unit for a shared prefix (0: none).
size_t workspace_size(const srkv_config* cfg, int32_t batch, int32_t ranges = 0) {
  if (!config_ok(cfg) || batch < 0) return 0;
  const int64_t units = (int64_t)batch * cfg->num_kv_heads;
  if (units > INT32_MAX - kMaxCtas) return 0;
  if (units * (2 + ranges) > INT32_MAX / 2) return 0;
  const int32_t G = cfg->num_q_heads / cfg->num_kv_heads;
  return ws_layout((int32_t)units, kMaxCtas, G, cfg->head_dim, ranges).total;
}

// Checks the decode arguments and fills `a`; SRKV_OK means there is work to launch.
srkv_status prepare_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                           const void* v_cache, int64_t num_pages, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                           const int32_t* sel, int32_t kmax, const int32_t* nsel, void* out,
                           void* workspace, size_t workspace_bytes, int32_t* error_flags,
                           DecodeArgs& a, int32_t ranges = 0) {
  if (!config_ok(cfg) || batch < 0 || max_blocks <= 0 || max_blocks > kMaxBlocks || kmax < 0 ||
      num_pages < 0)
    return SRKV_ERR_INVALID_ARG;
  if (batch == 0) return SRKV_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !nsel || !out || num_pages == 0)
    return SRKV_ERR_INVALID_ARG;
  if (kmax > 0 && !sel) return SRKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return SRKV_ERR_INVALID_ARG;
  const int32_t G = cfg->num_q_heads / cfg->num_kv_heads;
  const bool mma = mma_split_supported(*cfg);
  if (!mma && G > 16) return SRKV_ERR_UNSUPPORTED;
  const size_t need = workspace_size(cfg, batch, ranges);
  if (need == 0) return SRKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SRKV_ERR_WORKSPACE;
  const int32_t sms = sm_count();
  if (sms <= 0) return SRKV_ERR_CUDA;

  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.sel = sel;
  a.kmax = kmax;
  a.nsel = nsel;
  a.out = out;
  a.ws = static_cast<char*>(workspace);
  a.error_flags = error_flags;
  a.Hq = cfg->num_q_heads;
  a.Hkv = cfg->num_kv_heads;
  a.G = G;
  a.d = cfg->head_dim;
  a.init_tokens = cfg->init_tokens;
  a.local_tokens = cfg->local_tokens;
  a.scale_log2 = kLog2e / sqrtf((float)cfg->head_dim);
  a.ctas = mma ? mma_split_ctas(sms) : simt_split_ctas(sms);
  if (a.ctas > kMaxCtas) a.ctas = kMaxCtas;
  a.ctas_a = a.ctas;
  a.ctas_b = a.ctas;
  a.lay = ws_layout(batch * cfg->num_kv_heads, kMaxCtas, G, cfg->head_dim, ranges);
  a.early = 0;
  a.wait_late = 0;
  a.prefix_blocks = 0;
  a.prefix_ranges = 0;
  a.cascade_ctas = 0;
  a.prompt_lens = nullptr;
  a.reps = nullptr;
  a.sel_out = nullptr;
  a.nsel_out = nullptr;
  a.k_host = nullptr;
  a.v_host = nullptr;
  a.num_host_pages = 0;
  a.k_scale = nullptr;
  a.v_scale = nullptr;
  a.dense_boundary = cfg->dense_boundary;
  a.topk_percent = cfg->topk_percent;
  return SRKV_OK;
}

// Launches the split kernel and the combine.  early = 1 only when the previous kernel in
// the stream is this library's scoring kernel: list A then streams before that kernel
// finishes (it writes only sel and nsel).
srkv_status launch_decode(const srkv_config* cfg, DecodeArgs& a, int32_t early,
                          cudaStream_t s) {
  a.early = early;
  const cudaError_t e = mma_split_supported(*cfg) ? launch_split_mma(a, s)
                                                  : launch_split_simt(a, cfg->dtype, s);
  if (e != cudaSuccess) return SRKV_ERR_CUDA;
  return cuda_status(launch_combine(a, cfg->dtype, s));
}

srkv_status check_score(const srkv_config* cfg, const void* q, const float* reps,
                        int64_t num_pages, const int32_t* block_table, int32_t max_blocks,
                        const int32_t* seq_lens, int32_t batch, const int32_t* sel,
                        int32_t kmax, const int32_t* nsel) {
  if (!config_ok(cfg) || batch < 0 || max_blocks <= 0 || max_blocks > kMaxBlocks || kmax < 0 ||
      num_pages < 0)
    return SRKV_ERR_INVALID_ARG;
  if (batch == 0) return SRKV_OK;
  if (!q || !reps || !block_table || !seq_lens || !sel || !nsel || num_pages == 0)
    return SRKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(reps, 16)) return SRKV_ERR_INVALID_ARG;
  if (kmax < host_kmax_bound(*cfg, max_blocks)) return SRKV_ERR_INVALID_ARG;
  if ((int64_t)batch * cfg->num_kv_heads > INT32_MAX) return SRKV_ERR_UNSUPPORTED;
  if ((size_t)max_blocks * 8 > 200 * 1024) return SRKV_ERR_UNSUPPORTED;  // keys + pages on chip
  return SRKV_OK;
}

// Checks of a shared-prefix call beyond those of the plain one.
srkv_status check_prefix(const srkv_config* cfg, int32_t prefix_blocks, int32_t max_blocks) {
  if (!config_ok(cfg) || prefix_blocks < 0 || max_blocks <= 0) return SRKV_ERR_INVALID_ARG;
  if (prefix_blocks > max_blocks) return SRKV_ERR_INVALID_ARG;
  if (prefix_blocks > 0 && !cascade_supported(*cfg)) return SRKV_ERR_UNSUPPORTED;
  if (prefix_blocks > kMaxPrefixRanges * kMaxRangeBlocks) return SRKV_ERR_UNSUPPORTED;
  return SRKV_OK;
}

// How a shared prefix of prefix_blocks pages is split: the cascade kernel takes 3/8 of
// the SMs, with about eight (kv head, request group, block range) items per CTA (ranges of at
// most kMaxRangeBlocks blocks); the split decode keeps the other SMs, all resident at once.
void prefix_plan(const srkv_config& cfg, DecodeArgs& a, int32_t prefix_blocks) {
  const int32_t sms = sm_count();
  const int32_t G = cfg.num_q_heads / cfg.num_kv_heads;
  const int32_t groups = (a.batch + 128 / G - 1) / (128 / G);
  const int32_t cas = cascade_ctas(sms);
  const int64_t per = (int64_t)cfg.num_kv_heads * groups;
  int64_t nr = (8 * (int64_t)cas + per - 1) / per;
  const int32_t nr_min = (prefix_blocks + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
  if (nr > kMaxPrefixRanges) nr = kMaxPrefixRanges;
  if (nr > prefix_blocks) nr = prefix_blocks;
  if (nr < nr_min) nr = nr_min;
  a.prefix_blocks = prefix_blocks;
  a.prefix_ranges = (int32_t)nr;
  const int64_t items = per * nr;
  a.cascade_ctas = (int32_t)(items < cas ? items : cas);
  a.ctas = sms - a.cascade_ctas;
  if (a.ctas > kMaxCtas) a.ctas = kMaxCtas;
  a.ctas_a = a.ctas;
  a.ctas_b = a.ctas;
}

// srkv_retrieval_decode over a device pool [0, num_pages) and a host pool
// [num_pages, num_pages + num_host_pages) of page ids (num_host_pages = 0: no host pool).
srkv_status retrieval_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                             const void* v_cache, int64_t num_pages, const void* k_host,
                             const void* v_host, int64_t num_host_pages, const float* k_scale,
                             const float* v_scale, const float* reps,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, const int32_t* prompt_lens, int32_t batch,
                             int32_t* sel, int32_t kmax, int32_t* nsel, void* out,
                             void* workspace, size_t workspace_bytes, int32_t* error_flags,
                             cudaStream_t s, int32_t prefix_blocks = 0) {
  srkv_status st = check_score(cfg, q, reps, num_pages + num_host_pages, block_table, max_blocks,
                               seq_lens, batch, sel, kmax, nsel);
  if (st != SRKV_OK || batch == 0) return st;
  DecodeArgs a;
  const int32_t ranges = prefix_blocks > 0 ? kMaxPrefixRanges : 0;
  st = prepare_decode(cfg, q, k_cache, v_cache, num_pages, block_table, max_blocks, seq_lens,
                      batch, sel, kmax, nsel, out, workspace, workspace_bytes, error_flags, a,
                      ranges);
  if (st != SRKV_OK) return st;
  if (prefix_blocks > 0) {
    a.prompt_lens = prompt_lens;
    a.reps = reps;
    a.sel_out = sel;
    a.nsel_out = nsel;
    prefix_plan(*cfg, a, prefix_blocks);
    const int64_t scoring = score_topk_ctas(*cfg, max_blocks, batch);
    if (2 * scoring <= a.ctas) a.ctas_a = a.ctas - (int32_t)scoring;
    // scoring, then the shared-prefix attention behind it (waiting for the selection), then
    // the split decode, which streams the requests' own initial and window pages at once
    if (launch_score_topk(*cfg, q, reps, num_pages, block_table, max_blocks, seq_lens,
                          prompt_lens, batch, sel, kmax, nsel, error_flags, s) != cudaSuccess)
      return SRKV_ERR_CUDA;
    if (launch_cascade(a, true, s) != cudaSuccess) return SRKV_ERR_CUDA;
    return launch_decode(cfg, a, 1, s);
  }
  a.k_host = k_host;
  a.v_host = v_host;
  a.num_host_pages = num_host_pages;
  a.k_scale = k_scale;  // compressed pages when set
  a.v_scale = v_scale;
  // The scoring kernel, then the decode, which streams list A while the scoring finishes
  // and knows the selection counts it will write from the lengths.  A scoring CTA keeps its
  // SM to itself, so list A goes to the decode CTAs that find an SM free at once (the grid
  // is scheduled in block order); list B, read once the selection exists, to every CTA.
  a.prompt_lens = prompt_lens;
  a.reps = reps;
  a.sel_out = sel;
  a.nsel_out = nsel;
  const bool compressed = k_scale != nullptr;
  // A batch small enough for one cluster per unit to be resident: one kernel does it all.
  const int32_t cluster =
      fused_cluster_size(*cfg, batch * cfg->num_kv_heads, max_blocks, compressed);
  if (cluster > 0) return cuda_status(launch_fused(a, cluster, s));
  const bool early = mma_split_supported(*cfg);
  const int64_t scoring = score_topk_ctas(*cfg, max_blocks, batch, compressed);
  if (early && 2 * scoring <= a.ctas) a.ctas_a = a.ctas - (int32_t)scoring;
  if (launch_score_topk(*cfg, q, reps, num_pages + num_host_pages, block_table, max_blocks,
                        seq_lens, prompt_lens, batch, sel, kmax, nsel, error_flags, s,
                        compressed) != cudaSuccess)
    return SRKV_ERR_CUDA;
  return launch_decode(cfg, a, early ? 1 : 0, s);
}

}  // namespace
}  // namespace srkv

using namespace srkv;

extern "C" {

void srkv_default_config(srkv_config* cfg) {
  if (!cfg) return;
  cfg->num_q_heads = 32;
  cfg->num_kv_heads = 8;
  cfg->head_dim = 128;
  cfg->block_size = kBlock;
  cfg->init_tokens = 1024;
  cfg->local_tokens = 7192;
  cfg->topk_percent = 0.2;
  cfg->dense_boundary = 32768;
  cfg->dtype = SRKV_BF16;
}

const char* srkv_status_string(srkv_status s) {
  switch (s) {
    case SRKV_OK: return "ok";
    case SRKV_ERR_INVALID_ARG: return "invalid argument";
    case SRKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case SRKV_ERR_WORKSPACE: return "workspace missing or too small";
    case SRKV_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int64_t srkv_topk_count(int64_t n_candidates, double topk_percent) {
  return host_topk_count(n_candidates, topk_percent);
}

int64_t srkv_num_candidates(const srkv_config* cfg, int64_t seq_len) {
  if (!config_ok(cfg) || seq_len <= 0) return 0;
  return host_num_candidates(*cfg, seq_len);
}

int32_t srkv_kmax_bound(const srkv_config* cfg, int32_t max_blocks) {
  if (!config_ok(cfg) || max_blocks <= 0) return 0;
  return host_kmax_bound(*cfg, max_blocks);
}

srkv_status srkv_build_block_reps(const srkv_config* cfg, const void* k_cache,
                                  int64_t num_pages, const int32_t* page_ids,
                                  const int32_t* page_valid_tokens, int32_t n_pages,
                                  float* reps, int32_t* error_flags, srkv_stream stream) {
  if (!config_ok(cfg) || n_pages < 0 || num_pages < 0) return SRKV_ERR_INVALID_ARG;
  if (n_pages == 0) return SRKV_OK;
  if (!k_cache || !page_ids || !page_valid_tokens || !reps || num_pages == 0)
    return SRKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(reps, 16)) return SRKV_ERR_INVALID_ARG;
  if ((int64_t)n_pages * cfg->num_kv_heads > INT32_MAX) return SRKV_ERR_UNSUPPORTED;
  return cuda_status(launch_block_reps(*cfg, k_cache, num_pages, page_ids, page_valid_tokens,
                                       n_pages, reps, error_flags, (cudaStream_t)stream));
}

srkv_status srkv_quantize_kv_fp8(const srkv_config* cfg, const void* k_cache,
                                 const void* v_cache, int64_t num_pages,
                                 const int32_t* page_ids, int32_t n_pages, void* k_fp8,
                                 void* v_fp8, float* k_scale, float* v_scale,
                                 int32_t* error_flags, srkv_stream stream) {
  if (!config_ok(cfg) || n_pages < 0 || num_pages < 0) return SRKV_ERR_INVALID_ARG;
  if (cfg->dtype != SRKV_BF16) return SRKV_ERR_UNSUPPORTED;
  if (n_pages == 0) return SRKV_OK;
  if (!k_cache || !v_cache || !page_ids || !k_fp8 || !v_fp8 || !k_scale || !v_scale ||
      num_pages == 0)
    return SRKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_fp8, 16) ||
      !aligned(v_fp8, 16) || !aligned(k_scale, 16) || !aligned(v_scale, 16))
    return SRKV_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_fp8(*cfg, k_cache, v_cache, num_pages, page_ids, n_pages,
                                         k_fp8, v_fp8, k_scale, v_scale, error_flags,
                                         (cudaStream_t)stream));
}

srkv_status srkv_append_kv(const srkv_config* cfg, const void* k_new, const void* v_new,
                           void* k_cache, void* v_cache, int64_t num_pages,
                           const int32_t* block_table, int32_t max_blocks,
                           const int32_t* seq_lens, int32_t batch, float* reps,
                           int32_t* error_flags, srkv_stream stream) {
  if (!config_ok(cfg) || batch < 0 || max_blocks <= 0 || max_blocks > kMaxBlocks ||
      num_pages < 0)
    return SRKV_ERR_INVALID_ARG;
  if (batch == 0) return SRKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens || !reps ||
      num_pages == 0)
    return SRKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(reps, 16))
    return SRKV_ERR_INVALID_ARG;
  if ((int64_t)batch * cfg->num_kv_heads > INT32_MAX) return SRKV_ERR_UNSUPPORTED;
  return cuda_status(launch_append_kv(*cfg, k_new, v_new, k_cache, v_cache, num_pages,
                                      block_table, max_blocks, seq_lens, batch, reps,
                                      error_flags, (cudaStream_t)stream));
}

srkv_status srkv_score_topk(const srkv_config* cfg, const void* q, const float* reps,
                            int64_t num_pages, const int32_t* block_table, int32_t max_blocks,
                            const int32_t* seq_lens, const int32_t* prompt_lens, int32_t batch,
                            int32_t* sel, int32_t kmax, int32_t* nsel, int32_t* error_flags,
                            srkv_stream stream) {
  const srkv_status st = check_score(cfg, q, reps, num_pages, block_table, max_blocks, seq_lens,
                                     batch, sel, kmax, nsel);
  if (st != SRKV_OK || batch == 0) return st;
  return cuda_status(launch_score_topk(*cfg, q, reps, num_pages, block_table, max_blocks,
                                       seq_lens, prompt_lens, batch, sel, kmax, nsel,
                                       error_flags, (cudaStream_t)stream));
}

size_t srkv_decode_workspace_size(const srkv_config* cfg, int32_t batch) {
  return workspace_size(cfg, batch);
}

int32_t srkv_retrieval_decode_launches(const srkv_config* cfg, int32_t batch,
                                       int32_t max_blocks) {
  if (!config_ok(cfg) || batch < 0 || max_blocks <= 0) return 0;
  if (batch == 0) return 0;
  return fused_cluster_size(*cfg, batch * cfg->num_kv_heads, max_blocks) > 0 ? 1 : 3;
}

srkv_status srkv_sparse_paged_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                                     const void* v_cache, int64_t num_pages,
                                     const int32_t* block_table, int32_t max_blocks,
                                     const int32_t* seq_lens, int32_t batch,
                                     const int32_t* sel, int32_t kmax, const int32_t* nsel,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     int32_t* error_flags, srkv_stream stream) {
  DecodeArgs a;
  const srkv_status st = prepare_decode(cfg, q, k_cache, v_cache, num_pages, block_table,
                                        max_blocks, seq_lens, batch, sel, kmax, nsel, out,
                                        workspace, workspace_bytes, error_flags, a);
  if (st != SRKV_OK || batch == 0) return st;
  return launch_decode(cfg, a, 0, (cudaStream_t)stream);
}

size_t srkv_prefix_decode_workspace_size(const srkv_config* cfg, int32_t batch) {
  return workspace_size(cfg, batch, kMaxPrefixRanges);
}

srkv_status srkv_sparse_paged_decode_prefix(const srkv_config* cfg, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            int64_t num_pages, const int32_t* block_table,
                                            int32_t max_blocks, const int32_t* seq_lens,
                                            int32_t batch, int32_t prefix_blocks,
                                            const int32_t* sel, int32_t kmax,
                                            const int32_t* nsel, void* out, void* workspace,
                                            size_t workspace_bytes, int32_t* error_flags,
                                            srkv_stream stream) {
  srkv_status st = check_prefix(cfg, prefix_blocks, max_blocks);
  if (st != SRKV_OK) return st;
  DecodeArgs a;
  st = prepare_decode(cfg, q, k_cache, v_cache, num_pages, block_table, max_blocks, seq_lens,
                      batch, sel, kmax, nsel, out, workspace, workspace_bytes, error_flags, a,
                      kMaxPrefixRanges);
  if (st != SRKV_OK || batch == 0) return st;
  if (prefix_blocks == 0) return launch_decode(cfg, a, 0, (cudaStream_t)stream);
  prefix_plan(*cfg, a, prefix_blocks);
  // the shared-prefix attention first (a plain launch: every input is complete when it
  // starts); the split decode behind it reads only inputs until list B, where it waits for it
  if (launch_cascade(a, false, (cudaStream_t)stream) != cudaSuccess) return SRKV_ERR_CUDA;
  a.wait_late = 1;
  return launch_decode(cfg, a, 0, (cudaStream_t)stream);
}

srkv_status srkv_retrieval_decode(const srkv_config* cfg, const void* q, const void* k_cache,
                                  const void* v_cache, const float* reps, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_blocks,
                                  const int32_t* seq_lens, const int32_t* prompt_lens,
                                  int32_t batch, int32_t* sel, int32_t kmax, int32_t* nsel,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  int32_t* error_flags, srkv_stream stream) {
  return retrieval_decode(cfg, q, k_cache, v_cache, num_pages, nullptr, nullptr, 0, nullptr,
                          nullptr, reps,
                          block_table, max_blocks, seq_lens, prompt_lens, batch, sel, kmax, nsel,
                          out, workspace, workspace_bytes, error_flags, (cudaStream_t)stream);
}

// Staging of the host-buffer call: q, then the lengths, then the prompt lengths, each at a
// 256-byte boundary.
static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
static size_t staging_q_bytes(const srkv_config* cfg, int32_t batch) {
  return (size_t)batch * (size_t)cfg->num_q_heads * (size_t)cfg->head_dim *
         (cfg->dtype == SRKV_F32 ? 4u : 2u);
}

size_t srkv_host_staging_size(const srkv_config* cfg, int32_t batch) {
  if (!cfg || batch < 0 || cfg->num_q_heads <= 0 || cfg->head_dim <= 0) return 0;
  return round256(staging_q_bytes(cfg, batch)) + 2 * round256((size_t)batch * 4);
}

srkv_status srkv_retrieval_decode_host(const srkv_config* cfg, const void* q_host,
                                       const int32_t* seq_lens_host,
                                       const int32_t* prompt_lens_host, void* out_host,
                                       void* staging, size_t staging_bytes,
                                       const void* k_cache, const void* v_cache,
                                       const float* reps, int64_t num_pages,
                                       const int32_t* block_table, int32_t max_blocks,
                                       int32_t batch, int32_t* sel, int32_t kmax, int32_t* nsel,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       int32_t* error_flags, srkv_stream stream) {
  if (!cfg || batch < 0) return SRKV_ERR_INVALID_ARG;
  if (batch > 0 && (!q_host || !seq_lens_host || !out_host || !staging))
    return SRKV_ERR_INVALID_ARG;
  const size_t need = srkv_host_staging_size(cfg, batch);
  if (need == 0 || staging_bytes < need ||
      (reinterpret_cast<uintptr_t>(staging) & 255u) != 0)
    return SRKV_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  const size_t qb = staging_q_bytes(cfg, batch), lb = (size_t)batch * 4;
  unsigned char* q_dev = static_cast<unsigned char*>(staging);
  int32_t* lens_dev = reinterpret_cast<int32_t*>(q_dev + round256(qb));
  int32_t* prompt_dev = reinterpret_cast<int32_t*>(q_dev + round256(qb) + round256(lb));
  if (batch > 0) {
    // inputs laid out like the staging (one host buffer at the same offsets) go in one copy
    const unsigned char* qh = static_cast<const unsigned char*>(q_host);
    const bool packed =
        reinterpret_cast<const unsigned char*>(seq_lens_host) == qh + round256(qb) &&
        (!prompt_lens_host ||
         reinterpret_cast<const unsigned char*>(prompt_lens_host) ==
             qh + round256(qb) + round256(lb));
    bool ok;
    if (packed) {
      const size_t bytes = prompt_lens_host ? round256(qb) + round256(lb) + lb : round256(qb) + lb;
      ok = cudaMemcpyAsync(q_dev, q_host, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
    } else {
      ok = cudaMemcpyAsync(q_dev, q_host, qb, cudaMemcpyHostToDevice, s) == cudaSuccess &&
           cudaMemcpyAsync(lens_dev, seq_lens_host, lb, cudaMemcpyHostToDevice, s) ==
               cudaSuccess &&
           (!prompt_lens_host || cudaMemcpyAsync(prompt_dev, prompt_lens_host, lb,
                                                 cudaMemcpyHostToDevice, s) == cudaSuccess);
    }
    if (!ok) {
      (void)cudaGetLastError();
      return SRKV_ERR_CUDA;
    }
  }
  const srkv_status st =
      srkv_retrieval_decode(cfg, q_dev, k_cache, v_cache, reps, num_pages, block_table,
                            max_blocks, lens_dev, prompt_lens_host ? prompt_dev : nullptr,
                            batch, sel, kmax, nsel, out, workspace, workspace_bytes,
                            error_flags, stream);
  if (st != SRKV_OK) return st;
  if ((batch > 0 && cudaMemcpyAsync(out_host, out, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    (void)cudaGetLastError();
    return SRKV_ERR_CUDA;
  }
  return SRKV_OK;
}

srkv_status srkv_retrieval_decode_prefix(const srkv_config* cfg, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         const float* reps, int64_t num_pages,
                                         const int32_t* block_table, int32_t max_blocks,
                                         const int32_t* seq_lens, const int32_t* prompt_lens,
                                         int32_t batch, int32_t prefix_blocks, int32_t* sel,
                                         int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                         size_t workspace_bytes, int32_t* error_flags,
                                         srkv_stream stream) {
  const srkv_status st = check_prefix(cfg, prefix_blocks, max_blocks);
  if (st != SRKV_OK) return st;
  return retrieval_decode(cfg, q, k_cache, v_cache, num_pages, nullptr, nullptr, 0, nullptr,
                          nullptr, reps, block_table, max_blocks, seq_lens, prompt_lens, batch,
                          sel, kmax, nsel, out, workspace, workspace_bytes, error_flags,
                          (cudaStream_t)stream, prefix_blocks);
}

srkv_status srkv_retrieval_decode_tiered(const srkv_config* cfg, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         int64_t num_pages, const void* k_host,
                                         const void* v_host, int64_t num_host_pages,
                                         const float* reps, const int32_t* block_table,
                                         int32_t max_blocks, const int32_t* seq_lens,
                                         const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                                         int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                         size_t workspace_bytes, int32_t* error_flags,
                                         srkv_stream stream) {
  if (!cfg || num_host_pages < 0 || num_pages < 0 || num_pages > INT32_MAX - num_host_pages)
    return SRKV_ERR_INVALID_ARG;
  if (num_host_pages > 0) {
    if (!config_ok(cfg)) return SRKV_ERR_INVALID_ARG;
    if (!mma_split_supported(*cfg)) return SRKV_ERR_UNSUPPORTED;
    if (!k_host || !v_host || !aligned(k_host, 16) || !aligned(v_host, 16))
      return SRKV_ERR_INVALID_ARG;
    // The pool must be reachable from the device: pinned (page-locked) or managed host
    // memory, or device memory.  Pageable memory is refused.
    const void* hp[2] = {k_host, v_host};
    for (int i = 0; i < 2; ++i) {
      cudaPointerAttributes at;
      if (cudaPointerGetAttributes(&at, hp[i]) != cudaSuccess) {
        (void)cudaGetLastError();
        return SRKV_ERR_INVALID_ARG;
      }
      if (at.type == cudaMemoryTypeUnregistered || !at.devicePointer)
        return SRKV_ERR_INVALID_ARG;
      hp[i] = at.devicePointer;
    }
    k_host = hp[0];
    v_host = hp[1];
  }
  return retrieval_decode(cfg, q, k_cache, v_cache, num_pages, k_host, v_host, num_host_pages,
                          nullptr, nullptr, reps, block_table, max_blocks, seq_lens, prompt_lens,
                          batch, sel, kmax, nsel, out, workspace, workspace_bytes, error_flags,
                          (cudaStream_t)stream);
}

srkv_status srkv_retrieval_decode_fp8(const srkv_config* cfg, const void* q, const void* k_fp8,
                                      const void* v_fp8, const float* k_scale,
                                      const float* v_scale, const float* reps,
                                      int64_t num_pages, const int32_t* block_table,
                                      int32_t max_blocks, const int32_t* seq_lens,
                                      const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                                      int32_t kmax, int32_t* nsel, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t* error_flags,
                                      srkv_stream stream) {
  if (!config_ok(cfg)) return SRKV_ERR_INVALID_ARG;
  if (!mma_split_supported(*cfg) || cfg->head_dim != 128) return SRKV_ERR_UNSUPPORTED;
  if (batch > 0 && (!k_scale || !v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16)))
    return SRKV_ERR_INVALID_ARG;
  return retrieval_decode(cfg, q, k_fp8, v_fp8, num_pages, nullptr, nullptr, 0, k_scale, v_scale,
                          reps, block_table, max_blocks, seq_lens, prompt_lens, batch, sel, kmax,
                          nsel, out, workspace, workspace_bytes, error_flags,
                          (cudaStream_t)stream);
}

srkv_status srkv_selftest_wait_timeout(int32_t* error_flags, srkv_stream stream) {
  if (!error_flags) return SRKV_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout_selftest(error_flags, (cudaStream_t)stream));
}

// Scratch of srkv_sparse_paged_decode_noalloc: one array per device that loads the library.
static __device__ __align__(256) unsigned char g_noalloc_workspace[SRKV_NOALLOC_WORKSPACE_BYTES];

// Where that array sits in the current context.  The address belongs to a context, not to a
// device ordinal: after cudaDeviceReset (or under a context the caller created) the module is
// loaded again and the array may move, so the cached address is keyed by the context's
// process-unique id and looked up again whenever the current context differs.
struct NoallocSlot {
  unsigned long long ctx_id;
  void* address;
};
static NoallocSlot g_noalloc_slot[128];
static std::mutex g_noalloc_mu;

using CtxGetCurrent = CUresult (*)(CUcontext*);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the current context (false if there is none or it cannot be read).
static bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrent get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrent>(p);
  }();
  static CtxGetId get_id = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetId>(p);
  }();
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// The array's device address in the current context of device `dev`: cached, or looked up
// with cudaGetSymbolAddress (which also brings up the device's primary context if no
// context is current yet).  Null on failure.
static void* noalloc_address(int dev) {
  unsigned long long id = 0;
  const bool have_id = current_ctx_id(&id);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocSlot& slot = g_noalloc_slot[dev];
  if (have_id && slot.address && slot.ctx_id == id) return slot.address;
  void* ws = nullptr;
  if (cudaGetSymbolAddress(&ws, g_noalloc_workspace) != cudaSuccess || !ws) {
    (void)cudaGetLastError();
    slot.address = nullptr;
    return nullptr;
  }
  if (!current_ctx_id(&id)) return ws;  // no id to key it by: used for this call only
  slot.ctx_id = id;
  slot.address = ws;
  return ws;
}

srkv_status srkv_sparse_paged_decode_noalloc(const srkv_config* cfg, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             int64_t num_pages, const int32_t* block_table,
                                             int32_t max_blocks, const int32_t* seq_lens,
                                             int32_t batch, const int32_t* sel, int32_t kmax,
                                             const int32_t* nsel, void* out,
                                             int32_t* error_flags, srkv_stream stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return SRKV_ERR_CUDA;
  // once per context of the device, with it current: the array's device address
  void* ws = noalloc_address(dev);
  if (!ws) return SRKV_ERR_CUDA;
  DecodeArgs a;
  const srkv_status st = prepare_decode(cfg, q, k_cache, v_cache, num_pages, block_table,
                                        max_blocks, seq_lens, batch, sel, kmax, nsel, out, ws,
                                        SRKV_NOALLOC_WORKSPACE_BYTES, error_flags, a);
  if (st != SRKV_OK || batch == 0) return st;
  return launch_decode(cfg, a, 0, (cudaStream_t)stream);
}

}  // extern "C"
