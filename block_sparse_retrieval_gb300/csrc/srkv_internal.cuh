// srkv_internal.cuh -- device helpers and the per-unit page list shared by the decode
// kernels of libsrkv (sm_103a).  Not part of the public interface.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "srkv.h"

namespace srkv {

constexpr int kBlock = 128;               // tokens per page (the pages' block size)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded on-chip waits: 2 s

// ---- error flags -----------------------------------------------------------------------

__device__ __forceinline__ void raise_flags(int32_t* flags, uint32_t bits) {
  if (flags && bits) atomicOr(reinterpret_cast<unsigned int*>(flags), bits);
}

// ---- PTX wrappers ------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Adds `bytes` to the transaction count the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 16-byte copy global -> shared through L2 (an ordinary global load: the source may be
// device memory or host memory mapped into the device's address space).
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
// The mbarrier's current phase also waits for every cp.async this thread issued so far (the
// pending count rises by one now and falls by one when they have landed).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` until the phase completes: a
// waiting warp then sleeps instead of taking issue slots from the warps sharing its SM.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; gives up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// One-dimensional bulk copy global -> shared (TMA engine), completing on an mbarrier.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policies: data read once per step (the K/V pages) goes first, data every step
// reads again (the representation vectors) last.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_load with an L2 eviction policy.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Tiled TMA copy of a 3-D box (x innermost) into shared memory, completing on an mbarrier.
// x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
        "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte read-only global load with an L2 eviction policy.
__device__ __forceinline__ float4 ldg_f4_hint(const float* p, uint64_t policy) {
  float4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ float2 ldg_f2_hint(const float* p, uint64_t policy) {
  float2 v;
  asm volatile("ld.global.nc.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
               : "=f"(v.x), "=f"(v.y)
               : "l"(p), "l"(policy));
  return v;
}

// Programmatic dependent launch: let the next kernel in the stream be scheduled early, and
// wait for the previous one to finish (its writes visible) before reading its outputs.  Both
// are no-ops when the launch did not opt in.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launches `kernel` on `stream`, allowed to start before the previous kernel in the stream
// has finished (the kernel must call griddep_wait() before touching that kernel's outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held one row per four lanes.
// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate (the compressed-page decode: E4M3
// values widen to fp16 exactly).
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 codes (low byte -> low half) as two fp16 values (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// 16-byte shared-memory load (plain C++, so that the compiler orders it after the
// mbarrier waits, whose inline assembly clobbers memory).
__device__ __forceinline__ int4 lds128(const void* p) {
  return *reinterpret_cast<const int4*>(p);
}

// ---- geometry of one (request, kv head) unit ---------------------------------------------
//
// Initial-token blocks are [0, a), window blocks [wstart, nb) (those not already initial
// blocks); candidates meet the offload range [INIT, W).

struct Geom {
  int32_t L;       // clamped length
  int32_t nb;      // blocks holding tokens
  int32_t ie;      // end of the initial tokens: min(INIT, L)
  int32_t ws;      // window start: max(L - LOCAL, 0)
  int32_t W;       // L - LOCAL (may be negative)
  int32_t a;       // init blocks [0, a)
  int32_t wstart;  // window blocks [wstart, nb) that are not init blocks
  int32_t ns;      // clamped selection count
  int32_t pb;      // blocks [0, pb) are attended elsewhere (a shared prefix), not listed
  __device__ __forceinline__ int32_t npos() const { return a + ns + (nb - wstart); }
};

__device__ __forceinline__ Geom make_geom(int32_t seq_len, int32_t nsel, int32_t max_blocks,
                                          int32_t kmax, int32_t INIT, int32_t LOCAL,
                                          uint32_t& eflags) {
  Geom g;
  int32_t L = seq_len;
  const int32_t Lmax = max_blocks * kBlock;
  if (L < 0 || L > Lmax) {
    eflags |= SRKV_EFLAG_SEQ_LEN;
    L = L < 0 ? 0 : Lmax;
  }
  int32_t ns = nsel;
  if (ns < 0 || ns > kmax) {
    eflags |= SRKV_EFLAG_SELECTION;
    ns = ns < 0 ? 0 : kmax;
  }
  g.L = L;
  g.nb = (L + kBlock - 1) / kBlock;
  g.ie = INIT < L ? INIT : L;
  g.W = L - LOCAL;
  g.ws = g.W > 0 ? g.W : 0;
  g.a = (g.ie + kBlock - 1) / kBlock;
  const int32_t wb = g.ws < L ? g.ws / kBlock : g.nb;
  g.wstart = wb > g.a ? wb : g.a;
  g.ns = ns;
  g.pb = 0;
  return g;
}

// Blocks of a shared prefix of `prefix_blocks` pages that the cascade attends for this
// request: the whole pages of the prefix its length covers.
__device__ __forceinline__ int32_t prefix_of(const Geom& g, int32_t prefix_blocks) {
  const int32_t full = g.L / kBlock;
  return prefix_blocks < full ? prefix_blocks : full;
}

// Does logical block b meet the offload range [INIT, W)?
__device__ __forceinline__ bool is_candidate(int32_t b, int32_t INIT, int32_t W) {
  const int64_t lo = max((int64_t)b * kBlock, (int64_t)INIT);
  const int64_t hi = min((int64_t)b * kBlock + kBlock, (int64_t)W);
  return b >= 0 && lo < hi;
}

// What one list position loads: rows [lo, hi) of the page are read; row r is attended iff
// lo <= r < hi and (r < ie or r >= ws).
struct PageTask {
  int32_t page;  // physical page, -1 = nothing to load
  int32_t block;
  int32_t lo, hi, ie, ws;
};

// CTA c of C owns list positions [c*T/C, (c+1)*T/C) of a concatenated list.
__device__ __forceinline__ int64_t cta_begin(int64_t c, int64_t T, int64_t C) {
  return c * T / C;
}
// The CTA whose range holds position p (0 <= p < T).
__device__ __forceinline__ int64_t cta_of(int64_t p, int64_t T, int64_t C) {
  return ((p + 1) * C - 1) / T;
}

// Workspace layout of the decode (all offsets 256-byte aligned).  Partials of list A use
// slots [0, U + C), those of list B slots [U + C, 2 (U + C)).
struct WsLayout {
  size_t off_a;     // int64[U+1]: first list-A position of each unit; [U] = total
  size_t off_b;     // int64[U+1]: the same for list B
  size_t acc;       // float[slots][G][d]: unnormalised partial outputs
  size_t ml;        // float[slots][G][2]: running max (log2 domain) and sum
  size_t total;
  int32_t bank;     // U + C: slots per list
  int64_t cascade;  // first slot of the shared-prefix partials: unit u, range r at
                    // cascade + u * ranges + r
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Shared-prefix attention (decode_cascade.cu): at most kMaxPrefixRanges block ranges per
// prefix (one partial per unit and range), each at most kMaxRangeBlocks blocks long.
constexpr int32_t kMaxPrefixRanges = 8;
constexpr int32_t kMaxRangeBlocks = 256;

// `ranges`: partial slots per unit for a shared prefix (0 without one).
__host__ __device__ inline WsLayout ws_layout(int32_t units, int32_t ctas, int32_t G,
                                              int32_t d, int32_t ranges = 0) {
  WsLayout w;
  w.bank = units + ctas;
  w.cascade = 2 * (int64_t)w.bank;
  const size_t slots = 2 * (size_t)w.bank + (size_t)units * ranges;
  size_t off = 0;
  w.off_a = off;
  off = align256(off + sizeof(int64_t) * ((size_t)units + 1));
  w.off_b = off;
  off = align256(off + sizeof(int64_t) * ((size_t)units + 1));
  w.acc = off;
  off = align256(off + sizeof(float) * slots * G * d);
  w.ml = off;
  off = align256(off + sizeof(float) * 2 * slots * G);
  w.total = off;
  return w;
}

// Arguments shared by the split-phase decode kernels and the combine kernel.
struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t batch;
  const int32_t* sel;
  int32_t kmax;
  const int32_t* nsel;
  void* out;
  char* ws;
  WsLayout lay;
  int32_t* error_flags;
  int32_t Hq, Hkv, G, d;
  int32_t init_tokens, local_tokens;
  float scale_log2;  // log2(e) / sqrt(d)
  int32_t ctas;      // C, the split grid
  int32_t ctas_a;    // CTAs [0, ctas_a) share list A
  int32_t ctas_b;    // CTAs [0, ctas_b) share list B
  int32_t wait_late;  // 1: the previous kernel writes nothing list A reads, so the split
                      // waits for it only before list B (implied by early)
  // Shared prefix: blocks [0, prefix_blocks) of every request map to the same pages and are
  // attended by the cascade kernel (prefix_ranges ranges, cascade_ctas CTAs), not listed by
  // the split kernel.  0: no shared prefix.
  int32_t prefix_blocks;
  int32_t prefix_ranges;
  int32_t cascade_ctas;
  int32_t early;     // 1: the previous kernel is score_topk, so every input but sel and nsel
                     // may be read before it finishes (list A streams during the scoring)
  // early = 1 only: what score_topk derives its selection counts from, so that the
  // decode knows every nsel (selection_count) before the selection exists
  const int32_t* prompt_lens;
  int32_t dense_boundary;
  double topk_percent;
  const float* reps;  // the fused small-batch decode scores too, and writes the selection:
  int32_t* sel_out;
  int32_t* nsel_out;
  // Offload tier: page ids [num_pages, num_pages + num_host_pages) name pages of a pool in
  // host memory mapped into the device's address space (same [Hkv][128][d] page layout).
  const void* k_host;
  const void* v_host;
  int64_t num_host_pages;
  // Compressed pages (the E4M3 decode): fp32 scale of every (page, kv head, token) row.
  const float* k_scale;
  const float* v_scale;
};

// Page ids a block table may hold: the device pool, then the host pool.
__host__ __device__ __forceinline__ int64_t total_pages(const DecodeArgs& a) {
  return a.num_pages + a.num_host_pages;
}

// CTAs that share the positions of a list.
__host__ __device__ __forceinline__ int32_t list_ctas(const DecodeArgs& a, int list) {
  return list == 0 ? a.ctas_a : a.ctas_b;
}

// Shared memory a scoring CTA takes at least: with it no decode CTA (about 217 KB) fits on
// the same SM (228 KB), so the scoring never shares an SM with pages streaming in.
constexpr int kScoreExclusiveSmem = 16 * 1024;

// k = min(n, ceil(p*n - 1e-9)) with separately rounded operations (no contraction), so
// that the host and the device agree on every n.
__device__ __forceinline__ int32_t device_topk_count(int32_t n, double p) {
  if (n <= 0) return 0;
  const double x = ceil(__dadd_rn(__dmul_rn(p, (double)n), -1e-9));
  if (!(x > 0.0)) return 0;
  if (x > (double)n) return n;
  return (int32_t)x;
}

// Candidates of one request and how many of them score_topk keeps (it writes exactly k
// into nsel).  Candidates are the blocks meeting the offload range [INIT, L - LOCAL), from
// block b_lo = INIT / 128 on; a prompt shorter than the dense boundary keeps all of them,
// otherwise k = min(n, ceil(p n - 1e-9)); k is capped at kmax (flagged).  `prompt` is the
// prompt length, or L itself when the caller gives none.
struct SelCount {
  int32_t n, k;
  uint32_t flags;
};

// Candidates of a request of (clamped) length L: blocks from INIT / 128 up to the one
// holding token L - LOCAL - 1.
__device__ __forceinline__ int32_t candidate_count(int32_t L, int32_t LOCAL, int32_t INIT) {
  const int32_t W = L - LOCAL;
  return W > INIT ? (W + kBlock - 1) / kBlock - INIT / kBlock : 0;
}

__device__ __forceinline__ SelCount selection_count(int32_t L, int32_t prompt, int32_t max_blocks,
                                                    int32_t kmax, int32_t INIT, int32_t LOCAL,
                                                    int32_t dense_boundary, double p) {
  SelCount c;
  c.flags = 0;
  const int32_t Lmax = max_blocks * kBlock;
  if (L < 0 || L > Lmax) {
    c.flags |= SRKV_EFLAG_SEQ_LEN;
    L = L < 0 ? 0 : Lmax;
  }
  c.n = candidate_count(L, LOCAL, INIT);
  c.k = prompt < dense_boundary ? c.n : device_topk_count(c.n, p);
  if (c.k > kmax) {
    c.flags |= SRKV_EFLAG_SELECTION;
    c.k = kmax;
  }
  return c;
}

// ---- launchers (defined in the kernel files) ---------------------------------------------

cudaError_t launch_block_reps(const srkv_config& cfg, const void* k_cache, int64_t num_pages,
                              const int32_t* page_ids, const int32_t* valid, int32_t n,
                              float* reps, int32_t* error_flags, cudaStream_t stream);

// CTAs of the scoring grid (clusters of up to 8 per (request, kv head) unit); `compressed`:
// the decode behind it reads E4M3 pages.
int64_t score_topk_ctas(const srkv_config& cfg, int32_t max_blocks, int32_t batch,
                        bool compressed = false);

cudaError_t launch_wait_timeout_selftest(int32_t* error_flags, cudaStream_t stream);
cudaError_t launch_quantize_fp8(const srkv_config& cfg, const void* k_src, const void* v_src,
                                int64_t num_pages, const int32_t* page_ids, int32_t n_pages,
                                void* k8, void* v8, float* k_scale, float* v_scale,
                                int32_t* error_flags, cudaStream_t stream);
cudaError_t launch_append_kv(const srkv_config& cfg, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, int64_t num_pages,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t batch, float* reps,
                             int32_t* error_flags, cudaStream_t stream);

cudaError_t launch_score_topk(const srkv_config& cfg, const void* q, const float* reps,
                              int64_t num_pages, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* seq_lens,
                              const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                              int32_t kmax, int32_t* nsel, int32_t* error_flags,
                              cudaStream_t stream, bool compressed = false);

// Split phase on tensor cores (bf16, G <= 8, d in {64, 128}); grid = SM count.
bool mma_split_supported(const srkv_config& cfg);
int32_t mma_split_ctas(int32_t sm_count);
cudaError_t launch_split_mma(const DecodeArgs& a, cudaStream_t stream);

// Split phase on CUDA cores (any supported dtype / group).
int32_t simt_split_ctas(int32_t sm_count);
cudaError_t launch_split_simt(const DecodeArgs& a, int32_t dtype, cudaStream_t stream);

cudaError_t launch_combine(const DecodeArgs& a, int32_t dtype, cudaStream_t stream);

// Attention over a shared prefix for every request at once (bf16, d 128, group 1/2/4/8):
// partials into the workspace's cascade slots.  pdl: launched behind the previous kernel of
// the stream (it waits for that kernel before reading the selection).
bool cascade_supported(const srkv_config& cfg);
int32_t cascade_ctas(int32_t sm_count);
cudaError_t launch_cascade(const DecodeArgs& a, bool pdl, cudaStream_t stream);

// Scoring, selection and attention of a small batch in one kernel, one thread-block cluster
// per (request, kv head) unit: the cluster size to use for `units` units (0 = not
// applicable: dtype, head size, group, candidates per unit or residency), and its launch.
int32_t fused_cluster_size(const srkv_config& cfg, int32_t units, int32_t max_blocks,
                           bool e4m3 = false);
cudaError_t launch_fused(const DecodeArgs& a, int32_t cluster, cudaStream_t stream);

}  // namespace srkv
