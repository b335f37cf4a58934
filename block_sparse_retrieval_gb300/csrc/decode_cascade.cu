// decode_cascade.cu -- attention over a prefix of pages shared by every request of a batch,
// read once per kv head for all of them (cascade attention).
//
// KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV cache共享": when the
// requests of a batch share a prefix, FlashInfer's cascade inference runs the attention over
// the shared KV as one multi-query pass, and Hydragen splits prefix and suffix so that the
// prefix part becomes matrix-matrix products over all the requests' queries; the two parts
// are merged like Flash-Decoding partials.  Here the first `prefix_blocks` logical blocks of
// every request map to the same physical pages (the ATB reuse article, §2.1 and §3.3: prefix
// pages kept once and referenced by every request), and the attended rows of a shared block
// still follow the method of the openGauss DataVec page ("Overall Solution"): a request
// attends the block's initial-token rows, its window rows and, if the block is among its
// selected blocks, its rows inside the offload range.
//
// Work item = (kv head h, group of 128 / G requests, range of shared blocks).  One CTA per
// item at a time (persistent grid): a producer warp streams the range's (page, h) K and V
// slabs through a ring of tiled TMA copies (the decode's 128-byte-swizzled layout), skipping
// blocks no request of the group attends; 8 consumer warps each hold 16 query rows (16 / G
// requests x G heads) and run, per slab, S = Q K^T and O += P V on m16n8k16 bf16 MMAs (Q as
// the A operand, K and V fragments by ldmatrix) with an online softmax per row (log2 domain,
// fp32), masking every row's non-attended tokens.  A warp whose requests attend nothing in a
// slab skips it.  At the end of the item each row's partial (max, sum, unnormalised output)
// goes to the workspace, where the combine merges it with the partials of the request's own
// pages.  Every wait is bounded (SRKV_EFLAG_TIMEOUT).
#include "decode_mma.cuh"

namespace srkv {
namespace {

constexpr int kCasWarps = 8;
constexpr int kCasThreads = (kCasWarps + 1) * 32;
constexpr int kCasStages = 2;  // a stage's products outlast its copy; the query tiles need room
constexpr int kCasRows = 16 * kCasWarps;     // query rows of an item
constexpr int kCasWords = kMaxRangeBlocks / 32;  // selection bit words per request
constexpr int kChunkTokens = 64;                 // tokens of S held in registers at once
constexpr int kChunks = kBlock / kChunkTokens;

struct CasCfg {
  static constexpr int D = 128;
  static constexpr int kSlab = kBlock * D * 2;  // bf16 K or V slab: 32 KiB
  static constexpr size_t kOffK = 0;
  static constexpr size_t kOffV = kOffK + (size_t)kCasStages * kSlab;
  // per item (two buffers): request info int4 {prefix blocks, ie, ws, W}, selection bits
  // each consumer warp's query rows [16][D] bf16, chunk c of row r at c ^ (r mod 8)
  static constexpr size_t kOffQ = kOffV + (size_t)kCasStages * kSlab;
  static constexpr size_t kQWarp = 16 * D * 2;
  static constexpr size_t kOffReq = kOffQ + (size_t)kCasWarps * kQWarp;
  static constexpr size_t kReqBytes = (size_t)kCasRows * (sizeof(int4) + 4 * kCasWords);
  static constexpr size_t kOffInfo = kOffReq + 2 * kReqBytes;  // int4 per stage
  static constexpr size_t kOffBar = kOffInfo + sizeof(int4) * kCasStages;
  // full[kCasStages] (K), full_v[kCasStages], empty[kCasStages], item_free[2]
  static constexpr size_t kSmem = kOffBar + sizeof(uint64_t) * (3 * kCasStages + 2);
  static constexpr size_t kSmemAlloc = kSmem + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory opt-in limit");
};

// Stage flags (besides kNewUnit = first stage of an item, kSegEnd = last, kLast = sentinel).
constexpr uint32_t kEmptyStage = 16;  // no slab: an item with no attended block

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Item geometry: item i -> (kv head, request group, block range), ranges [rho*Ps/NR, ...).
struct Item {
  int32_t h, grp, rho, b_lo, b_hi;
};
__device__ __forceinline__ Item item_of(int64_t i, int32_t groups, int32_t NR, int32_t Ps) {
  Item it;
  it.grp = (int32_t)(i % groups);  // consecutive items read the same slabs (L2)
  const int64_t hr = i / groups;
  it.rho = (int32_t)(hr % NR);
  it.h = (int32_t)(hr / NR);
  it.b_lo = (int32_t)((int64_t)it.rho * Ps / NR);
  it.b_hi = (int32_t)((int64_t)(it.rho + 1) * Ps / NR);
  return it;
}

// Rows [e1, e2, s_lo, s_hi) of block b that request info `ri` attends: t < e1, t >= e2, or
// s_lo <= t < s_hi (its selected rows inside the offload range).
struct RowMask {
  int32_t e1, e2, s_lo, s_hi;
  __device__ __forceinline__ bool any() const { return e1 > 0 || e2 < kBlock || s_lo < s_hi; }
  __device__ __forceinline__ bool at(int32_t t) const {
    return t < e1 || t >= e2 || (t >= s_lo && t < s_hi);
  }
  // Bit i: token c0 + i of the block is attended (i < 64).
  __device__ __forceinline__ uint64_t chunk_bits(int32_t c0) const {
    return span_bits(0, e1, c0) | span_bits(e2, kBlock, c0) | span_bits(s_lo, s_hi, c0);
  }
  __device__ __forceinline__ static uint64_t span_bits(int32_t lo, int32_t hi, int32_t c0) {
    lo = lo - c0 < 0 ? 0 : (lo - c0 > 64 ? 64 : lo - c0);
    hi = hi - c0 < 0 ? 0 : (hi - c0 > 64 ? 64 : hi - c0);
    if (hi <= lo) return 0ull;
    const uint64_t upto_hi = hi == 64 ? ~0ull : (1ull << hi) - 1ull;
    return upto_hi & ~((1ull << lo) - 1ull);
  }
};
__device__ __forceinline__ int32_t clamp_row(int32_t x) {
  return x < 0 ? 0 : (x > kBlock ? kBlock : x);
}
__device__ __forceinline__ RowMask row_mask(const int4& ri, bool selected, int32_t b,
                                            int32_t INIT) {
  RowMask m;
  const int32_t base = b * kBlock;
  if (b >= ri.x) {  // not a shared block of this request (or no request): nothing
    m.e1 = 0;
    m.e2 = kBlock;
    m.s_lo = m.s_hi = 0;
    return m;
  }
  m.e1 = clamp_row(ri.y - base);
  m.e2 = clamp_row(ri.z - base);
  m.s_lo = selected ? clamp_row(INIT - base) : 0;
  m.s_hi = selected ? clamp_row(ri.w - base) : 0;
  return m;
}

// 9 warps: one sub-partition holds three of them, so a thread has at most 168 registers
// (16 K registers per sub-partition).
template <int G>
__global__ void __launch_bounds__(kCasThreads, 1)
    cascade_kernel(const DecodeArgs a, const __grid_constant__ TmaMaps maps) {
  using C = CasCfg;
  constexpr int D = C::D;
  constexpr int RPC = kCasRows / G;  // requests per item
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  int4* sInfo = reinterpret_cast<int4*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + kCasStages;
  uint64_t* empty = full_v + kCasStages;
  uint64_t* item_free = empty + kCasStages;  // [2]: the item buffer may be rewritten
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t Ps = a.prefix_blocks, NR = a.prefix_ranges;
  const int32_t groups = (a.batch + RPC - 1) / RPC;
  const int64_t items = (int64_t)a.Hkv * groups * NR;

  if (tid == 0) {
    for (int s = 0; s < kCasStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&empty[s], kCasWarps);
    }
    mbar_init(&item_free[0], kCasWarps);
    mbar_init(&item_free[1], kCasWarps);
    fence_mbar_init();
  }
  __syncthreads();
  // The split decode behind this kernel streams the requests' own pages meanwhile; every
  // input this kernel reads may be the previous kernel's output (the selection is), so wait.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == kCasWarps) {
    // ---------------------------------------------------------------- producer
    uint32_t eflags = 0;
    bool abort = false;
    int64_t it = 0, n_item = 0;
    const uint64_t once = l2_policy_evict_first();
    for (int64_t ii = blockIdx.x; ii < items && !abort; ii += gridDim.x, ++n_item) {
      const Item itm = item_of(ii, groups, NR, Ps);
      const int par = (int)(n_item & 1);
      if (n_item >= 2) {  // the consumers are through the item that used this buffer
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&item_free[par], (uint32_t)(((n_item >> 1) - 1) & 1));
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          abort = true;
          break;
        }
      }
      int4* rinfo = reinterpret_cast<int4*>(smem + C::kOffReq + par * C::kReqBytes);
      uint32_t* rsel = reinterpret_cast<uint32_t*>(rinfo + kCasRows);
      // request info: prefix blocks of the request (full shared pages), ie, ws, W
      int32_t ref_ps = 0, ref_r = -1;  // the group's request with the longest shared part
      for (int i = lane; i < RPC; i += 32) {
        const int32_t r = itm.grp * RPC + i;
        int4 ri = make_int4(0, 0, 0, 0);
        uint32_t* bits = rsel + i * kCasWords;  // this lane's request only
#pragma unroll
        for (int w = 0; w < kCasWords; ++w) bits[w] = 0u;
        if (r < a.batch) {
          uint32_t dummy = 0;
          const Geom g = make_geom(a.seq_lens[r], 0, a.max_blocks, a.kmax, a.init_tokens,
                                   a.local_tokens, dummy);
          ri = make_int4(min(Ps, g.L / kBlock), g.ie, g.ws, g.W);
          if (ri.x > ref_ps) {
            ref_ps = ri.x;
            ref_r = r;
          }
          const int64_t u = (int64_t)r * a.Hkv + itm.h;
          int32_t ns = a.nsel[u];
          ns = ns < 0 ? 0 : (ns > a.kmax ? a.kmax : ns);
          const int32_t* su = a.sel + u * a.kmax;
          for (int32_t j0 = 0; j0 < ns; j0 += 16) {  // 16 independent loads a round
            int32_t bb[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) bb[x] = j0 + x < ns ? su[j0 + x] : -1;
#pragma unroll
            for (int x = 0; x < 16; ++x)
              if (bb[x] >= itm.b_lo && bb[x] < itm.b_hi)
                bits[(bb[x] - itm.b_lo) >> 5] |= 1u << ((bb[x] - itm.b_lo) & 31);
            if (bb[15] >= itm.b_hi) break;  // ascending: the rest lies beyond the range
          }
        }
        rinfo[i] = ri;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {  // the reference request: longest shared part
        const int32_t ops = __shfl_xor_sync(0xffffffffu, ref_ps, o);
        const int32_t orr = __shfl_xor_sync(0xffffffffu, ref_r, o);
        if (ops > ref_ps || (ops == ref_ps && orr >= 0 && (ref_r < 0 || orr < ref_r))) {
          ref_ps = ops;
          ref_r = orr;
        }
      }
      __syncwarp();
      // the range's blocks in batches of 32 (lane l: block b0 + l): attended by some request
      // of the group, the page (the reference request's; every request must map the block to
      // it), and whether it is valid.  All batches first, so that the last attended block,
      // which closes the item's segment, is known before the first stage goes out.
      const int32_t b_end = min(itm.b_hi, ref_ps);
      uint32_t need_m[kCasWords];
      int32_t pages[kCasWords];
      int32_t last = -1;
#pragma unroll
      for (int k = 0; k < kCasWords; ++k) {
        const int32_t b = itm.b_lo + 32 * k + lane;
        bool need = false;
        int32_t page = -1;
        if (itm.b_lo + 32 * k >= b_end) {  // beyond the range (warp-uniform)
          pages[k] = -1;
          need_m[k] = 0u;
          continue;
        }
        if (b < b_end) {
          const int32_t bit = b - itm.b_lo;
          for (int i = 0; i < RPC && !need; ++i) {
            const bool sb = (rsel[i * kCasWords + (bit >> 5)] >> (bit & 31)) & 1u;
            need = row_mask(rinfo[i], sb, b, a.init_tokens).any();
          }
          page = a.block_table[(int64_t)ref_r * a.max_blocks + b];
        }
        // the shared-prefix contract: every request of the group that holds block b whole maps
        // it to the reference page (predicated loads, all issued before any compare)
        uint32_t bad = 0;
#pragma unroll 16
        for (int i = 0; i < RPC; ++i) {
          const int32_t r = itm.grp * RPC + i;
          const bool chk = b < b_end && r < a.batch && b < rinfo[i].x;
          const int32_t pr = chk ? a.block_table[(int64_t)r * a.max_blocks + b] : page;
          bad |= pr != page ? 1u : 0u;
        }
        if (bad) eflags |= SRKV_EFLAG_PREFIX;
        if (b < b_end) {
          if (page < 0 || (int64_t)page >= a.num_pages) {
            if (need) eflags |= SRKV_EFLAG_PAGE_RANGE;
            need = false;
          }
        }
        pages[k] = page;
        need_m[k] = __ballot_sync(0xffffffffu, need);
        if (need_m[k]) last = itm.b_lo + 32 * k + 31 - __clz(need_m[k]);
      }
      bool first = true;
#pragma unroll
      for (int k = 0; k < kCasWords; ++k) {
        for (uint32_t m = need_m[k]; m && !abort; m &= m - 1) {
          const int l = __ffs(m) - 1;
          const int32_t bl = itm.b_lo + 32 * k + l;
          const int32_t pg = __shfl_sync(0xffffffffu, pages[k], l);
          if (lane == 0) {
            const int s = (int)(it % kCasStages);
            if (it >= kCasStages &&
                !mbar_wait(&empty[s], (uint32_t)((it / kCasStages - 1) & 1))) {
              abort = true;
              eflags |= SRKV_EFLAG_TIMEOUT;
            } else {
              const uint32_t fl = (first ? kNewUnit : 0u) | (bl == last ? kSegEnd : 0u);
              sInfo[s] = make_int4(bl, par, (int32_t)fl, (int32_t)ii);
              mbar_arrive_expect_tx(&full[s], (uint32_t)C::kSlab);
              mbar_arrive_expect_tx(&full_v[s], (uint32_t)C::kSlab);
#pragma unroll
              for (int x = 0; x < 2; ++x)
                tma_load_3d(smem + C::kOffK + (size_t)s * C::kSlab + (size_t)x * kBlock * 128,
                            &maps.k, x * 64, itm.h * kBlock, pg, &full[s], once);
#pragma unroll
              for (int x = 0; x < 2; ++x)
                tma_load_3d(smem + C::kOffV + (size_t)s * C::kSlab + (size_t)x * kBlock * 128,
                            &maps.v, x * 64, itm.h * kBlock, pg, &full_v[s], once);
            }
          }
          abort = __shfl_sync(0xffffffffu, abort, 0);
          if (abort) break;
          first = false;
          ++it;
        }
      }
      if (first && !abort) {  // nothing attended: one empty stage still opens and closes it
        if (lane == 0) {
          const int s = (int)(it % kCasStages);
          if (it >= kCasStages && !mbar_wait(&empty[s], (uint32_t)((it / kCasStages - 1) & 1))) {
            abort = true;
            eflags |= SRKV_EFLAG_TIMEOUT;
          } else {
            sInfo[s] = make_int4(-1, par, (int32_t)(kNewUnit | kSegEnd | kEmptyStage), (int32_t)ii);
            mbar_arrive(&full[s]);
            mbar_arrive(&full_v[s]);
          }
        }
        abort = __shfl_sync(0xffffffffu, abort, 0);
        if (!abort) ++it;
      }
    }
    if (lane == 0) {
      const int s = (int)(it % kCasStages);
      if (!abort &&
          (it < kCasStages || mbar_wait(&empty[s], (uint32_t)((it / kCasStages - 1) & 1)))) {
        sInfo[s] = make_int4(-1, 0, (int32_t)kLast, -1);
        mbar_arrive(&full[s]);
        mbar_arrive(&full_v[s]);
        ++it;
      } else if (!abort) {
        eflags |= SRKV_EFLAG_TIMEOUT;
      }
      // every copy lands before the CTA exits (the last kCasStages stages are the latest use
      // of each stage)
      const int64_t first_i = it > kCasStages ? it - kCasStages : 0;
      for (int64_t i = first_i; i < it; ++i)
        if (!mbar_wait(&full[i % kCasStages], (uint32_t)((i / kCasStages) & 1)) ||
            !mbar_wait(&full_v[i % kCasStages], (uint32_t)((i / kCasStages) & 1))) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          break;
        }
    }
    eflags = __reduce_or_sync(0xffffffffu, eflags);
    if (lane == 0) raise_flags(a.error_flags, eflags);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int g = lane >> 2, tq = lane & 3;
  // the warp's 16 rows: row i = (request w * 16 / G + i / G of the group, head i % G)
  const int rq0 = (warp * 16 + g) / G, rq1 = (warp * 16 + g + 8) / G;  // in-group requests
  const int j0 = g % G;  // head of both rows (16 / G requests of G heads each)
  // the warp's query tile (A operand of S = Q K^T, read back with ldmatrix)
  unsigned char* qtile = smem + C::kOffQ + (size_t)warp * C::kQWarp;
  const uint32_t qbase = smem_u32(qtile);
  float o[16][4];        // O rows g, g + 8 x d = 8 nt + 2 tq, + 1
  float mrow[2], lrow[2];
  int32_t r0 = 0, r1 = 0;
  bool ok0 = false, ok1 = false;
  int4 ri0 = make_int4(0, 0, 0, 0), ri1 = ri0;
  const uint32_t* sel0 = nullptr;
  const uint32_t* sel1 = nullptr;
  Item itm{0, 0, 0, 0, 0};
  int par = 0;
  const float sl2 = a.scale_log2;
  for (int64_t it = 0;; ++it) {
    const int s = (int)(it % kCasStages);
    const uint32_t ph = (uint32_t)((it / kCasStages) & 1);
    if (!mbar_wait(&full[s], ph)) {
      if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      break;
    }
    const int4 inf = sInfo[s];
    const uint32_t fl = (uint32_t)inf.z;
    if (fl & kLast) break;
    if (fl & kNewUnit) {
      itm = item_of(inf.w, groups, NR, Ps);
      par = inf.y;
      const int4* rinfo = reinterpret_cast<const int4*>(smem + C::kOffReq + par * C::kReqBytes);
      const uint32_t* rsel = reinterpret_cast<const uint32_t*>(rinfo + kCasRows);
      r0 = itm.grp * RPC + rq0;
      r1 = itm.grp * RPC + rq1;
      ok0 = r0 < a.batch;
      ok1 = r1 < a.batch;
      ri0 = rinfo[rq0];
      ri1 = rinfo[rq1];
      sel0 = rsel + rq0 * kCasWords;
      sel1 = rsel + rq1 * kCasWords;
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
      const int64_t qrow0 = ((int64_t)r0 * a.Hq + (int64_t)itm.h * G + j0) * D;
      const int64_t qrow1 = ((int64_t)r1 * a.Hq + (int64_t)itm.h * G + j0) * D;
      // rows g and g + 8 of the tile: lane (g, tq) copies 16-byte chunks tq, tq + 4, ...
      // (the previous item's last products have read the tile: the warp is past them)
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int ch = tq + 4 * cc;  // 16-byte chunk of the row (d = 8 ch .. 8 ch + 7)
        const int4 z = make_int4(0, 0, 0, 0);
        const int4 v0 = ok0 ? *reinterpret_cast<const int4*>(q + qrow0 + 8 * ch) : z;
        const int4 v1 = ok1 ? *reinterpret_cast<const int4*>(q + qrow1 + 8 * ch) : z;
        *reinterpret_cast<int4*>(qtile + g * 256 + ((ch ^ (g & 7)) << 4)) = v0;
        *reinterpret_cast<int4*>(qtile + (g + 8) * 256 + ((ch ^ ((g + 8) & 7)) << 4)) = v1;
      }
      __syncwarp();
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
      mrow[0] = mrow[1] = -INFINITY;
      lrow[0] = lrow[1] = 0.f;
    }
    const int32_t b = inf.x;
    bool v_waited = false;
    if (!(fl & kEmptyStage)) {
      const int32_t bit = b - itm.b_lo;
      const bool s0 = ok0 && ((sel0[bit >> 5] >> (bit & 31)) & 1u);
      const bool s1 = ok1 && ((sel1[bit >> 5] >> (bit & 31)) & 1u);
      const RowMask m0 = ok0 ? row_mask(ri0, s0, b, a.init_tokens) : RowMask{0, kBlock, 0, 0};
      const RowMask m1 = ok1 ? row_mask(ri1, s1, b, a.init_tokens) : RowMask{0, kBlock, 0, 0};
      if (__any_sync(0xffffffffu, m0.any() || m1.any())) {
        const uint32_t kbase = smem_u32(smem + C::kOffK + (size_t)s * C::kSlab);
        const uint32_t vbase = smem_u32(smem + C::kOffV + (size_t)s * C::kSlab);
        const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix, row within it
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {  // kChunkTokens-token chunks
          // ---- S = Q K^T over the chunk's tokens: kChunkTokens / 8 n-tiles of 8 tokens
          float sacc[kChunkTokens / 8][4];
#pragma unroll
          for (int nt = 0; nt < kChunkTokens / 8; ++nt)
            sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
          // k-steps outside, n-tiles inside: one Q fragment per k-step feeds every n-tile,
          // and the kChunkTokens / 8 accumulators are independent chains
          const int qr = lane & 15;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // Q fragment: matrices (rows 0-7, d 16kk..), (rows 8-15, same), (rows 0-7, d
            // 16kk + 8..), (rows 8-15, same); lane l addresses row (l & 15)
            uint32_t qa[4];
            const int qch = 2 * kk + (lane >> 4);
            ldsm_x4(qbase + qr * 256 + ((qch ^ (qr & 7)) << 4), qa);
#pragma unroll
            for (int np = 0; np < kChunkTokens / 16; ++np) {  // pairs of n-tiles
              const int tok = kChunkTokens * c + 16 * np + (mi >> 1) * 8 + mr;
              uint32_t kb[4];
              ldsm_x4(kbase + swz(tok, 2 * kk + (mi & 1)), kb);
              mma_16816(sacc[2 * np], qa[0], qa[1], qa[2], qa[3], kb[0], kb[1]);
              mma_16816(sacc[2 * np + 1], qa[0], qa[1], qa[2], qa[3], kb[2], kb[3]);
            }
          }
          // ---- mask, online softmax (log2 domain) for rows g (x = 0) and g + 8 (x = 1): the
          // attended tokens of the chunk as bit masks; a chunk whole for every row of the
          // warp (the common case: initial, window and selected blocks are attended whole)
          // needs no per-token test
          static_assert(kChunkTokens <= 64, "a chunk's attended tokens fit one 64-bit mask");
          constexpr uint64_t kWhole = kChunkTokens == 64 ? ~0ull : (1ull << kChunkTokens) - 1ull;
          const uint64_t cb0 = m0.chunk_bits(kChunkTokens * c);
          const uint64_t cb1 = m1.chunk_bits(kChunkTokens * c);
          float mx[2] = {-INFINITY, -INFINITY};
          if (__all_sync(0xffffffffu, (cb0 & cb1 & kWhole) == kWhole)) {
#pragma unroll
            for (int nt = 0; nt < kChunkTokens / 8; ++nt) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                sacc[nt][e] *= sl2;
                sacc[nt][2 + e] *= sl2;
                mx[0] = fmaxf(mx[0], sacc[nt][e]);
                mx[1] = fmaxf(mx[1], sacc[nt][2 + e]);
              }
            }
          } else {
            const uint64_t lb0 = cb0 >> (2 * tq), lb1 = cb1 >> (2 * tq);
#pragma unroll
            for (int nt = 0; nt < kChunkTokens / 8; ++nt) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const uint64_t bit = 1ull << (8 * nt + e);
                sacc[nt][e] = (lb0 & bit) ? sacc[nt][e] * sl2 : -INFINITY;
                sacc[nt][2 + e] = (lb1 & bit) ? sacc[nt][2 + e] * sl2 : -INFINITY;
                mx[0] = fmaxf(mx[0], sacc[nt][e]);
                mx[1] = fmaxf(mx[1], sacc[nt][2 + e]);
              }
            }
          }
          float alpha[2], base[2];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], 1));
            mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], 2));
            const float mn = fmaxf(mrow[x], mx[x]);
            base[x] = mn == -INFINITY ? 0.f : mn;
            alpha[x] = fast_exp2(mrow[x] - base[x]);
            mrow[x] = mn;
            lrow[x] *= alpha[x];
          }
          if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {  // a new max
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
              o[nt][0] *= alpha[0];
              o[nt][1] *= alpha[0];
              o[nt][2] *= alpha[1];
              o[nt][3] *= alpha[1];
            }
          }
          // P as the A operand: k16 step j covers n-tiles 2j, 2j + 1 (bf16, as the MMA sees it)
          uint32_t pa[kChunkTokens / 16][4];
#pragma unroll
          for (int j = 0; j < kChunkTokens / 16; ++j) {
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const int nt = 2 * j + hlf;
              const uint32_t p0 = pack_bf16(fast_exp2(sacc[nt][0] - base[0]),
                                            fast_exp2(sacc[nt][1] - base[0]));
              const uint32_t p1 = pack_bf16(fast_exp2(sacc[nt][2] - base[1]),
                                            fast_exp2(sacc[nt][3] - base[1]));
              lrow[0] += bf16_lo(p0) + bf16_hi(p0);
              lrow[1] += bf16_lo(p1) + bf16_hi(p1);
              pa[j][2 * hlf] = p0;
              pa[j][2 * hlf + 1] = p1;
            }
          }
          // ---- O += P V, once V has landed
          if (!v_waited) {
            if (!mbar_wait(&full_v[s], ph)) {
              if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
              return;
            }
            v_waited = true;
          }
#pragma unroll
          for (int j = 0; j < kChunkTokens / 16; ++j) {
            const int tok = kChunkTokens * c + 16 * j + (mi & 1) * 8 + mr;
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {  // pairs of d n-tiles
              uint32_t vb[4];
              ldsm_x4_trans(vbase + swz(tok, 2 * dp + (mi >> 1)), vb);
              mma_16816(o[2 * dp], pa[j][0], pa[j][1], pa[j][2], pa[j][3], vb[0], vb[1]);
              mma_16816(o[2 * dp + 1], pa[j][0], pa[j][1], pa[j][2], pa[j][3], vb[2], vb[3]);
            }
          }
        }
      }
    }
    if (!v_waited && !(fl & kEmptyStage)) {  // V's copy must land before the stage is reused
      if (!mbar_wait(&full_v[s], ph)) {
        if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
        break;
      }
    }
    warp_arrive(&empty[s]);
    if (fl & kSegEnd) {
      // the item's partial for the warp's rows: (max, sum, unnormalised output)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        lrow[x] += __shfl_xor_sync(0xffffffffu, lrow[x], 1);
        lrow[x] += __shfl_xor_sync(0xffffffffu, lrow[x], 2);
      }
      float* accw = reinterpret_cast<float*>(a.ws + a.lay.acc);
      float* mlw = reinterpret_cast<float*>(a.ws + a.lay.ml);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const bool okx = x == 0 ? ok0 : ok1;
        if (!okx) continue;
        const int32_t r = x == 0 ? r0 : r1;
        const int64_t slot = a.lay.cascade + ((int64_t)r * a.Hkv + itm.h) * NR + itm.rho;
        float* accp = accw + (slot * G + j0) * D;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<float2*>(accp + 8 * nt + 2 * tq) =
              make_float2(o[nt][2 * x], o[nt][2 * x + 1]);
        if (tq == 0) {
          mlw[(slot * G + j0) * 2] = mrow[x];
          mlw[(slot * G + j0) * 2 + 1] = lrow[x];
        }
      }
      warp_arrive(&item_free[par]);
    }
  }
}

}  // namespace

bool cascade_supported(const srkv_config& cfg) {
  const int32_t G = cfg.num_q_heads / cfg.num_kv_heads;
  return cfg.dtype == SRKV_BF16 && cfg.head_dim == 128 && (G == 1 || G == 2 || G == 4 || G == 8);
}

// The split decode behind the cascade streams the requests' own pages (bound by bytes); the
// cascade runs the shared pages' products (bound by the tensor pipe).  On the 64-request,
// 16384-token shared-prefix batch, 3/8 of the SMs for the cascade balanced the two best
// (363 us against 474 us with a quarter and 409 us with a third).
int32_t cascade_ctas(int32_t sm_count) { return sm_count * 3 / 8; }

cudaError_t launch_cascade(const DecodeArgs& a, bool pdl, cudaStream_t stream) {
  using C = CasCfg;
  static bool configured[128][4] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  const int gi = a.G == 8 ? 3 : a.G == 4 ? 2 : a.G == 2 ? 1 : 0;
  void (*kern)(const DecodeArgs, const TmaMaps) =
      a.G == 8 ? cascade_kernel<8> : a.G == 4 ? cascade_kernel<4>
                                              : a.G == 2 ? cascade_kernel<2> : cascade_kernel<1>;
  if (!configured[dev][gi]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured[dev][gi] = true;
  }
  TmaMaps maps;
  if (!encode_cache_map(&maps.k, a.k_cache, a.num_pages, a.Hkv, 128, false) ||
      !encode_cache_map(&maps.v, a.v_cache, a.num_pages, a.Hkv, 128, false))
    return cudaErrorInvalidValue;
  if (pdl)
    return launch_pdl(kern, dim3((unsigned)a.cascade_ctas), dim3(kCasThreads), C::kSmemAlloc,
                      stream, a, maps);
  kern<<<(unsigned)a.cascade_ctas, kCasThreads, C::kSmemAlloc, stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace srkv
