// decode_plan.cuh -- how the split grid divides the attended pages of all units.
//
// The attended set of a (request, kv head) unit (openGauss DataVec page, "Overall
// Solution": the selected blocks are concatenated with initial_tokens and the
// sliding_window) is walked as two page lists:
//   list A: the initial-token blocks [0, a) and the window blocks [wstart, nb), reading
//           only their initial / window rows.  It depends on the sequence length alone, so
//           it can be streamed before the selection exists;
//   list B: the selected blocks, reading only their rows inside the offload range
//           [INIT, W).  A selected block that also holds initial or window tokens (the
//           window start is not page-aligned) is read by both lists, each for its own rows:
//           the two row sets are disjoint and their union is the attended set.
// Flash-decoding style split (KV-cache survey "大模型推理百倍加速之KV cache篇", section
// "Share--KV cache共享": partial results are merged like Flash-Decoding): the lists of all
// units are concatenated in unit order, T positions per list, and CTA c of C takes
// positions [c*T/C, (c+1)*T/C) of each list, so every SM gets the same number of pages
// whatever the request lengths.  A CTA writes one partial (max, sum, unnormalised output)
// per unit its range touches, into slot u + c of the list's bank: along the staircase of
// (unit, CTA) pairs each step raises u or c, so the slot is unique.
#pragma once

#include "srkv_internal.cuh"

namespace srkv {

constexpr int kListA = 0, kListB = 1;

// Blocks below g.pb (a shared prefix, attended by the cascade kernel) are left out of list A:
// its initial blocks are [pb, a), its window blocks [max(wstart, pb), nb).
__device__ __forceinline__ int32_t list_a_count(const Geom& g) {
  const int32_t ia = g.a > g.pb ? g.a - g.pb : 0;
  return ia + (g.nb - (g.wstart > g.pb ? g.wstart : g.pb));
}

// Position j of list A: the page and the rows to read (init / window rows only).
__device__ __forceinline__ PageTask resolve_a(const Geom& g, int32_t j, const int32_t* bt_r,
                                              int64_t num_pages, uint32_t& eflags) {
  PageTask t;
  t.page = -1;
  t.block = -1;
  t.lo = t.hi = t.ie = t.ws = 0;
  const int32_t ia = g.a > g.pb ? g.a - g.pb : 0;
  const int32_t b = j < ia ? g.pb + j : (g.wstart > g.pb ? g.wstart : g.pb) + (j - ia);
  const int32_t base = b * kBlock;
  const int32_t cnt = min(kBlock, g.L - base);
  const int32_t ie = min(max(g.ie - base, 0), cnt);
  const int32_t ws = min(max(g.ws - base, 0), cnt);
  const int32_t lo = ie > 0 ? 0 : ws;
  const int32_t hi = ws < cnt ? cnt : ie;
  if (lo >= hi) return t;
  const int32_t page = bt_r[b];
  if (page < 0 || (int64_t)page >= num_pages) {
    eflags |= SRKV_EFLAG_PAGE_RANGE;
    return t;
  }
  t.page = page;
  t.block = b;
  t.lo = lo;
  t.hi = hi;
  t.ie = ie;
  t.ws = ws;
  return t;
}

// Position i of list B: selected block sel_u[i], rows inside [INIT, W).  Entries that are
// not candidates or not ascending are skipped and flagged.
__device__ __forceinline__ PageTask resolve_b(const Geom& g, int32_t i, const int32_t* sel_u,
                                              const int32_t* bt_r, int64_t num_pages,
                                              int32_t INIT, uint32_t& eflags) {
  PageTask t;
  t.page = -1;
  t.block = -1;
  t.lo = t.hi = t.ie = t.ws = 0;
  const int32_t b = sel_u[i];
  if (!is_candidate(b, INIT, g.W) || (i > 0 && sel_u[i - 1] >= b)) {
    eflags |= SRKV_EFLAG_SELECTION;
    return t;
  }
  if (b < g.pb) return t;  // a shared-prefix block: the cascade kernel attends it
  const int32_t base = b * kBlock;
  const int32_t cnt = min(kBlock, g.L - base);
  const int32_t lo = max(INIT - base, 0);
  const int32_t hi = min(g.W - base, cnt);
  if (lo >= hi) return t;
  const int32_t page = bt_r[b];
  if (page < 0 || (int64_t)page >= num_pages) {
    eflags |= SRKV_EFLAG_PAGE_RANGE;
    return t;
  }
  t.page = page;
  t.block = b;
  t.lo = lo;
  t.hi = hi;
  t.ie = hi;  // every loaded row is attended
  t.ws = hi;
  return t;
}

// Selection count of unit u: read from nsel, or, when the scoring kernel is still running
// (early), the count it is bound to write (selection_count), from the lengths alone.
__device__ __forceinline__ int32_t nsel_of(const DecodeArgs& a, int32_t u) {
  if (!a.early) return a.nsel[u];
  const int32_t r = u / a.Hkv;
  const int32_t L = a.seq_lens[r];
  const int32_t prompt = a.prompt_lens ? a.prompt_lens[r] : L;
  return selection_count(L, prompt, a.max_blocks, a.kmax, a.init_tokens, a.local_tokens,
                         a.dense_boundary, a.topk_percent)
      .k;
}

__device__ __forceinline__ Geom unit_geom(const DecodeArgs& a, int32_t u, uint32_t& eflags) {
  Geom g = make_geom(a.seq_lens[u / a.Hkv], nsel_of(a, u), a.max_blocks, a.kmax, a.init_tokens,
                     a.local_tokens, eflags);
  g.pb = prefix_of(g, a.prefix_blocks);
  return g;
}

// Geometry without the selection count (list A, readable before the selection exists).
__device__ __forceinline__ Geom unit_geom_a(const DecodeArgs& a, int32_t u, uint32_t& eflags) {
  Geom g = make_geom(a.seq_lens[u / a.Hkv], 0, a.max_blocks, a.kmax, a.init_tokens,
                     a.local_tokens, eflags);
  g.pb = prefix_of(g, a.prefix_blocks);
  return g;
}

__device__ __forceinline__ int32_t list_count(const DecodeArgs& a, int list, int32_t u,
                                              uint32_t& eflags) {
  if (list == kListA) return list_a_count(unit_geom_a(a, u, eflags));
  int32_t ns = nsel_of(a, u);
  if (ns < 0 || ns > a.kmax) {
    eflags |= SRKV_EFLAG_SELECTION;
    ns = ns < 0 ? 0 : a.kmax;
  }
  return ns;
}

struct ListRange {
  int64_t T;      // positions of the list over all units
  int64_t begin;  // this CTA's first position
  int64_t end;    // one past its last
  int32_t u0;     // unit holding `begin`
  int64_t base0;  // first position of unit u0
};

// Warp-level plan of one list for CTA `c` of `C`; every lane returns the same range.  When
// `offsets` is not null the list's unit offsets [U + 1] are written (used by the combine).
// When `prefix` is not null, prefix[k] receives the first position of the units of lane k's
// chunk (chunk = ceil(U / 32) units) and prefix[32] the total.
__device__ __forceinline__ ListRange warp_plan(const DecodeArgs& a, int list, int64_t c,
                                               int64_t C, int64_t* offsets, int64_t* prefix,
                                               uint32_t& eflags) {
  const int lane = threadIdx.x & 31;
  const int32_t U = a.batch * a.Hkv;
  const int32_t chunk = (U + 31) / 32;
  const int32_t u_lo = min(U, lane * chunk), u_hi = min(U, u_lo + chunk);
  int64_t local = 0;
  for (int32_t u = u_lo; u < u_hi; ++u) local += list_count(a, list, u, eflags);
  int64_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int64_t excl = incl - local;
  ListRange rg;
  rg.T = __shfl_sync(0xffffffffu, incl, 31);
  if (prefix) {
    prefix[lane] = excl;
    if (lane == 31) prefix[32] = rg.T;
  }
  rg.begin = cta_begin(c < C ? c : C, rg.T, C);  // a CTA c >= C has no position
  rg.end = cta_begin(c < C ? c + 1 : C, rg.T, C);
  int32_t u0 = 0;
  int64_t base0 = 0;
  const bool mine = rg.begin < rg.end && excl <= rg.begin && rg.begin < excl + local;
  if (mine || offsets) {
    int64_t pos = excl;
    uint32_t dummy = 0;
    bool found = false;
    for (int32_t u = u_lo; u < u_hi; ++u) {
      const int32_t n = list_count(a, list, u, dummy);
      if (offsets) offsets[u] = pos;
      if (mine && !found && rg.begin < pos + n) {
        u0 = u;
        base0 = pos;
        found = true;
      }
      pos += n;
    }
    if (offsets && lane == 31) offsets[U] = rg.T;
  }
  const uint32_t who = __ballot_sync(0xffffffffu, mine);
  const int src = who ? __ffs(who) - 1 : 0;
  rg.u0 = __shfl_sync(0xffffffffu, u0, src);
  rg.base0 = __shfl_sync(0xffffffffu, base0, src);
  return rg;
}

}  // namespace srkv
