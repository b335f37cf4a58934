// select.cuh -- top-k selection of (request, kv head) units on a thread-block cluster,
// shared by the scoring kernel and the fused small-batch decode.
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Overall Solution": sparse retrieval computes the inner product of the current query with
// every representation vector and keeps the topK closest blocks.  Scores become
// order-preserving 32-bit keys (NaN and out-of-range pages rank lowest); the k largest keys
// are kept, equal keys going to the lower block index, written in ascending block order.
//
//   score_share: one warp per candidate, q_bar . rep in fp32 (fixed lane order); the key is
//                stored into the leader CTA's shared memory and counted into the leader's
//                histogram of the top 8 key bits (or of the top 12 and the top 8), through
//                distributed shared memory;
//   warp_boundary: from the 8- and 12-bit histograms, the 12-bit bin holding the k-th key
//                (the fused decode ranks that bin with one warp when it is small);
//   radix_narrow: MSB-first radix passes of 8 bits (the first from the 8-bit histogram)
//                until the bin holding the k-th key has at most 32 keys (or four passes,
//                when the k-th key is known exactly);
//   finish_fast: one warp ranks that bin (score, then lower block); a kept key's output slot
//                is the number of kept keys before it in block order, from ballot counts.
#pragma once

#include "srkv_internal.cuh"

namespace srkv {

__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;            // NaN ranks below everything
  if (s == 0.0f) s = 0.0f;          // -0 and +0 tie
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the warp of one int per lane; *total gets the sum.
__device__ __forceinline__ int32_t warp_exclusive_scan(int32_t v, int lane, int32_t* total) {
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Store to the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_u32(uint32_t* local, uint32_t rank, uint32_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
// 16-byte store to the same shared-memory offset in CTA `rank` (16-byte aligned).
__device__ __forceinline__ void st_cluster_int4(int4* local, uint32_t rank, int4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
// Address of the same shared-memory offset in CTA `rank`, for the shared::cluster forms.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  return remote;
}
// Asynchronous 16- / 8-byte stores into another CTA's shared memory (shared::cluster
// addresses) that count their bytes on an mbarrier of that CTA when they land.
__device__ __forceinline__ void st_async_f4(uint32_t remote, float4 v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
      : "memory");
}
__device__ __forceinline__ void st_async_f2(uint32_t remote, float2 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(remote), "f"(v.x), "f"(v.y), "r"(remote_bar)
               : "memory");
}
// Atomic add to the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ void red_cluster_add(int32_t* local, uint32_t rank, int32_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
// Atomic add to the same shared-memory offset in CTA `rank`, returning the old value.
__device__ __forceinline__ uint32_t atom_cluster_add(uint32_t* local, uint32_t rank, uint32_t v) {
  uint32_t remote, old;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(remote), "r"(v) : "memory");
  return old;
}
// Load of the int2 at the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ int2 ld_cluster_int2(const int2* local, uint32_t rank) {
  uint32_t remote;
  int2 v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival that orders nothing: for a thread whose earlier accesses to other CTAs were all
// observed already (through an mbarrier those CTAs waited on).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Every warp finds the digit holding the remaining-th largest key from a 256-bin histogram.
__device__ __forceinline__ void find_digit(const int32_t* hist, int lane, int32_t remaining,
                                           int32_t* digit, int32_t* rem_out, int32_t* cnt_out) {
  int32_t c[8], local = 0;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    c[b] = hist[lane * 8 + b];
    local += c[b];
  }
  int32_t suffix = local;  // keys in this lane's bins and above
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_down_sync(0xffffffffu, suffix, o);
    if (lane + o < 32) suffix += y;
  }
  int32_t above = suffix - local, dg = -1, rm = 0, cn = 0;
#pragma unroll
  for (int b = 7; b >= 0; --b) {
    if (above < remaining && above + c[b] >= remaining) {
      dg = lane * 8 + b;
      rm = remaining - above;
      cn = c[b];
    }
    above += c[b];
  }
  const uint32_t who = __ballot_sync(0xffffffffu, dg >= 0);
  const int src = __ffs(who) - 1;
  *digit = __shfl_sync(0xffffffffu, dg, src);
  *rem_out = __shfl_sync(0xffffffffu, rm, src);
  *cnt_out = __shfl_sync(0xffffffffu, cn, src);
}

constexpr int kFastRounds = 4;  // finish_fast handles n <= 4 * (selecting threads)

// Distributed-shared-memory helpers.
__device__ __forceinline__ void* map_cluster_ptr(void* local, uint32_t rank) {
  void* remote;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(remote) : "l"(local), "r"(rank));
  return remote;
}
// Arrives on the mbarrier at the same offset in CTA `rank`, releasing this thread's prior
// memory accesses at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}
// The same, counting `n` arrivals.
__device__ __forceinline__ void mbar_arrive_cluster_n(uint64_t* local, uint32_t rank, uint32_t n) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(remote),
               "r"(n)
               : "memory");
}
// Waits (bounded, acquire at cluster scope) for the phase with the given parity.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Scores candidates [s_lo, i_hi) of unit (r, h), one warp per candidate, 8 candidates of a
// warp in one round of loads; lane x of the warp stores its x-th key into the leader's
// keys[i] and counts it into the leader's histogram of the top kHistBits key bits, hist
// (and, with leader_coarse, into that of the top 8 bits; with leader_pages, the
// candidate's page into the leader's pages[i]).  `pages` holds the share's pages at
// [i - s_lo].  issued() runs once, right after the warp's first round of vector loads has
// been issued (before any of them is used; it may wait, e.g. for the cluster barrier that
// makes the leader's shared memory safe to write).  Returns the error flags seen (pages out
// of range).
//
// stored(n) runs on lane 0 of the warp once the warp's lanes have written the round's n >= 1
// keys (after a warp barrier that orders their writes before it, e.g. to release them all
// with one arrival).
// kHistBits: the histogram counts the top kHistBits bits of the keys (2^kHistBits bins).
template <int D, int kWarps, int kHistBits = 8, int UNROLL = 8, typename Issued,
          typename Stored>
__device__ __forceinline__ uint32_t score_share(const float* qbar, const int32_t* pages,
                                                int32_t s_lo, int32_t i_hi, const float* reps,
                                                int64_t num_pages, int32_t Hkv, int32_t h,
                                                uint32_t* leader_keys, int32_t* leader_hist,
                                                int32_t* leader_coarse, int32_t* leader_pages,
                                                int warp, int lane,
                                                Issued issued, Stored stored) {
  constexpr int EPL = D / 32;  // elements per lane: 4 (d 128) or 2 (d 64)
  uint32_t eflags = 0;
  float qv[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] = qbar[lane * EPL + e];
  const uint64_t keep = l2_policy_evict_last();  // the vectors are read again every step
  static_assert(UNROLL <= 32, "lane x holds candidate x of the round");
  bool first = true;
  for (int32_t i0 = s_lo + warp; i0 < i_hi; i0 += kWarps * UNROLL) {
    float part[UNROLL];
    bool ok[UNROLL];
    float4 v[UNROLL];
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {  // every load of the round first
      const int32_t i = i0 + x * kWarps;
      ok[x] = false;
      v[x] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < i_hi) {
        const int32_t page = pages[i - s_lo];
        ok[x] = page >= 0 && (int64_t)page < num_pages;
        if (ok[x]) {
          const float* rep = reps + ((int64_t)page * Hkv + h) * D + lane * EPL;
          if constexpr (EPL == 4) {
            v[x] = ldg_f4_hint(rep, keep);
          } else {
            const float2 w = ldg_f2_hint(rep, keep);
            v[x].x = w.x;
            v[x].y = w.y;
          }
        }
      }
    }
    if (first) issued();
    first = false;
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {
      if constexpr (EPL == 4)
        part[x] = qv[0] * v[x].x + qv[1] * v[x].y + qv[2] * v[x].z + qv[3] * v[x].w;
      else
        part[x] = qv[0] * v[x].x + qv[1] * v[x].y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int x = 0; x < UNROLL; ++x) part[x] += __shfl_xor_sync(0xffffffffu, part[x], o);
    float mine = part[0];
    bool mine_ok = ok[0];
#pragma unroll
    for (int x = 1; x < UNROLL; ++x)
      if (lane == x) {
        mine = part[x];
        mine_ok = ok[x];
      }
    const int32_t i = i0 + lane * kWarps;
    const bool valid = lane < UNROLL && i < i_hi;
    if (valid && !mine_ok) eflags |= SRKV_EFLAG_PAGE_RANGE;
    const uint32_t key = mine_ok ? score_key(mine) : 0u;
    if (valid) {
      st_cluster_u32(&leader_keys[i], 0, key);
      if (leader_pages)
        st_cluster_u32(reinterpret_cast<uint32_t*>(&leader_pages[i]), 0,
                       (uint32_t)pages[i - s_lo]);
    }
    const uint32_t digit = valid ? key >> (32 - kHistBits) : 0xffffffffu;
    const uint32_t peers = __match_any_sync(0xffffffffu, digit);
    if (valid && lane == __ffs(peers) - 1) {
      red_cluster_add(&leader_hist[digit], 0, __popc(peers));
      if (kHistBits > 8 && leader_coarse)
        red_cluster_add(&leader_coarse[digit >> (kHistBits - 8)], 0, __popc(peers));
    }
    const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    __syncwarp();
    if (lane == 0 && nvalid > 0) stored(nvalid);
  }
  return __reduce_or_sync(0xffffffffu, eflags);
}

// Where the radix passes stop: keys with (key & pmask) == prefix form the boundary bin, of
// which `remaining` are kept; `ranked`: the bin has at most 32 keys (else the bin is the
// keys equal to the k-th, kept lowest blocks first).
struct RadixState {
  uint32_t prefix, pmask;
  int32_t remaining;
  bool ranked;
};

// hist[0] holds the histogram of the top 8 bits of keys[0, n); hist[1], hist[2] are zero.
// Every selecting thread (tid < kThreads) calls it; bar() synchronises them.
template <int kThreads, typename Bar>
__device__ __forceinline__ RadixState radix_narrow(const uint32_t* keys, int32_t n, int32_t k,
                                                   int32_t (*hist)[256], int tid, Bar bar) {
  constexpr int kWarps = kThreads / 32;
  const int lane = tid & 31, warp = tid >> 5;
  RadixState rs;
  rs.prefix = 0;
  rs.pmask = 0;
  rs.remaining = k;
  rs.ranked = false;
  (void)kWarps;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int32_t* hcur = hist[pass % 3];
    if (pass > 0) {
      for (int i = tid; i < 256; i += kThreads) hist[(pass + 1) % 3][i] = 0;
      for (int32_t i0 = warp * 32; i0 < n; i0 += kThreads) {
        const int32_t i = i0 + lane;
        const uint32_t kk = i < n ? keys[i] : 0u;
        const bool in = i < n && (kk & rs.pmask) == rs.prefix;
        const uint32_t digit = in ? (kk >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&hcur[digit], __popc(peers));
      }
      bar();
    }
    int32_t dg, rm, cnt;
    find_digit(hcur, lane, rs.remaining, &dg, &rm, &cnt);
    rs.prefix |= (uint32_t)dg << shift;
    rs.pmask |= 0xffu << shift;
    rs.remaining = rm;
    if (pass < 3 && cnt <= 32) {  // uniform: every warp read the same histogram
      rs.ranked = true;
      break;
    }
  }
  return rs;
}

// Where the k-th largest key lies, from the histograms of the top 8 key bits (coarse, 256
// bins) and of the top 12 (fine, 4096 bins) of the same keys: the fine bin (digit), the keys
// in higher fine bins (above) and in the bin (cnt).  One warp; every lane gets the result.
// 1 <= k <= the histograms' total (else the bin reported holds INT32_MAX keys).
struct Boundary {
  int32_t digit, above, cnt;
};
__device__ __forceinline__ Boundary warp_boundary(const int32_t* coarse, const int32_t* fine,
                                                  int32_t k, int lane) {
  Boundary bd;
  bd.digit = 0;
  bd.above = 0;
  bd.cnt = INT32_MAX;
  int32_t d8, rem, cnt8;
  find_digit(coarse, lane, k, &d8, &rem, &cnt8);  // rem: keys to take from coarse bin d8
  if (d8 < 0) return bd;
  // lane j < 16 holds fine bin 16 d8 + 15 - j: the bins from the top down
  const int32_t c = lane < 16 ? fine[16 * d8 + 15 - lane] : 0;
  int32_t pre = c;  // keys in this lane's bin and the higher ones of the coarse bin
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, pre, o);
    if (lane >= o) pre += y;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, lane < 16 && pre >= rem);
  if (hit == 0u) return bd;
  const int j = __ffs(hit) - 1;
  bd.digit = 16 * d8 + 15 - j;
  bd.cnt = __shfl_sync(0xffffffffu, c, j);
  bd.above = k - rem + __shfl_sync(0xffffffffu, pre, j) - bd.cnt;
  return bd;
}

// Scratch of finish_fast.
template <int kThreads>
struct FinishShared {
  int32_t bnd_idx[32];
  int32_t wcnt[2][kFastRounds * (kThreads / 32)];  // per (round, warp): above / in the bin
  uint32_t take;
};

// n <= kFastRounds * kThreads.  A key above the boundary bin is kept; inside the bin, taken
// in block order, the ranked ones are kept, or (not ranked) the first `remaining`.  A kept
// key's output slot = kept keys before it in block order = keys above the bin before it +
// kept bin keys before it.  emit(slot, i) for every kept candidate i; returns the count.
template <int kThreads, typename Bar, typename Emit>
__device__ __forceinline__ int32_t finish_fast(const uint32_t* keys, int32_t n,
                                               const RadixState& rs, FinishShared<kThreads>& fs,
                                               int tid, Bar bar, Emit emit) {
  constexpr int kWarps = kThreads / 32;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t b_above[kFastRounds], b_in[kFastRounds];
#pragma unroll
  for (int rr = 0; rr < kFastRounds; ++rr) {
    const int32_t i = rr * kThreads + tid;
    const uint32_t hi = i < n ? keys[i] & rs.pmask : 0u;
    b_above[rr] = __ballot_sync(0xffffffffu, i < n && hi > rs.prefix);
    b_in[rr] = __ballot_sync(0xffffffffu, i < n && hi == rs.prefix);
    if (lane == 0) {
      fs.wcnt[0][rr * kWarps + warp] = __popc(b_above[rr]);
      fs.wcnt[1][rr * kWarps + warp] = __popc(b_in[rr]);
    }
  }
  bar();
  // exclusive prefixes over (round, warp) in block order: lane j holds entry j
  constexpr int kEntries = kFastRounds * kWarps;
  static_assert(kEntries <= 32, "one warp scans the per-(round, warp) counts");
  int32_t tot_above, tot_in;
  const int32_t pa = warp_exclusive_scan(lane < kEntries ? fs.wcnt[0][lane] : 0, lane, &tot_above);
  const int32_t pi = warp_exclusive_scan(lane < kEntries ? fs.wcnt[1][lane] : 0, lane, &tot_in);
  const uint32_t lt = (1u << lane) - 1u;
  int32_t t_in[kFastRounds], a_before[kFastRounds];
#pragma unroll
  for (int rr = 0; rr < kFastRounds; ++rr) {
    t_in[rr] = __shfl_sync(0xffffffffu, pi, rr * kWarps + warp) + __popc(b_in[rr] & lt);
    a_before[rr] = __shfl_sync(0xffffffffu, pa, rr * kWarps + warp) + __popc(b_above[rr] & lt);
  }
  uint32_t take_mask = 0;
  if (rs.ranked) {  // tot_in <= 32
#pragma unroll
    for (int rr = 0; rr < kFastRounds; ++rr)
      if ((b_in[rr] >> lane) & 1u) fs.bnd_idx[t_in[rr]] = rr * kThreads + tid;
    bar();
    if (warp == 0) {
      const uint32_t key = lane < tot_in ? keys[fs.bnd_idx[lane]] : 0u;
      int32_t rank = 0;  // higher score, or equal score and lower block (lane)
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
        rank += j < tot_in && (kj > key || (kj == key && j < lane));
      }
      const uint32_t m = __ballot_sync(0xffffffffu, lane < tot_in && rank < rs.remaining);
      if (lane == 0) fs.take = m;
    }
    bar();
    take_mask = fs.take;
  }
#pragma unroll
  for (int rr = 0; rr < kFastRounds; ++rr) {
    const int32_t t = t_in[rr];
    const int32_t bin_before =
        rs.ranked ? __popc(t < 32 ? take_mask & ((1u << t) - 1u) : take_mask)
                  : min(t, rs.remaining);
    const bool take = ((b_above[rr] >> lane) & 1u) ||
                      (((b_in[rr] >> lane) & 1u) &&
                       (rs.ranked ? ((take_mask >> t) & 1u) != 0 : t < rs.remaining));
    if (take) emit(a_before[rr] + bin_before, rr * kThreads + tid);
  }
  return tot_above + (rs.ranked ? __popc(take_mask) : min(tot_in, rs.remaining));
}

}  // namespace srkv
