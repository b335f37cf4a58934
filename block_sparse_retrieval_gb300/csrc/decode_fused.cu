// decode_fused.cu -- block-sparse retrieval decode of a small batch in one kernel.
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Overall Solution": the query is scored against every offload block's representation
// vector, the topK closest blocks are kept and attended together with the initial tokens and
// the sliding window; the KV-cache survey ("Share--KV cache共享") merges partial attention
// results the Flash-Decoding way.  Here one thread-block cluster does all of it for one
// (request, kv head) unit, so nothing crosses a kernel boundary or global memory between
// the steps:
//   * every CTA scores its share of the candidates (select.cuh: keys, page ids and the
//     histograms of the top 12 and top 8 key bits go to the leader, CTA 0, through
//     distributed shared memory); the shares split the most candidates the block table
//     allows, so the table entries load alongside the request's length;
//   * meanwhile the other CTAs' producer warps stream their share of the initial and window
//     pages (list A) into the stage ring (decode_mma.cuh), through the scoring and the
//     selection;
//   * the leader selects: one warp finds the 12-bit bin holding the k-th largest key; the 8
//     warps lay every key above it out as the pool of kept blocks (page and block ids) in
//     the leader's shared memory, a round of 32 keys each in turn; one warp ranks the bin's
//     few keys for the rest; the warps release each streaming CTA with its first kStatic
//     pool entries (written into that CTA's shared memory) and an mbarrier arrival; sel /
//     nsel are written after that.  A bin too large to rank at once falls back to radix
//     narrowing and the ordered finish;
//   * each streaming CTA attends its share of list A, then its kStatic entries, then takes
//     kept blocks from the rest of the pool one at a time (an atomic counter in the leader's
//     shared memory) until it is empty, so the CTAs whose pages arrive sooner take more and
//     all finish within about one page of each other; the merged partial (max, sum,
//     unnormalised output) of the whole segment goes into the leader's shared memory;
//   * the leader merges the partials and writes the output.
// The partials land with asynchronous stores that count their bytes on one mbarrier of the
// leader.  Every wait is bounded (SRKV_EFLAG_TIMEOUT); every thread ends at one cluster
// barrier, so no CTA leaves while another may still reach its shared memory (the leader's
// consumers arrive on it as soon as every partial has landed, before they merge).
#include "decode_mma.cuh"
#include "select.cuh"

namespace srkv {
namespace {

constexpr int kSelThreads = kConsumerWarps * 32;  // the consumer warps score and select
constexpr int32_t kMaxCand = kFastRounds * kSelThreads;  // candidates per unit (1024)
constexpr int kMaxShare = 256;                             // candidates scored per CTA
constexpr int kMaxCluster = 16;                            // CTAs per unit, at most
// Kept blocks a streaming CTA gets with the release (pool entries q, q + S, ... of streaming
// CTA q of S), before it takes the rest from the shared counter.  A pool of at most
// kStatic * S entries (176 kept blocks with clusters of 12) goes out with the release whole:
// every CTA's pages and the merge order are then fixed, so the output is bitwise
// reproducible; longer pools are balanced through the counter (timing decides who takes
// which of the rest).
constexpr int kStatic = 16;
static_assert(kStatic % 2 == 0, "the release carries kStatic / 2 16-byte stores");
// The scoring counts the top 12 bits of the keys besides the top 8: on score sets like the
// method's (a few hundred candidates, scores spread over a few units) the 12-bit bin holding
// the k-th largest key then holds a few keys, and the selection finishes in one pass over the
// keys and one rank of that bin.
constexpr int kHistBits = 12;
constexpr int kBins = 1 << kHistBits;
constexpr int kBinRank = 32;  // boundary bins up to this size are ranked by one warp
static_assert(kMaxCand <= 1024, "bin ranks pack a candidate index into 10 bits");

template <int D, bool F8 = false>
struct FusedCfg {
  using C = Cfg<D, F8>;
  // after the ring (every CTA)
  // keys_ready, list_ready, parts_ready, scored
  static constexpr size_t kOffBars = (C::kSmem + 15) & ~size_t(15);
  static constexpr size_t kOffQbar = kOffBars + 4 * sizeof(uint64_t);
  static constexpr size_t kOffShare = kOffQbar + sizeof(float) * D;
  static constexpr size_t kOffMail = kOffShare + sizeof(int32_t) * kMaxShare;  // kStatic int2
  static constexpr size_t kSmem = kOffMail + sizeof(int2) * kStatic;
  static constexpr size_t kSmemAlloc = kSmem + 1024;
  // the leader streams no pages: its K ring holds the selection state ...
  static constexpr size_t kOffKeys = C::kOffK;
  static constexpr size_t kOffPages = kOffKeys + sizeof(uint32_t) * kMaxCand;
  static constexpr size_t kOffHist = kOffPages + sizeof(int32_t) * kMaxCand;
  static constexpr size_t kOffHist12 = kOffHist + sizeof(int32_t) * 3 * 256;  // 16-byte aligned
  static constexpr size_t kOffFin = kOffHist12 + sizeof(int32_t) * kBins;
  static constexpr size_t kOffKept = (kOffFin + sizeof(FinishShared<kSelThreads>) + 15) & ~size_t(15);
  static constexpr size_t kOffPool = kOffKept + sizeof(int32_t) * kMaxCand;  // int2 (page, block)
  static constexpr size_t kOffTaken = kOffPool + sizeof(int2) * kMaxCand;    // pool counter
  static constexpr size_t kOffBnd = kOffTaken + 16;  // boundary-bin candidates, their ranks' keys
  static constexpr size_t kOffBinKey = kOffBnd + sizeof(int32_t) * kBinRank;
  static constexpr size_t kOffKeepBits = kOffBinKey + sizeof(uint32_t) * kBinRank;  // a bit per candidate
  static constexpr size_t kOffFast = kOffKeepBits + sizeof(uint32_t) * (kMaxCand / 32);
  // per 32-key round: keys above the boundary bin, keys in it
  static constexpr size_t kOffRounds = kOffFast + 16;
  static constexpr size_t kSelEnd = kOffRounds + sizeof(int32_t) * 2 * (kMaxCand / 32);
  // ... and its V ring the streaming CTAs' partials: acc [15][8][D], then (m, l) [15][8][2]
  static constexpr size_t kOffPartAcc = C::kOffV;
  static constexpr size_t kOffPartMl = kOffPartAcc + sizeof(float) * (kMaxCluster - 1) * 8 * D;
  static constexpr size_t kPartEnd = kOffPartMl + sizeof(float) * (kMaxCluster - 1) * 8 * 2;
  static_assert(kSelEnd <= C::kOffV, "selection state fits in the K ring");
  static_assert(kOffHist % 16 == 0 && kOffBinKey % 16 == 0 && kOffMail % 16 == 0,
                "vector accesses");
  static_assert(kPartEnd <= C::kOffQ, "partials fit in the V ring");
  static_assert(kSmemAlloc <= 232448, "shared memory opt-in limit");
  // Stages of list A a streaming CTA copies before its own scoring loads have returned.
  // Those loads queue behind the copies already issued (a full ring is ~17 MB over the
  // cluster's SMs), so the rest of the ring waits for them; two stages still keep the
  // consumers fed once they turn to the pages.
  static constexpr int kEarlyStages = 2;
  static_assert(kEarlyStages < C::kStages, "the ring is never filled before the scoring");
};

// Share [q*n/S, (q+1)*n/S) of n items for part q of S (n * S < 2^31: n <= 1024 kept or
// candidate blocks, or list-A pages of one request, S < 16).
__device__ __forceinline__ int32_t share_begin(int32_t q, int32_t n, int32_t S) {
  return n * q / S;
}

// Grid: one cluster of CS CTAs per unit; 8 consumer warps + 1 producer warp per CTA.
template <int D, bool F8>
__global__ void __maxnreg__(128) fused_decode_kernel(const DecodeArgs a,
                                                     const __grid_constant__ TmaMaps maps) {
  using C = Cfg<D, F8>;
  using F = FusedCfg<D, F8>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* keys_ready = reinterpret_cast<uint64_t*>(smem + F::kOffBars);
  uint64_t* list_ready = keys_ready + 1;
  uint64_t* parts_ready = keys_ready + 2;
  uint64_t* scored = keys_ready + 3;
  float* qbar = reinterpret_cast<float*>(smem + F::kOffQbar);
  int32_t* share = reinterpret_cast<int32_t*>(smem + F::kOffShare);
  int2* mail = reinterpret_cast<int2*>(smem + F::kOffMail);  // the release's pool entries
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + F::kOffKeys);    // leader
  int32_t* pages = reinterpret_cast<int32_t*>(smem + F::kOffPages);    // leader
  int32_t(*hist)[256] = reinterpret_cast<int32_t(*)[256]>(smem + F::kOffHist);  // leader
  FinishShared<kSelThreads>& fin = *reinterpret_cast<FinishShared<kSelThreads>*>(smem + F::kOffFin);
  int32_t* kept_list = reinterpret_cast<int32_t*>(smem + F::kOffKept);  // leader
  int2* pool = reinterpret_cast<int2*>(smem + F::kOffPool);              // leader
  uint32_t* taken = reinterpret_cast<uint32_t*>(smem + F::kOffTaken);    // leader
  int32_t* hist12 = reinterpret_cast<int32_t*>(smem + F::kOffHist12);    // leader
  int32_t* bnd = reinterpret_cast<int32_t*>(smem + F::kOffBnd);          // leader
  uint32_t* bin_key = reinterpret_cast<uint32_t*>(smem + F::kOffBinKey);  // leader
  uint32_t* keepbits = reinterpret_cast<uint32_t*>(smem + F::kOffKeepBits);  // leader
  int32_t* fast_flag = reinterpret_cast<int32_t*>(smem + F::kOffFast);   // leader: flag, digit
  int32_t* rounds = reinterpret_cast<int32_t*>(smem + F::kOffRounds);   // leader
  float* part_acc = reinterpret_cast<float*>(smem + F::kOffPartAcc);  // leader
  float* part_ml = reinterpret_cast<float*>(smem + F::kOffPartMl);    // leader

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank(), CS = cluster_size();
  const int32_t S = (int32_t)CS - 1;  // streaming CTAs
  const int32_t u = blockIdx.x / CS;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  const bool leader = crank == 0;
  bool arrived = false;  // on the closing cluster barrier (warp-uniform)

  if (tid == 0) {
    init_ring<D, F8>(smem);
    mbar_init(keys_ready, kMaxCand);            // one per candidate, the rest at once
    mbar_init(list_ready, 1);                   // the leader, once the pool is laid out
    mbar_init(parts_ready, 1);                  // the leader, expecting every partial's bytes
    mbar_init(scored, kConsumerWarps);          // each consumer warp, its scores computed
    fence_mbar_init();
    // the streaming CTAs' partials land with asynchronous stores that count their bytes
    if (leader)
      mbar_arrive_expect_tx(parts_ready, (uint32_t)(S * a.G * (D + 2)) * (uint32_t)sizeof(float));
  }
  if (leader) {  // the histograms (contiguous) and the pool counter
    int4* h4 = reinterpret_cast<int4*>(&hist[0][0]);
    for (int i = tid; i < (3 * 256 + kBins) / 4; i += blockDim.x) h4[i] = make_int4(0, 0, 0, 0);
    if (tid == 0) *taken = (uint32_t)(kStatic * S);  // entries below go with the release
  }
  __syncthreads();
  cluster_arrive();  // this CTA's barriers and the leader's histogram are ready (waited for
                     // before the first access to another CTA)
  // Launched behind the previous kernel of the stream (programmatic launch): everything above
  // touches shared memory only; every input may be that kernel's output, so wait for it here.
  griddep_wait();
  griddep_launch_dependents();

  // The group's query values (thread e < D, a consumer: element e of its G heads), loaded
  // ahead of the lengths: they do not depend on them, and the scoring waits for both
  constexpr int kMaxG = 8;  // the MMA decode's largest group
  static_assert(D <= kSelThreads, "one consumer thread per query element");
  float qv[kMaxG] = {};
  if (tid < D) {
    const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) +
                              ((int64_t)r * a.Hq + (int64_t)h * a.G) * D + tid;
#pragma unroll
    for (int j = 0; j < kMaxG; ++j)
      if (j < a.G) qv[j] = __bfloat162float(qp[(int64_t)j * D]);
  }

  // This CTA's page of each candidate of its scoring share.  The shares split the candidates
  // a request of the table can have at most (nmax), not the request's own: the table entries
  // then load alongside the request's length instead of after it.
  const int32_t b_lo = a.init_tokens / kBlock;
  const int32_t Wmax = a.max_blocks * kBlock - a.local_tokens;
  const int32_t nmax = Wmax > a.init_tokens ? (Wmax + kBlock - 1) / kBlock - b_lo : 0;
  const int32_t s_lo = share_begin((int32_t)crank, nmax, (int32_t)CS);
  const int32_t s_hi = share_begin((int32_t)crank + 1, nmax, (int32_t)CS);  // <= kMaxShare apart
  const int32_t* bt_r = a.block_table + (int64_t)r * a.max_blocks;
  int32_t my_page = -1;  // b_lo + nmax <= max_blocks: inside the request's table row
  if (tid < s_hi - s_lo) my_page = bt_r[b_lo + s_lo + tid];

  // The unit's sizes: list A and the candidates n (<= nmax) from the length alone; the kept
  // count k (what the selection will write) takes a few double-precision steps, so each role
  // computes it where it first needs it (the producer once list A is out).
  const int32_t L_in = a.seq_lens[r];
  const int32_t prompt = a.prompt_lens ? a.prompt_lens[r] : L_in;
  uint32_t geflags = 0;
  const Geom g = make_geom(L_in, 0, a.max_blocks, a.kmax, a.init_tokens, a.local_tokens, geflags);
  const int32_t n = candidate_count(g.L, a.local_tokens, a.init_tokens);
  auto kept_count = [&] {
    return selection_count(L_in, prompt, a.max_blocks, a.kmax, a.init_tokens, a.local_tokens,
                           a.dense_boundary, a.topk_percent)
        .k;
  };
  const int32_t nA = list_a_count(g);
  const int32_t q = (int32_t)crank - 1;  // streaming rank
  const int32_t a0 = leader ? 0 : share_begin(q, nA, S), a1 = leader ? 0 : share_begin(q + 1, nA, S);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    cluster_wait();
    if (!leader) {
      uint32_t eflags = 0;
      bool abort = false;
      int64_t it = 0, armed = 0;
      int32_t k = -1;  // the kept count, computed while the producer waits anyway
      // list A: 32 positions resolved at once, handed out in order.  The first kEarlyStages
      // copies go out at once; the rest of the ring waits for this CTA's scoring loads,
      // which would otherwise return only after every copy ahead of them had landed (holding
      // all of list A back costs the stream more than the scoring gains)
      for (int32_t j0 = a0; j0 < a1 && !abort; j0 += 32) {
        const int32_t cnt = min(32, a1 - j0);
        PageTask task;
        task.page = -1;
        task.lo = task.hi = task.ie = task.ws = 0;
        if (lane < cnt) task = resolve_a(g, j0 + lane, bt_r, total_pages(a), eflags);
        for (int l = 0; l < cnt && !abort; ++l) {
          PageTask tl;
          tl.page = __shfl_sync(0xffffffffu, task.page, l);
          tl.lo = __shfl_sync(0xffffffffu, task.lo, l);
          tl.hi = __shfl_sync(0xffffffffu, task.hi, l);
          tl.ie = __shfl_sync(0xffffffffu, task.ie, l);
          tl.ws = __shfl_sync(0xffffffffu, task.ws, l);
          if (it == F::kEarlyStages) {  // the rest once this CTA's scores are in
            k = kept_count();             // (its steps overlap the wait)
            bool ok = true;
            if (lane == 0) ok = mbar_wait(scored, 0);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
              eflags |= SRKV_EFLAG_TIMEOUT;
              abort = true;
              break;
            }
          }
          issue_stage_warp<D, F8>(a, maps, smem, it, u, it == 0 ? kNewUnit : 0u, tl, armed, abort,
                              eflags, lane);
          ++it;
        }
      }
      if (k < 0) k = kept_count();
      // list B: the kStatic entries that came with the release, then kept blocks from the
      // leader's pool until it is empty.  Lane 0 takes the entries (a cluster atomic, then a
      // cluster load) one ahead: the first atomic goes out before the release's entries are
      // issued, each next one before the current entry waits for a free stage; the other
      // lanes read an entry only after that wait.  The release is waited for even with
      // nothing to take: the leader's writes into this CTA are then all done before it ends.
      if (!abort) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_cluster(list_ready, 0);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          abort = true;
        }
      }
      uint32_t first = 0xffffffffu;  // lane 0: the first entry taken from the counter
      if (k > 0 && !abort && lane == 0) first = atom_cluster_add(taken, 0, 1u);
      auto issue_b = [&](const int2 e) {  // kept block (page, block id)
        PageTask t;
        t.page = -1;
        t.lo = t.hi = t.ie = t.ws = 0;
        const int32_t base = e.y * kBlock, rows = min(kBlock, g.L - base);
        const int32_t lo = max(a.init_tokens - base, 0), hi = min(g.W - base, rows);
        if (lo < hi && e.x >= 0 && (int64_t)e.x < total_pages(a)) {
          t.page = e.x;
          t.block = e.y;
          t.lo = lo;
          t.hi = hi;
          t.ie = hi;  // every loaded row is attended
          t.ws = hi;
        } else if (lo < hi) {
          eflags |= SRKV_EFLAG_PAGE_RANGE;
        }
        issue_stage_warp<D, F8>(a, maps, smem, it, u, it == 0 ? kNewUnit : 0u, t, armed, abort,
                            eflags, lane);
        ++it;
      };
      if (k > 0 && !abort) {
#pragma unroll 1
        for (int j = 0; j < kStatic && !abort; ++j) {
          const int2 e = mail[j];
          if (e.y < 0) break;  // beyond the pool
          issue_b(e);
        }
      }
      auto take = [&](int2& e) -> bool {  // lane 0
        const uint32_t i = atom_cluster_add(taken, 0, 1u);
        if (i >= (uint32_t)k) return false;
        e = ld_cluster_int2(pool + i, 0);
        return true;
      };
      int2 e0 = make_int2(-1, 0);  // lane 0's entry
      bool have = false;
      if (lane == 0 && first < (uint32_t)k) {
        e0 = ld_cluster_int2(pool + first, 0);
        have = true;
      }
      have = __shfl_sync(0xffffffffu, have, 0) && !abort;
      while (have && !abort) {
        const int2 e = make_int2(__shfl_sync(0xffffffffu, e0.x, 0), __shfl_sync(0xffffffffu, e0.y, 0));
        int2 next0 = make_int2(-1, 0);
        bool more = false;
        if (lane == 0) more = take(next0);
        issue_b(e);
        e0 = next0;
        have = __shfl_sync(0xffffffffu, more, 0);
      }
      if (lane == 0) {
        // the sentinel closes the segment (empty if this CTA took no page)
        PageTask none;
        none.page = -1;
        none.lo = none.hi = none.ie = none.ws = 0;
        issue_stage<D, F8>(a, maps, smem, it, -1, kLast | kSegEnd, none, armed, abort, eflags);
        uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
        uint64_t* full_v = full + C::kStages;
        const int64_t first = armed > C::kStages ? armed - C::kStages : 0;
        for (int64_t i = first; i < armed; ++i)  // every copy lands before the CTA ends
          if (!mbar_wait(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1)) ||
              !mbar_wait(&full_v[i % C::kStages], (uint32_t)((i / C::kStages) & 1))) {
            eflags |= SRKV_EFLAG_TIMEOUT;
            break;
          }
      }
      eflags = __reduce_or_sync(0xffffffffu, eflags | geflags);
      if (lane == 0) raise_flags(a.error_flags, eflags);
    }
  } else {
    // ------------------------------------------------------------------ consumers
    auto bar = [] { named_bar_sync(1, kSelThreads); };
    // 1. this CTA's share of the candidates: table entries and the group query sum
    if (tid < s_hi - s_lo) share[tid] = my_page;
    if (tid < D) {  // the group query sum, in head order
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxG; ++j)
        if (j < a.G) s += qv[j];
      qbar[tid] = s;
    }
    bar();
    // 2. scores into the leader (keys, pages, histograms of the top 12 and 8 key bits)
    // keys go to the leader once every CTA has passed its setup (cluster barrier)
    // (a share of more than 8 per warp takes rounds of 16: fewer round trips, longer
    // reductions per round)
    bool waited = false;
    auto issued = [&] {
      cluster_wait();
      waited = true;
    };
    // one arrival for the round's keys, pages and counts of the warp (fewer remote arrivals
    // on the leader's barrier than one per key)
    auto stored = [&](uint32_t cnt) { mbar_arrive_cluster_n(keys_ready, 0, cnt); };
    const uint32_t eflags =
        s_hi - s_lo <= kConsumerWarps * 8
            ? score_share<D, kConsumerWarps, kHistBits, 8>(
                  qbar, share, s_lo, min(s_hi, n), a.reps, total_pages(a), a.Hkv, h, keys,
                  hist12, &hist[0][0], pages, warp, lane, issued, stored)
            : score_share<D, kConsumerWarps, kHistBits, 16>(
                  qbar, share, s_lo, min(s_hi, n), a.reps, total_pages(a), a.Hkv, h, keys,
                  hist12, &hist[0][0], pages, warp, lane, issued, stored);
    if (!waited) cluster_wait();  // a warp without candidates
    if (lane == 0) mbar_arrive(scored);
    if (lane == 0 && eflags) raise_flags(a.error_flags, eflags);
    // the arrivals the leader's barrier expects beyond the n candidates, at once
    if (leader && tid == 0 && n < kMaxCand)
      mbar_arrive_cluster_n(keys_ready, 0, (uint32_t)(kMaxCand - n));

    if (leader) {
      // 3. select the k kept blocks, lay them out as the pool of kept blocks (page, block),
      // release the streaming CTAs, then write sel / nsel for the caller (nobody in the
      // cluster reads them)
      const int32_t k = kept_count();
      if (!mbar_wait_cluster(keys_ready, 0)) {
        if (tid == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      }
      int32_t kept = 0;
      int32_t* sel_u = a.sel_out + (int64_t)u * a.kmax;
      const bool partial = k > 0 && k < n;
      // Streaming CTA qq's release: its pool entries qq, qq + S, ... (up to kStatic; (-1, -1)
      // beyond the pool) into its shared memory, then its list_ready (which orders them).
      auto release = [&](int32_t qq) {
        int2 e[kStatic];
#pragma unroll
        for (int j = 0; j < kStatic; ++j) {
          const int32_t p = qq + j * S;
          e[j] = p < k ? pool[p] : make_int2(-1, -1);
        }
        int4* m4 = reinterpret_cast<int4*>(mail);
#pragma unroll
        for (int j = 0; j < kStatic; j += 2)
          st_cluster_int4(m4 + j / 2, (uint32_t)qq + 1,
                          make_int4(e[j].x, e[j].y, e[j + 1].x, e[j + 1].y));
        mbar_arrive_cluster(list_ready, (uint32_t)qq + 1);
      };
      if (partial) {
        // Warp 0: the 12-bit bin holding the k-th largest key.  Every key above it is kept:
        // into the pool (the keys above, in block order) and the kept bits; the bin's keys
        // (at most kBinRank) are ranked and the first k - (keys above) follow in the pool.
        // The pass over the keys is shared by the 8 warps, a round of 32 keys each in turn.
        // (The count checks only matter if some scores never arrived: flagged.)
        if (warp == 0) {
          const Boundary bd = warp_boundary(&hist[0][0], hist12, k, lane);
          if (lane == 0) {
            fast_flag[0] = bd.cnt <= kBinRank;
            fast_flag[1] = bd.digit;
          }
        }
        bar();
        if (fast_flag[0]) {
          constexpr int kRounds = kMaxCand / 32 / kConsumerWarps;  // a warp's rounds at most
          const uint32_t lt = (1u << lane) - 1u;
          const uint32_t dsel = (uint32_t)fast_flag[1];
          uint32_t kk[kRounds], ma[kRounds], mb[kRounds];
          int32_t pg[kRounds];
#pragma unroll
          for (int x = 0; x < kRounds; ++x) {  // round warp + 8 x: keys 32 (warp + 8 x) + lane
            const int32_t rr = warp + kConsumerWarps * x, i = 32 * rr + lane;
            kk[x] = i < n ? keys[i] : 0u;
            pg[x] = i < n ? pages[i] : -1;
          }
#pragma unroll
          for (int x = 0; x < kRounds; ++x) {
            const int32_t rr = warp + kConsumerWarps * x, i = 32 * rr + lane;
            const uint32_t dg = kk[x] >> (32 - kHistBits);
            ma[x] = __ballot_sync(0xffffffffu, i < n && dg > dsel);
            mb[x] = __ballot_sync(0xffffffffu, i < n && dg == dsel);
            if (lane == 0 && 32 * rr < n) {
              rounds[rr] = __popc(ma[x]);
              rounds[kMaxCand / 32 + rr] = __popc(mb[x]);
              keepbits[rr] = ma[x];
            }
          }
          bar();
          // every warp scans the rounds' counts; its own rounds' keys go to their places
          const int32_t nr = (n + 31) >> 5;
          int32_t na = 0, nb = 0;
          const int32_t pa = warp_exclusive_scan(lane < nr ? rounds[lane] : 0, lane, &na);
          const int32_t pb = warp_exclusive_scan(lane < nr ? rounds[kMaxCand / 32 + lane] : 0,
                                                 lane, &nb);
#pragma unroll
          for (int x = 0; x < kRounds; ++x) {
            const int32_t rr = warp + kConsumerWarps * x, i = 32 * rr + lane;
            if (32 * rr >= n) break;  // uniform
            const int32_t sa = __shfl_sync(0xffffffffu, pa, rr) + __popc(ma[x] & lt);
            const int32_t sb = __shfl_sync(0xffffffffu, pb, rr) + __popc(mb[x] & lt);
            if (((ma[x] >> lane) & 1u) && sa < k) pool[sa] = make_int2(pg[x], b_lo + i);
            if (((mb[x] >> lane) & 1u) && sb < kBinRank) {
              // rank key: the key's low bits (its top bits are the bin's), then the lower
              // block; unique, larger = kept first
              bnd[sb] = i;
              bin_key[sb] = ((kk[x] & ((1u << (32 - kHistBits)) - 1u)) << 10) |
                            (uint32_t)(kMaxCand - 1 - i);
            }
          }
          bar();
          if (warp == 0) {
            const int32_t nbin = min(nb, kBinRank), nab = min(na, k);
            const uint32_t mine = lane < nbin ? bin_key[lane] : 0u;
            int32_t rank = 0;
#pragma unroll
            for (int j = 0; j < kBinRank; j += 4) {
              const uint4 v = *reinterpret_cast<const uint4*>(bin_key + j);
              rank += (j < nbin && v.x > mine) + (j + 1 < nbin && v.y > mine) +
                      (j + 2 < nbin && v.z > mine) + (j + 3 < nbin && v.w > mine);
            }
            const bool take = lane < nbin && rank < k - nab;
            const uint32_t m = __ballot_sync(0xffffffffu, take);
            if (take) {
              const int32_t i = bnd[lane], slot = nab + __popc(m & lt);
              if (slot < k) pool[slot] = make_int2(pages[i], b_lo + i);
              atomicOr(&keepbits[i >> 5], 1u << (i & 31));
            }
            for (int32_t p = nab + __popc(m) + lane; p < k; p += 32) pool[p] = make_int2(-1, 0);
          }
          bar();  // the pool is complete
          // the releases: every entry store first (one 16-byte store per thread), then, once
          // the barrier orders them all, one arrival per streaming CTA
          for (int32_t x = tid; x < S * (kStatic / 2); x += kSelThreads) {
            const int32_t qq = x / (kStatic / 2), j = 2 * (x % (kStatic / 2));
            const int32_t p0 = qq + j * S, p1 = p0 + S;
            const int2 e0 = p0 < k ? pool[p0] : make_int2(-1, -1);
            const int2 e1 = p1 < k ? pool[p1] : make_int2(-1, -1);
            st_cluster_int4(reinterpret_cast<int4*>(mail) + j / 2, (uint32_t)qq + 1,
                            make_int4(e0.x, e0.y, e1.x, e1.y));
          }
          bar();
          if (tid < S) mbar_arrive_cluster(list_ready, (uint32_t)tid + 1);
        }
      }
      bar();
      if (partial && *fast_flag) {
        // sel in block order: a kept candidate's slot = kept candidates of the earlier words
        // of the kept bits + the earlier bits of its own word
        const uint32_t lt = (1u << lane) - 1u;
        const int32_t words = (n + 31) >> 5;
        const int32_t wofs =
            warp_exclusive_scan(lane < words ? __popc(keepbits[lane]) : 0, lane, &kept);
        for (int32_t i0 = 0; i0 < n; i0 += kSelThreads) {
          const int32_t i = i0 + tid, w = (i0 >> 5) + warp;
          const uint32_t bits = i < n ? keepbits[w] : 0u;
          const int32_t pos = __shfl_sync(0xffffffffu, wofs, w) + __popc(bits & lt);
          if (((bits >> lane) & 1u) && pos < k) sel_u[pos] = b_lo + i;
        }
        kept = min(kept, k);
      } else {
        // k == n (every candidate), k == 0, or a boundary bin too large to rank at once:
        // radix narrowing from the top-8-bit histogram, then the ordered finish
        if (k == n) {
          for (int32_t i = tid; i < n; i += kSelThreads) kept_list[i] = i;
          kept = n;
        } else if (k > 0) {
          const RadixState rs = radix_narrow<kSelThreads>(keys, n, k, hist, tid, bar);
          kept = finish_fast<kSelThreads>(keys, n, rs, fin, tid, bar,
                                          [&](int32_t pos, int32_t i) { kept_list[pos] = i; });
        }
        bar();
        // the pool: k entries (an entry the selection did not fill has no page); the barrier
        // orders every thread's entries before the releases below
        for (int32_t p = tid; p < k; p += kSelThreads)
          pool[p] = p < kept ? make_int2(pages[kept_list[p]], b_lo + kept_list[p]) : make_int2(-1, 0);
        bar();
        for (int32_t qq = tid; qq < S; qq += kSelThreads) release(qq);
        for (int32_t p = tid; p < kept; p += kSelThreads) sel_u[p] = b_lo + kept_list[p];
      }
      if (tid == 0) {
        a.nsel_out[u] = kept;
        if (kept != k) raise_flags(a.error_flags, SRKV_EFLAG_SELECTION);
      }
      // 4. merge the streaming CTAs' partials: query head w % G, half w / G of d (G <= 4; with
      // G = 8, both halves of head w).  Once they are all in, no CTA reaches another's shared
      // memory any more (each streaming CTA waited for its release, so the leader's writes
      // into it are done): the leader's consumers arrive on the closing cluster barrier with
      // nothing to order, and the barrier completes while they merge.
      if (!mbar_wait_cluster(parts_ready, 0)) {
        if (tid == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      }
      cluster_arrive_relaxed();
      arrived = true;
      const int32_t hw = a.G <= 4 ? 2 : 1;  // warps per head
      if (warp < a.G * hw) {
        // lane qq holds the (max, sum) of streaming CTA qq; weights by shuffles, then every
        // lane adds its d-slice of the weighted partials
        constexpr int V = D / 64;  // values per lane in half of d
        const int32_t head = warp % a.G;
        float m = -INFINITY, l = 0.f;  // a CTA that attended nothing wrote (-inf, 0)
        if (lane < S) {
          m = part_ml[(lane * a.G + head) * 2];
          l = part_ml[(lane * a.G + head) * 2 + 1];
        }
        float mx = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float w = mx == -INFINITY ? 0.f : fast_exp2(m - mx);  // 0 for an absent part
        float l_run = w * l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
        for (int32_t half = warp / a.G; half < 2; half += hw) {
          // every streaming CTA wrote a partial (zeros if it attended nothing).  The loads and
          // weight shuffles of a batch of 8 slots are unconditional, so they issue together
          // (the partial area holds kMaxCluster - 1 slots, so every address is in it); a
          // select drops the slots beyond S and those of weight 0
          const int32_t d0 = half * (D / 2) + lane * V;
          float acc[V];
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
          for (int b0 = 0; b0 < kMaxCluster - 1; b0 += 8) {
            float x[8][V], wv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int qq = b0 + j < kMaxCluster - 1 ? b0 + j : kMaxCluster - 2;
              wv[j] = __shfl_sync(0xffffffffu, w, qq);
              const float* src = part_acc + (qq * a.G + head) * D + d0;
              if constexpr (V == 2) {
                const float2 v2 = *reinterpret_cast<const float2*>(src);
                x[j][0] = v2.x;
                x[j][1] = v2.y;
              } else {
                x[j][0] = *src;
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool use = b0 + j < S && wv[j] != 0.f;
#pragma unroll
              for (int e = 0; e < V; ++e) acc[e] = use ? fmaf(wv[j], x[j][e], acc[e]) : acc[e];
            }
          }
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) +
                             ((int64_t)r * a.Hq + (int64_t)h * a.G + head) * D + d0;
          if constexpr (V == 2) {
            const float x0 = l_run > 0.f ? acc[0] / l_run : 0.f;
            const float x1 = l_run > 0.f ? acc[1] / l_run : 0.f;
            *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(x0, x1);
          } else {
            *o = __float2bfloat16_rn(l_run > 0.f ? acc[0] / l_run : 0.f);
          }
        }
      }
    } else {
      // 3'. attend list A, then the kept blocks taken from the pool, as one segment; the
      // merged partial goes to the leader's shared memory
      consumer_loop<D, F8>(a, smem, lane, warp,
                       [&](const SoftmaxState<D>& st, const StageInfo&, Lane ln) {
                         // asynchronous stores, each counted on the leader's parts_ready
                         const uint32_t acc_r = cluster_addr(part_acc + (int64_t)q * a.G * D, 0);
                         const uint32_t ml_r = cluster_addr(part_ml + (int64_t)q * a.G * 2, 0);
                         const uint32_t bar_r = cluster_addr(parts_ready, 0);
                         emit_partial<D, F8>(
                             st, ln, a.G,
                             [&](int i, float4 v) { st_async_f4(acc_r + 4u * i, v, bar_r); },
                             [&](int j, float2 v) { st_async_f2(ml_r + 4u * j, v, bar_r); });
                       });
    }
  }
  // nobody leaves while another CTA may still reach its shared memory
  __syncwarp();
  if (!arrived) cluster_arrive();
  cluster_wait();
}

}  // namespace

// Clusters of `cs` CTAs of fused_decode_kernel<D, F8> that can be resident at once (0 on error).
template <int D, bool F8>
int32_t max_active_clusters(int32_t cs) {
  using F = FusedCfg<D, F8>;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cs);
  lc.blockDim = dim3((kConsumerWarps + 1) * 32);
  lc.dynamicSmemBytes = F::kSmemAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaFuncSetAttribute(fused_decode_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)F::kSmemAlloc);
  cudaFuncSetAttribute(fused_decode_kernel<D, F8>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                       1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fused_decode_kernel<D, F8>, &lc) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  return n;
}

// Cluster size for `units` units (0 = the fused path does not apply): the largest of 16 down
// to 4 CTAs per unit such that every cluster is resident at once (on a GB300: 16 CTAs for up
// to 7 units, 12 for 8, 10 for up to 13, 9 for up to 15, 6 for up to 23, 5 for up to 28, 4
// for up to 36).  e4m3: compressed pages.  Clusters of fewer than 8 only for bf16 pages, d 128, top-k
// ratio <= 0.3: there the dynamic pool's balance beats the three kernels on every SM (batch 4
// x 131072 on clusters of 4: 60.4 against 67.4 us at 0.1, 91.1 against 96.1 at 0.2), while at
// 0.4 and at 1.0 the three kernels' 152 streaming SMs win (151.3 against 152.6 us, 322
// against 337).
int32_t fused_cluster_size(const srkv_config& cfg, int32_t units, int32_t max_blocks,
                           bool e4m3) {
  if (!mma_split_supported(cfg) || units <= 0) return 0;
  if (e4m3 && cfg.head_dim != 128) return 0;
  const int64_t W = (int64_t)max_blocks * kBlock - cfg.local_tokens;
  const int64_t nmax = W > cfg.init_tokens ? (W + kBlock - 1) / kBlock - cfg.init_tokens / kBlock : 0;
  if (nmax > kMaxCand) return 0;
  // [device][d 64, d 128, d 128 compressed][cluster 16 - c]: max active + 1
  constexpr int kSizes = kMaxCluster - 3;  // 16 .. 4
  static int32_t cached[128][3][kSizes];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  const int di = e4m3 ? 2 : cfg.head_dim == 128 ? 1 : 0;
  for (int c = 0; c < kSizes; ++c) {
    const int32_t cs = kMaxCluster - c;
    if (nmax > (int64_t)kMaxShare * cs) continue;  // per-CTA scoring share
    if (cs < 8 && (di != 1 || cfg.topk_percent > 0.3)) continue;
    if (cached[dev][di][c] == 0) {
      const int32_t n = di == 2   ? max_active_clusters<128, true>(cs)
                        : di == 1 ? max_active_clusters<128, false>(cs)
                                  : max_active_clusters<64, false>(cs);
      cached[dev][di][c] = n + 1;
    }
    if (units <= cached[dev][di][c] - 1) return cs;
  }
  return 0;
}

template <int D, bool F8>
cudaError_t launch_fused_t(const DecodeArgs& a, int32_t cluster, cudaStream_t stream) {
  TmaMaps maps;
  if (!encode_cache_map(&maps.k, a.k_cache, a.num_pages, a.Hkv, D, F8) ||
      !encode_cache_map(&maps.v, a.v_cache, a.num_pages, a.Hkv, D, F8))
    return cudaErrorInvalidValue;
  const int64_t grid = (int64_t)a.batch * a.Hkv * cluster;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3((kConsumerWarps + 1) * 32);
  lc.dynamicSmemBytes = FusedCfg<D, F8>::kSmemAlloc;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, fused_decode_kernel<D, F8>, a, maps);
}

cudaError_t launch_fused(const DecodeArgs& a, int32_t cluster, cudaStream_t stream) {
  if (a.k_scale) return launch_fused_t<128, true>(a, cluster, stream);  // compressed pages
  return a.d == 128 ? launch_fused_t<128, false>(a, cluster, stream)
                    : launch_fused_t<64, false>(a, cluster, stream);
}

}  // namespace srkv
