// decode_split_mma.cu -- split phase of sparse paged decode on tensor cores (bf16).
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Overall Solution": the selected blocks are concatenated with the initial tokens and the
// sliding window and take part in attention; the ATB reuse article (§1.1) gives
// softmax(QK^T/sqrt(d_k))V and (§2.2, §3.1) reads K/V page by page through a page table
// staged on chip.  Each (page, kv head) slab of K or V is contiguous (S*d*2 bytes), so a
// page is moved by two one-dimensional TMA bulk copies into shared memory.
//
// CTA = 1 producer warp + 8 consumer warps, one CTA per SM (persistent), each CTA owning
// an equal share of all units' page lists (see decode_plan.cuh).
//   producer: plans list A (initial + window pages) and list B (selected pages) with
//             warp-level scans, resolves 32 list positions at once (one per lane), and lane 0
//             streams the pages through a ring of stages (3 x 64 KiB for d = 128) with tiled
//             TMA copies (128-byte swizzle, 64-column boxes of a whole 128-row slab),
//             completion counted on an mbarrier per stage.  When the previous
//             kernel is the scoring kernel, list A is streamed before that kernel finishes
//             (programmatic launch) and the producer waits for the selection only before
//             list B; a sentinel stage ends the consumers' loop;
//   consumers: warp w owns rows [16w, 16w+16) of every page; MMA row m of the tile is token
//             m ^ 4 (m odd) or m (m even), which with the swizzle lets every 8-lane phase
//             of a 16-byte fragment load hit 8 distinct bank groups.  The group's queries are the
//             N = 8 side of m16n8k16 bf16 MMAs, keys/values the M = 16 side:
//               S^T[16 tok x 8 heads]  = K[16 x d] . Q^T[d x 8]
//               O^T[d x 8 heads]      += V^T[d x 16 tok] . P[16 tok x 8]
//             (the contraction index of each product may be permuted consistently on
//             both operands, which lets every fragment come from 16-byte shared loads;
//             P^T -> P is one movmatrix.trans per 8x8 block).  Online softmax in fp32,
//             log2 domain; the sum uses the bf16-rounded weights the MMA sees.
//   at the end of a unit's segment the 8 warps merge (max, sum, acc) through shared memory
//   and warp 0 writes the partial to slot unit + CTA of the workspace.
// Every wait is bounded (SRKV_EFLAG_TIMEOUT); rows outside the loaded range are masked in
// the logits and zeroed in V, so stale shared memory never reaches the output.
#include "decode_plan.cuh"

namespace srkv {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr uint32_t kNewUnit = 1, kSegEnd = 2, kBankB = 4, kLast = 8;

struct StageInfo {
  int32_t unit;
  int32_t flags;
  int32_t lo, hi, ie, ws;
  int32_t pad[2];
};

template <int D>
struct Cfg {
  static constexpr int kSlab = kBlock * D * 2;          // bytes of one K or V slab
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kQBytes = 8 * D * 2;              // up to 8 query heads
  static constexpr int MT = D / 16;                      // PV m-tiles over d
  static constexpr int KJ = D / 32;                      // 16-byte K chunks per thread-row
  static constexpr int NCH = D / 64;                     // 16-byte V chunks per token
  static constexpr int kMergeStride = MT * 4 + 4;        // floats per lane in a merge slot
  static constexpr int kMergeSlot = 32 * kMergeStride;   // floats per merge slot

  static constexpr size_t kOffK = 0;
  static constexpr size_t kOffV = kOffK + (size_t)kStages * kSlab;
  static constexpr size_t kOffQ = kOffV + (size_t)kStages * kSlab;
  static constexpr size_t kOffMerge = kOffQ + (size_t)kStages * kQBytes;
  static constexpr size_t kOffInfo = kOffMerge + sizeof(float) * 4 * kMergeSlot;
  static constexpr size_t kOffBar = kOffInfo + sizeof(StageInfo) * kStages;
  // full (K, query, stage info)[kStages], full_v[kStages], empty[kStages], merge w1, w2, r2
  static constexpr size_t kSmem = kOffBar + sizeof(uint64_t) * (3 * kStages + 3);
  static constexpr size_t kSmemAlloc = kSmem + 1024;  // the swizzled stages need 1 KiB alignment
  static constexpr int kBoxes = D / 64;                // 64-column TMA boxes per slab
  static constexpr int kBoxBytes = kBlock * 128;       // 128 rows of 128 bytes
};

// Tensor maps of the K and V caches, [page][kv head * 128 + row][d] (bf16).
struct TmaMaps {
  CUtensorMap k, v;
};

// MMA tile row m -> token row within the 16-row tile (an involution).
__device__ __forceinline__ int tile_token(int m) { return m ^ ((m & 1) << 2); }

// Byte offset of (row, 16-byte chunk c) in a slab loaded with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (uint32_t)((c >> 3) * (kBlock * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

struct Lane {
  int g, t;
};

template <int D>
struct SoftmaxState {
  float acc[Cfg<D>::MT][4];
  float m[2];  // running max (log2 domain) of heads 2t, 2t+1; uniform over g
  float l[2];  // running sum: per-lane part until reduced at the end of a segment
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < Cfg<D>::MT; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }
  // this <- this (+) other, both with reduced l.
  __device__ __forceinline__ void merge(const float* o_acc, float om0, float om1, float ol0,
                                        float ol1) {
    const float om[2] = {om0, om1}, ol[2] = {ol0, ol1};
    float fa[2], fb[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const float mx = fmaxf(m[x], om[x]);
      const float base = mx == -INFINITY ? 0.f : mx;
      fa[x] = fast_exp2(m[x] - base);
      fb[x] = fast_exp2(om[x] - base);
      l[x] = l[x] * fa[x] + ol[x] * fb[x];
      m[x] = mx;
    }
#pragma unroll
    for (int i = 0; i < Cfg<D>::MT; ++i) {
      acc[i][0] = acc[i][0] * fa[0] + o_acc[i * 4 + 0] * fb[0];
      acc[i][1] = acc[i][1] * fa[1] + o_acc[i * 4 + 1] * fb[1];
      acc[i][2] = acc[i][2] * fa[0] + o_acc[i * 4 + 2] * fb[0];
      acc[i][3] = acc[i][3] * fa[1] + o_acc[i * 4 + 3] * fb[1];
    }
  }
  __device__ __forceinline__ void store(float* slot, int lane) const {
    float* p = slot + lane * Cfg<D>::kMergeStride;
#pragma unroll
    for (int i = 0; i < Cfg<D>::MT; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) p[i * 4 + c] = acc[i][c];
    p[Cfg<D>::MT * 4 + 0] = m[0];
    p[Cfg<D>::MT * 4 + 1] = m[1];
    p[Cfg<D>::MT * 4 + 2] = l[0];
    p[Cfg<D>::MT * 4 + 3] = l[1];
  }
  __device__ __forceinline__ void merge_from(const float* slot, int lane) {
    const float* p = slot + lane * Cfg<D>::kMergeStride;
    merge(p, p[Cfg<D>::MT * 4 + 0], p[Cfg<D>::MT * 4 + 1], p[Cfg<D>::MT * 4 + 2],
          p[Cfg<D>::MT * 4 + 3]);
  }
};

// Value index v (0 .. 2*MT-1) of a lane -> head-dim index; the lane with g owns the 16-byte
// chunks g, g+8 (d 128) of every row.
template <int D>
__device__ __forceinline__ int d_of(int g, int v) {
  return 8 * (g + 8 * (v >> 3)) + (v & 7);
}

// Hands stage `it` to the consumers: waits until it is free, writes its description and
// arms its mbarrier with the bytes of the copies it starts (called by one producer lane).
template <int D>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const TmaMaps& maps,
                                            unsigned char* smem, int64_t it, int32_t u,
                                            uint32_t fl, const PageTask& t, int64_t& armed,
                                            bool& abort, uint32_t& eflags) {
  using C = Cfg<D>;
  if (abort) return;
  StageInfo* sInfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;
  const int s = (int)(it % C::kStages);
  if (it >= C::kStages && !mbar_wait(&empty[s], (uint32_t)((it / C::kStages - 1) & 1))) {
    abort = true;
    eflags |= SRKV_EFLAG_TIMEOUT;
    return;
  }
  StageInfo& inf = sInfo[s];
  const bool load = t.page >= 0;
  inf.unit = u;
  inf.flags = (int32_t)fl;
  inf.lo = load ? t.lo : 0;
  inf.hi = load ? t.hi : 0;
  inf.ie = t.ie;
  inf.ws = t.ws;
  // The whole 128-row slab is copied (the swizzle needs whole 1 KiB atoms); rows outside
  // [lo, hi) are masked by the consumers.
  // K and the query complete `full`, V completes `full_v`, so the logits can start while V
  // is still arriving.
  const bool rows = load && t.hi > t.lo;
  const uint32_t qbytes = (uint32_t)(a.G * D * 2);
  mbar_arrive_expect_tx(&full[s], (rows ? (uint32_t)C::kSlab : 0u) +
                                      ((fl & kNewUnit) ? qbytes : 0u));
  mbar_arrive_expect_tx(&full_v[s], rows ? (uint32_t)C::kSlab : 0u);
  ++armed;
  if (u < 0) return;
  const int32_t h = u % a.Hkv, r = u / a.Hkv;
  const uint64_t once = l2_policy_evict_first();  // pages are read once per step
  if (rows) {
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_3d(smem + C::kOffK + (size_t)s * C::kSlab + (size_t)b * C::kBoxBytes, &maps.k,
                  64 * b, h * kBlock, t.page, &full[s], once);
  }
  if (fl & kNewUnit)
    bulk_load(smem + C::kOffQ + (size_t)s * C::kQBytes,
              static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * D,
              qbytes, &full[s]);
  if (rows) {
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_3d(smem + C::kOffV + (size_t)s * C::kSlab + (size_t)b * C::kBoxBytes, &maps.v,
                  64 * b, h * kBlock, t.page, &full_v[s], once);
  }
}

// One arrival per warp: the warp's lanes synchronise (ordering their shared-memory accesses)
// and one lane arrives for all of them.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// 128 registers: a quarter-SM register file (16K) then holds this CTA's three warps on one
// sub-partition (12K) beside one warp of a combine CTA, so the combine is resident and
// waiting when the last partial is written.
template <int D>
__global__ void __maxnreg__(128) split_mma_kernel(const DecodeArgs a,
                                                  const __grid_constant__ TmaMaps maps) {
  using C = Cfg<D>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sK = smem + C::kOffK;
  unsigned char* sV = smem + C::kOffV;
  unsigned char* sQ = smem + C::kOffQ;
  float* sMerge = reinterpret_cast<float*>(smem + C::kOffMerge);
  StageInfo* sInfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;
  uint64_t* mb_w1 = empty + C::kStages;
  uint64_t* mb_w2 = mb_w1 + 1;
  uint64_t* mb_r2 = mb_w1 + 2;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The combine may be scheduled once every CTA has passed this point (it waits for this
  // grid before reading partials).  Without the early mode the inputs are only read after
  // the previous kernel in the stream has finished, and the combine reads them too.
  if (!a.early) griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&empty[s], kConsumerWarps);  // one arrival per consumer warp
    }
    mbar_init(mb_w1, 4);
    mbar_init(mb_w2, 3);
    mbar_init(mb_r2, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    uint32_t eflags = 0;
    bool abort = false;
    int64_t it = 0;     // stages handed out so far (uniform over the warp)
    int64_t armed = 0;  // stages lane 0 armed
    // Both lists are planned first: list B's counts are the selection counts, known from
    // the lengths alone in the early mode.  CTA 0 leaves each list's unit offsets for the
    // combine kernel.
    ListRange rgs[2];
#pragma unroll
    for (int list = kListA; list <= kListB; ++list) {
      int64_t* offsets = blockIdx.x == 0
                             ? reinterpret_cast<int64_t*>(a.ws + (list == kListA ? a.lay.off_a
                                                                                 : a.lay.off_b))
                             : nullptr;
      rgs[list] = warp_plan(a, list, blockIdx.x, list_ctas(a, list), offsets, nullptr, eflags);
    }
    for (int list = kListA; list <= kListB && !abort; ++list) {
      if (list == kListB && a.early) griddep_wait();  // the selection must exist from here on
      const ListRange rg = rgs[list];
      const int64_t npos = rg.end - rg.begin;
      if (npos <= 0) continue;
      const uint32_t bank = list == kListB ? kBankB : 0u;
      int32_t cu = rg.u0;  // walk state: unit and position within its list
      int64_t cj = rg.begin - rg.base0;
      uint32_t dummy = 0;
      Geom cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
      int32_t cn = list == kListA ? list_a_count(cg) : cg.ns;
      for (int64_t done = 0; done < npos && !abort; done += 32) {
        const int cnt = npos - done < 32 ? (int)(npos - done) : 32;
        // Assign positions done .. done+cnt-1 to lanes (uniform walk over the units).
        int32_t my_u = 0, my_j = 0;
        Geom my_g = cg;
        uint32_t my_flags = 0;
        for (int l = 0; l < cnt; ++l) {
          while (cj >= cn) {
            ++cu;
            cj = 0;
            cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
            cn = list == kListA ? list_a_count(cg) : cg.ns;
          }
          const int64_t p = rg.begin + done + l;
          if (lane == l) {
            my_u = cu;
            my_j = (int32_t)cj;
            my_g = cg;
            my_flags = bank | ((cj == 0 || p == rg.begin) ? kNewUnit : 0u) |
                       ((cj == cn - 1 || p == rg.end - 1) ? kSegEnd : 0u);
          }
          ++cj;
        }
        PageTask task;
        task.page = -1;
        task.lo = task.hi = task.ie = task.ws = 0;
        if (lane < cnt) {
          const int32_t* bt_r = a.block_table + (int64_t)(my_u / a.Hkv) * a.max_blocks;
          // Early mode: the count the plan assumed must be the one the scoring wrote.
          const int32_t written = list == kListB && a.early ? a.nsel[my_u] : my_g.ns;
          task = list == kListA
                     ? resolve_a(my_g, my_j, bt_r, a.num_pages, eflags)
                     : resolve_b(my_g, my_j, a.sel + (int64_t)my_u * a.kmax, bt_r, a.num_pages,
                                 a.init_tokens, eflags);
          if (list == kListB && (my_j >= written || (my_j == 0 && written != my_g.ns))) {
            eflags |= SRKV_EFLAG_SELECTION;
            if (my_j >= written) task.page = -1;
          }
        }
        for (int l = 0; l < cnt; ++l) {
          PageTask t;
          const int32_t u = __shfl_sync(0xffffffffu, my_u, l);
          const uint32_t fl = __shfl_sync(0xffffffffu, my_flags, l);
          t.page = __shfl_sync(0xffffffffu, task.page, l);
          t.lo = __shfl_sync(0xffffffffu, task.lo, l);
          t.hi = __shfl_sync(0xffffffffu, task.hi, l);
          t.ie = __shfl_sync(0xffffffffu, task.ie, l);
          t.ws = __shfl_sync(0xffffffffu, task.ws, l);
          if (lane == 0) issue_stage<D>(a, maps, smem, it, u, fl, t, armed, abort, eflags);
          abort = __shfl_sync(0xffffffffu, abort, 0);
          ++it;
        }
      }
    }
    if (lane == 0) {
      PageTask none;
      none.page = -1;
      none.lo = none.hi = none.ie = none.ws = 0;
      issue_stage<D>(a, maps, smem, it, -1, kLast, none, armed, abort, eflags);  // sentinel
      // Drain: every copy this CTA issued must land before the CTA exits.
      const int64_t first = armed > C::kStages ? armed - C::kStages : 0;
      for (int64_t i = first; i < armed; ++i)
        if (!mbar_wait(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1)) ||
            !mbar_wait(&full_v[i % C::kStages], (uint32_t)((i / C::kStages) & 1))) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          break;
        }
    }
    eflags = __reduce_or_sync(0xffffffffu, eflags);
    if (lane == 0) raise_flags(a.error_flags, eflags);
    return;
  }

  // -------------------------------------------------------------------- consumers
  const Lane ln{lane >> 2, lane & 3};
  const int row0 = warp * 16;
  SoftmaxState<D> st;
  st.reset();
  uint32_t qb[C::KJ][4];
#pragma unroll
  for (int j = 0; j < C::KJ; ++j) qb[j][0] = qb[j][1] = qb[j][2] = qb[j][3] = 0u;
  bool abort = false;
  int32_t merges = 0;
  for (int64_t it = 0;; ++it) {
    const int s = (int)(it % C::kStages);
    if (!mbar_wait(&full[s], (uint32_t)((it / C::kStages) & 1))) {
      if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      break;
    }
    const StageInfo inf = sInfo[s];
    if (inf.flags & kLast) break;
    if (inf.flags & kNewUnit) {
      st.reset();
      const unsigned char* q = sQ + (size_t)s * C::kQBytes;
#pragma unroll
      for (int j = 0; j < C::KJ; ++j) {
        if (ln.g < a.G) {
          const int4 v = lds128(q + ((size_t)ln.g * D + 32 * j + 8 * ln.t) * 2);
          qb[j][0] = v.x;
          qb[j][1] = v.y;
          qb[j][2] = v.z;
          qb[j][3] = v.w;
        } else {
          qb[j][0] = qb[j][1] = qb[j][2] = qb[j][3] = 0u;
        }
      }
    }
    if (row0 < inf.hi && row0 + 16 > inf.lo) {
      const unsigned char* k = sK + (size_t)s * C::kSlab;
      const unsigned char* v = sV + (size_t)s * C::kSlab;
      // ---- S^T = K . Q^T
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int ra = row0 + tile_token(ln.g), rb = ra + 8;
#pragma unroll
      for (int j = 0; j < C::KJ; ++j) {
        const int4 k0 = lds128(k + swz(ra, 4 * j + ln.t));
        const int4 k1 = lds128(k + swz(rb, 4 * j + ln.t));
        mma_16816(sacc, k0.x, k1.x, k0.y, k1.y, qb[j][0], qb[j][1]);
        mma_16816(sacc, k0.z, k1.z, k0.w, k1.w, qb[j][2], qb[j][3]);
      }
      // ---- mask, online softmax (log2 domain)
      const bool va = ra >= inf.lo && ra < inf.hi && (ra < inf.ie || ra >= inf.ws);
      const bool vb = rb >= inf.lo && rb < inf.hi && (rb < inf.ie || rb >= inf.ws);
      const float s0 = va ? sacc[0] * a.scale_log2 : -INFINITY;
      const float s1 = va ? sacc[1] * a.scale_log2 : -INFINITY;
      const float s2 = vb ? sacc[2] * a.scale_log2 : -INFINITY;
      const float s3 = vb ? sacc[3] * a.scale_log2 : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;
      const float base1 = mn1 == -INFINITY ? 0.f : mn1;
      const float alpha0 = fast_exp2(st.m[0] - base0);
      const float alpha1 = fast_exp2(st.m[1] - base1);
      st.m[0] = mn0;
      st.m[1] = mn1;
      const uint32_t p01 = pack_bf16(fast_exp2(s0 - base0), fast_exp2(s1 - base1));
      const uint32_t p23 = pack_bf16(fast_exp2(s2 - base0), fast_exp2(s3 - base1));
      st.l[0] = st.l[0] * alpha0 + bf16_lo(p01) + bf16_lo(p23);
      st.l[1] = st.l[1] * alpha1 + bf16_hi(p01) + bf16_hi(p23);
#pragma unroll
      for (int i = 0; i < C::MT; ++i) {
        st.acc[i][0] *= alpha0;
        st.acc[i][1] *= alpha1;
        st.acc[i][2] *= alpha0;
        st.acc[i][3] *= alpha1;
      }
      const uint32_t b0 = movmatrix_trans(p01);  // (head g, tokens 2t, 2t+1)
      const uint32_t b1 = movmatrix_trans(p23);  // (head g, tokens 2t+8, 2t+9)
      // ---- O^T += V^T . P, once V has landed
      if (!mbar_wait(&full_v[s], (uint32_t)((it / C::kStages) & 1))) {
        if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
        break;
      }
      int4 vt[4][C::NCH];
      const int trow[4] = {row0 + tile_token(2 * ln.t), row0 + tile_token(2 * ln.t + 1),
                           row0 + tile_token(2 * ln.t + 8), row0 + tile_token(2 * ln.t + 9)};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const bool in = trow[x] >= inf.lo && trow[x] < inf.hi;
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          vt[x][c] = in ? lds128(v + swz(trow[x], ln.g + 8 * c))
                        : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < C::MT; ++i) {
        const int v0 = i, v1 = C::MT + i;  // value indices of rows g and g+8
        const int c0 = v0 >> 3, e0 = v0 & 7, c1 = v1 >> 3, e1 = v1 & 7;
        const uint32_t sel0 = (e0 & 1) ? 0x7632u : 0x5410u;
        const uint32_t sel1 = (e1 & 1) ? 0x7632u : 0x5410u;
        auto word = [](const int4& x, int w) -> uint32_t {
          return (uint32_t)(w == 0 ? x.x : w == 1 ? x.y : w == 2 ? x.z : x.w);
        };
        const uint32_t a0 = __byte_perm(word(vt[0][c0], e0 >> 1), word(vt[1][c0], e0 >> 1), sel0);
        const uint32_t a1 = __byte_perm(word(vt[0][c1], e1 >> 1), word(vt[1][c1], e1 >> 1), sel1);
        const uint32_t a2 = __byte_perm(word(vt[2][c0], e0 >> 1), word(vt[3][c0], e0 >> 1), sel0);
        const uint32_t a3 = __byte_perm(word(vt[2][c1], e1 >> 1), word(vt[3][c1], e1 >> 1), sel1);
        mma_16816(st.acc[i], a0, a1, a2, a3, b0, b1);
      }
    }
    // release the stage
    warp_arrive(&empty[s]);

    if (inf.flags & kSegEnd) {
      // ---- reduce the per-lane sums, merge the 8 warps, write the partial
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
        st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
      }
      const uint32_t ph = (uint32_t)(merges & 1);
      if (warp >= 4) {
        if (merges > 0 && !mbar_wait(mb_r2, ph ^ 1u)) abort = true;
        st.store(sMerge + (warp - 4) * C::kMergeSlot, lane);
        warp_arrive(mb_w1);
      } else {
        if (!mbar_wait(mb_w1, ph)) abort = true;
        st.merge_from(sMerge + warp * C::kMergeSlot, lane);
        if (warp >= 1) {
          st.store(sMerge + warp * C::kMergeSlot, lane);
          warp_arrive(mb_w2);
        } else {
          if (!mbar_wait(mb_w2, ph)) abort = true;
          for (int w = 1; w < 4; ++w) st.merge_from(sMerge + w * C::kMergeSlot, lane);
          warp_arrive(mb_r2);
          // warp 0 writes the partial of (unit, this CTA) into the list's bank
          const int64_t slot = ((inf.flags & kBankB) ? (int64_t)a.lay.bank : 0) + inf.unit +
                               blockIdx.x;
          float* accp = reinterpret_cast<float*>(a.ws + a.lay.acc) + slot * a.G * D;
          float* mlp = reinterpret_cast<float*>(a.ws + a.lay.ml) + slot * a.G * 2;
          const int h0 = 2 * ln.t, h1 = h0 + 1;
          // values 4k..4k+3 of a lane sit at 4 consecutive d (d_of): 16-byte stores
#pragma unroll
          for (int k4 = 0; k4 < C::MT; k4 += 4) {
            const int da = d_of<D>(ln.g, k4), db = d_of<D>(ln.g, C::MT + k4);
            if (h0 < a.G) {
              *reinterpret_cast<float4*>(accp + h0 * D + da) = make_float4(
                  st.acc[k4][0], st.acc[k4 + 1][0], st.acc[k4 + 2][0], st.acc[k4 + 3][0]);
              *reinterpret_cast<float4*>(accp + h0 * D + db) = make_float4(
                  st.acc[k4][2], st.acc[k4 + 1][2], st.acc[k4 + 2][2], st.acc[k4 + 3][2]);
            }
            if (h1 < a.G) {
              *reinterpret_cast<float4*>(accp + h1 * D + da) = make_float4(
                  st.acc[k4][1], st.acc[k4 + 1][1], st.acc[k4 + 2][1], st.acc[k4 + 3][1]);
              *reinterpret_cast<float4*>(accp + h1 * D + db) = make_float4(
                  st.acc[k4][3], st.acc[k4 + 1][3], st.acc[k4 + 2][3], st.acc[k4 + 3][3]);
            }
          }
          if (ln.g == 0) {
            if (h0 < a.G) {
              mlp[h0 * 2 + 0] = st.m[0];
              mlp[h0 * 2 + 1] = st.l[0];
            }
            if (h1 < a.G) {
              mlp[h1 * 2 + 0] = st.m[1];
              mlp[h1 * 2 + 1] = st.l[1];
            }
          }
        }
      }
      ++merges;
      if (abort) {
        if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
        break;
      }
    }
  }
}

}  // namespace

bool mma_split_supported(const srkv_config& cfg) {
  const int32_t G = cfg.num_q_heads / cfg.num_kv_heads;
  return cfg.dtype == SRKV_BF16 && (cfg.head_dim == 128 || cfg.head_dim == 64) && G >= 1 &&
         G <= 8;
}

int32_t mma_split_ctas(int32_t sm_count) { return sm_count; }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiled encode_tiled() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [num_pages][Hkv * 128][d] bf16, boxes of 64 columns x 128 rows, 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_pages, int32_t Hkv,
                      int32_t d) {
  const EncodeTiled fn = encode_tiled();
  if (!fn || num_pages > INT32_MAX || (int64_t)Hkv * kBlock > INT32_MAX) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hkv * kBlock, (cuuint64_t)num_pages};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * kBlock * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kBlock, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t stream) {
  // The shared-memory opt-in is set once per device (not during graph capture).
  static bool configured[128] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(split_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg<D>::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  TmaMaps maps;
  if (!encode_cache_map(&maps.k, a.k_cache, a.num_pages, a.Hkv, D) ||
      !encode_cache_map(&maps.v, a.v_cache, a.num_pages, a.Hkv, D))
    return cudaErrorInvalidValue;
  return launch_pdl(split_mma_kernel<D>, dim3(a.ctas), dim3(kThreads), Cfg<D>::kSmemAlloc, stream,
                    a, maps);
}

cudaError_t launch_split_mma(const DecodeArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace srkv
