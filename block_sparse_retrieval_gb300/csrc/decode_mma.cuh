// decode_mma.cuh -- pieces shared by the tensor-core decode kernels: the stage ring (tiled
// TMA copies of whole K/V slabs with a 128-byte swizzle, one mbarrier for K and the query and
// one for V), the softmax state of a warp, and the consumer loop that turns stages into
// partial results (max, sum, unnormalised output) per segment.
//
// Attention is softmax(QK^T/sqrt(d_k))V over the attended rows of each page (ATB reuse
// article, §1.1); the consumer warps run it on m16n8k16 bf16 MMAs with the group's queries as
// the N = 8 side:  S^T[16 tok x 8 heads] = K[16 x d] . Q^T[d x 8],  O^T[d x 8] += V^T . P.
// MMA tile row m holds token m ^ 4 (m odd) or m (m even): with the swizzle, every 8-lane
// phase of a 16-byte fragment load then reads 8 distinct bank groups.  The contraction index
// of each product may be permuted consistently on both operands, so every fragment comes
// from 16-byte shared loads; P^T -> P is one movmatrix.trans per 8x8 block.  Online softmax
// in fp32, log2 domain; the sum uses the bf16-rounded weights the MMA sees.  Rows outside a
// stage's loaded range are masked in the logits and zeroed in V.  Over compressed pages (E4M3
// codes with fp32 row scales) K's scale multiplies the logits and V's scale the weights, so
// both products take the widened codes as they are.
#pragma once

#include "decode_plan.cuh"

namespace srkv {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr uint32_t kNewUnit = 1, kSegEnd = 2, kBankB = 4, kLast = 8;
// Compressed pages: factor on the V-scaled weights and on their sum (a power of two).
constexpr float kPScale = 256.f;

struct StageInfo {
  int32_t unit;
  int32_t flags;
  int32_t lo, hi, ie, ws;
  int32_t pad[2];
};

// F8: the pages hold E4M3 codes (one byte per value) and each stage also carries the 128
// K and 128 V row scales of its page.
template <int D, bool F8 = false>
struct Cfg {
  static_assert(!F8 || D == 128, "compressed pages: d 128");
  static constexpr int kElem = F8 ? 1 : 2;              // bytes per cached value
  static constexpr int kSlab = kBlock * D * kElem;      // bytes of one K or V slab
  static constexpr int kStages = F8 ? 5 : (D == 128 ? 3 : 6);
  static constexpr int kQBytes = 8 * D * 2;              // up to 8 query heads
  static constexpr int MT = D / 16;                      // PV m-tiles over d
  static constexpr int KJ = D / 32;                      // 16-byte K chunks per thread-row
  static constexpr int NCH = D / 64;                     // 16-byte V chunks per token
  static constexpr int kMergeStride = MT * 4 + 4;        // floats per lane in a merge slot
  static constexpr int kMergeSlot = 32 * kMergeStride;   // floats per merge slot

  static constexpr size_t kOffK = 0;
  static constexpr size_t kOffV = kOffK + (size_t)kStages * kSlab;
  static constexpr size_t kOffQ = kOffV + (size_t)kStages * kSlab;
  static constexpr int kScaleBytes = F8 ? 2 * kBlock * 4 : 0;  // K, then V row scales
  static constexpr size_t kOffScale = kOffQ + (size_t)kStages * kQBytes;
  static constexpr size_t kOffMerge = kOffScale + (size_t)kStages * kScaleBytes;
  static constexpr size_t kOffInfo = kOffMerge + sizeof(float) * 4 * kMergeSlot;
  static constexpr size_t kOffBar = kOffInfo + sizeof(StageInfo) * kStages;
  // full (K, query, stage info)[kStages], full_v[kStages], empty[kStages], merge w1, w2, r2
  static constexpr size_t kSmem = kOffBar + sizeof(uint64_t) * (3 * kStages + 3);
  static constexpr size_t kSmemAlloc = kSmem + 1024;  // the swizzled stages need 1 KiB alignment
  static constexpr int kBoxes = D * kElem / 128;       // 128-byte-wide TMA boxes per slab
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
template <int D, bool F8 = false>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const TmaMaps& maps,
                                            unsigned char* smem, int64_t it, int32_t u,
                                            uint32_t fl, const PageTask& t, int64_t& armed,
                                            bool& abort, uint32_t& eflags) {
  using C = Cfg<D, F8>;
  if (abort) return;
  StageInfo* sInfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;
  const int s = (int)(it % C::kStages);
  if (it >= C::kStages && !mbar_wait(&empty[s], (uint32_t)((it / C::kStages - 1) & 1))) {
    // Copies already armed may still be landing in the ring: every caller, on this path as
    // on the normal one, waits (bounded) for the last kStages armed stages before its CTA ends.
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
  constexpr uint32_t kRowScales = F8 ? kBlock * 4 : 0;  // one fp32 scale per row
  if (!F8 && rows && t.page >= a.num_pages) {
    // A page of the host pool: the producer warp copies its slabs and then arrives
    // (issue_stage_warp); here only the query's bytes are announced and requested.
    if (fl & kNewUnit) {
      const int32_t h = u % a.Hkv, r = u / a.Hkv;
      mbar_expect_tx(&full[s], qbytes);
      bulk_load(smem + C::kOffQ + (size_t)s * C::kQBytes,
                static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * D,
                qbytes, &full[s]);
    }
    return;
  }
  // (compressed pages: both row-scale vectors complete `full`, since V's scales go into the
  // weights, which are formed before V is read)
  mbar_arrive_expect_tx(&full[s], (rows ? (uint32_t)C::kSlab + 2 * kRowScales : 0u) +
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
                  b * 128 / C::kElem, h * kBlock, t.page, &full[s], once);
    if constexpr (F8)
      bulk_load_hint(smem + C::kOffScale + (size_t)s * C::kScaleBytes,
                     a.k_scale + ((int64_t)t.page * a.Hkv + h) * kBlock, kRowScales, &full[s],
                     once);
  }
  if (fl & kNewUnit)
    bulk_load(smem + C::kOffQ + (size_t)s * C::kQBytes,
              static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * D,
              qbytes, &full[s]);
  if (rows) {
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_3d(smem + C::kOffV + (size_t)s * C::kSlab + (size_t)b * C::kBoxBytes, &maps.v,
                  b * 128 / C::kElem, h * kBlock, t.page, &full_v[s], once);
    if constexpr (F8)
      bulk_load_hint(smem + C::kOffScale + (size_t)s * C::kScaleBytes + kRowScales,
                     a.v_scale + ((int64_t)t.page * a.Hkv + h) * kBlock, kRowScales,
                     &full[s], once);
  }
}

// issue_stage for the whole producer warp (every lane calls it with the same arguments).  A
// page of the host pool is copied by all 32 lanes, 16 bytes per cp.async, into the layout the
// tensor-map copies produce (128-byte swizzle), so the consumers read both kinds of stage
// alike: over NVLink-C2C the host pool is read in place, with no staging copy in HBM.  Each
// lane ties its copies to the stage's barriers, then lane 0 arrives.
template <int D, bool F8 = false>
__device__ __forceinline__ void issue_stage_warp(const DecodeArgs& a, const TmaMaps& maps,
                                                 unsigned char* smem, int64_t it, int32_t u,
                                                 uint32_t fl, const PageTask& t, int64_t& armed,
                                                 bool& abort, uint32_t& eflags, int lane) {
  using C = Cfg<D, F8>;
  // (compressed pages have no host pool)
  const bool host = !F8 && t.page >= 0 && t.hi > t.lo && t.page >= a.num_pages;  // uniform
  if (lane == 0) issue_stage<D, F8>(a, maps, smem, it, u, fl, t, armed, abort, eflags);
  abort = __shfl_sync(0xffffffffu, abort, 0);
  if (!host || abort) return;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  const int s = (int)(it % C::kStages);
  const int64_t slab = ((int64_t)(t.page - a.num_pages) * a.Hkv + u % a.Hkv) * kBlock * D;
  const __nv_bfloat16* ks = static_cast<const __nv_bfloat16*>(a.k_host) + slab;
  const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(a.v_host) + slab;
  const uint32_t k_dst = smem_u32(smem + C::kOffK + (size_t)s * C::kSlab);
  const uint32_t v_dst = smem_u32(smem + C::kOffV + (size_t)s * C::kSlab);
  constexpr int kPerRow = D / 8;  // 16-byte chunks per row
  // lane i copies chunks i, i + 32, ...: consecutive lanes read consecutive 16 bytes
#pragma unroll 8
  for (int i = lane; i < kBlock * kPerRow; i += 32)
    cp_async_16(k_dst + swz(i / kPerRow, i % kPerRow), ks + (int64_t)i * 8);
  cp_async_mbar_arrive(&full[s]);
#pragma unroll 8
  for (int i = lane; i < kBlock * kPerRow; i += 32)
    cp_async_16(v_dst + swz(i / kPerRow, i % kPerRow), vs + (int64_t)i * 8);
  cp_async_mbar_arrive(&full_v[s]);
  __syncwarp();  // every lane's pending-count increments precede the arrivals below
  if (lane == 0) {
    mbar_arrive(&full[s]);
    mbar_arrive(&full_v[s]);
    ++armed;
  }
}

// One arrival per warp: the warp's lanes synchronise (ordering their shared-memory accesses)
// and one lane arrives for all of them.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// A merged state (acc, m, l of the lane's two heads) as a partial of acc[G][D] and ml[G][2]
// floats: put4(i, v) for the 16-byte piece at acc[i], put2(j, v) for (m, l) at ml[j].
template <int D, bool F8, typename Put4, typename Put2>
__device__ __forceinline__ void emit_partial(const SoftmaxState<D>& st, Lane ln, int G,
                                             Put4 put4, Put2 put2) {
  using C = Cfg<D>;
  const int h0 = 2 * ln.t, h1 = h0 + 1;
  if constexpr (F8) {
    // compressed pages: m-tile i row g holds d = 16g + 2i, row g + 8 holds d = 16g + 2i + 1,
    // so the lane's 16 values per head are d = 16g .. 16g + 15 in the order
    // (i 0 row g, i 0 row g+8, i 1 row g, ...)
#pragma unroll
    for (int k4 = 0; k4 < C::MT; k4 += 2) {
      const int dd = 16 * ln.g + 2 * k4;
      if (h0 < G)
        put4(h0 * D + dd,
             make_float4(st.acc[k4][0], st.acc[k4][2], st.acc[k4 + 1][0], st.acc[k4 + 1][2]));
      if (h1 < G)
        put4(h1 * D + dd,
             make_float4(st.acc[k4][1], st.acc[k4][3], st.acc[k4 + 1][1], st.acc[k4 + 1][3]));
    }
  } else {
    // values 4k..4k+3 of a lane sit at 4 consecutive d (d_of): 16-byte pieces
#pragma unroll
    for (int k4 = 0; k4 < C::MT; k4 += 4) {
      const int da = d_of<D>(ln.g, k4), db = d_of<D>(ln.g, C::MT + k4);
      if (h0 < G) {
        put4(h0 * D + da, make_float4(st.acc[k4][0], st.acc[k4 + 1][0], st.acc[k4 + 2][0],
                                      st.acc[k4 + 3][0]));
        put4(h0 * D + db, make_float4(st.acc[k4][2], st.acc[k4 + 1][2], st.acc[k4 + 2][2],
                                      st.acc[k4 + 3][2]));
      }
      if (h1 < G) {
        put4(h1 * D + da, make_float4(st.acc[k4][1], st.acc[k4 + 1][1], st.acc[k4 + 2][1],
                                      st.acc[k4 + 3][1]));
        put4(h1 * D + db, make_float4(st.acc[k4][3], st.acc[k4 + 1][3], st.acc[k4 + 2][3],
                                      st.acc[k4 + 3][3]));
      }
    }
  }
  if (ln.g == 0) {
    if (h0 < G) put2(h0 * 2, make_float2(st.m[0], st.l[0]));
    if (h1 < G) put2(h1 * 2, make_float2(st.m[1], st.l[1]));
  }
}

// Writes a merged state as a partial through generic pointers (global memory or another
// CTA's shared memory).
template <int D, bool F8 = false>
__device__ __forceinline__ void store_partial(float* accp, float* mlp, const SoftmaxState<D>& st,
                                              Lane ln, int G) {
  emit_partial<D, F8>(
      st, ln, G, [&](int i, float4 v) { *reinterpret_cast<float4*>(accp + i) = v; },
      [&](int j, float2 v) {
        mlp[j] = v.x;
        mlp[j + 1] = v.y;
      });
}

// The 8 consumer warps' loop over the stages the producer hands out, until the sentinel.
// At the end of each segment (a stage flagged kSegEnd; the sentinel may carry the flag too,
// closing a segment whose length the producer did not know in advance) the warps merge their
// states and warp 0 calls write_partial(state, stage info, lane) with the merged state.
template <int D, bool F8 = false, typename WritePartial>
__device__ __forceinline__ void consumer_loop(const DecodeArgs& a, unsigned char* smem, int lane,
                                              int warp, WritePartial&& write_partial) {
  using C = Cfg<D, F8>;
  unsigned char* sK = smem + C::kOffK;
  unsigned char* sV = smem + C::kOffV;
  unsigned char* sQ = smem + C::kOffQ;
  const float* sScale = reinterpret_cast<const float*>(smem + C::kOffScale);
  float* sMerge = reinterpret_cast<float*>(smem + C::kOffMerge);
  StageInfo* sInfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;
  uint64_t* mb_w1 = empty + C::kStages;
  uint64_t* mb_w2 = mb_w1 + 1;
  uint64_t* mb_r2 = mb_w1 + 2;
  const Lane ln{lane >> 2, lane & 3};
  const int row0 = warp * 16;
  SoftmaxState<D> st;
  st.reset();
  uint32_t qb[C::KJ][4];
#pragma unroll
  for (int j = 0; j < C::KJ; ++j) qb[j][0] = qb[j][1] = qb[j][2] = qb[j][3] = 0u;
  bool abort = false;
  int32_t merges = 0;
  // End of a segment: reduce the per-lane sums, merge the 8 warps, write the partial.
  auto close_segment = [&](const StageInfo& inf) {
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
        write_partial(st, inf, ln);
      }
    }
    ++merges;
  };
  for (int64_t it = 0;; ++it) {
    const int s = (int)(it % C::kStages);
    if (!mbar_wait(&full[s], (uint32_t)((it / C::kStages) & 1))) {
      if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      break;
    }
    const StageInfo inf = sInfo[s];
    if (inf.flags & kLast) {  // the sentinel; it may close the last segment
      if (inf.flags & kSegEnd) {
        close_segment(inf);
        if (abort && lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
      }
      break;
    }
    if (inf.flags & kNewUnit) {
      st.reset();
      const unsigned char* q = sQ + (size_t)s * C::kQBytes;
      if constexpr (F8) {
        // fp16 query in the order the E4M3 K fragments take d (see the S^T product below):
        // k-step m of lane t covers d = 64 (m >= 4) + 16 t + 4 (m mod 4) + 0..3
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          uint32_t lo = 0u, hi = 0u;
          if (ln.g < a.G) {
            const uint2 w = *reinterpret_cast<const uint2*>(
                q + ((size_t)ln.g * D + 64 * (m >> 2) + 16 * ln.t + 4 * (m & 3)) * 2);
            lo = pack_f16(bf16_lo(w.x), bf16_hi(w.x));
            hi = pack_f16(bf16_lo(w.y), bf16_hi(w.y));
          }
          qb[m >> 1][2 * (m & 1)] = lo;
          qb[m >> 1][2 * (m & 1) + 1] = hi;
        }
      } else {
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
    }
    if (row0 < inf.hi && row0 + 16 > inf.lo) {
      const unsigned char* k = sK + (size_t)s * C::kSlab;
      const unsigned char* v = sV + (size_t)s * C::kSlab;
      // ---- S^T = K . Q^T
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int ra = row0 + tile_token(ln.g), rb = ra + 8;
      if constexpr (F8) {
        // a row is 128 codes in 8 chunks of 16; lane t reads chunks t and t + 4 of rows ra,
        // rb, and byte pairs of a chunk widen to fp16 pairs (exact): 8 k-steps of 16
        const int4 kq[2][2] = {{lds128(k + swz(ra, ln.t)), lds128(k + swz(rb, ln.t))},
                               {lds128(k + swz(ra, 4 + ln.t)), lds128(k + swz(rb, 4 + ln.t))}};
        auto word = [](const int4& x, int w) -> uint32_t {
          return (uint32_t)(w == 0 ? x.x : w == 1 ? x.y : w == 2 ? x.z : x.w);
        };
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint32_t wa = word(kq[m >> 2][0], m & 3), wb = word(kq[m >> 2][1], m & 3);
          mma_16816_f16(sacc, e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb),
                        e4m3x2_to_f16x2(wa >> 16), e4m3x2_to_f16x2(wb >> 16),
                        qb[m >> 1][2 * (m & 1)], qb[m >> 1][2 * (m & 1) + 1]);
        }
        // the rows' K scales (a masked row's scale is never used)
        const float* ks = sScale + (size_t)s * (C::kScaleBytes / 4);
        const float ka = ks[ra], kb = ks[rb];
        sacc[0] *= ka;
        sacc[1] *= ka;
        sacc[2] *= kb;
        sacc[3] *= kb;
      } else {
#pragma unroll
        for (int j = 0; j < C::KJ; ++j) {
          const int4 k0 = lds128(k + swz(ra, 4 * j + ln.t));
          const int4 k1 = lds128(k + swz(rb, 4 * j + ln.t));
          mma_16816(sacc, k0.x, k1.x, k0.y, k1.y, qb[j][0], qb[j][1]);
          mma_16816(sacc, k0.z, k1.z, k0.w, k1.w, qb[j][2], qb[j][3]);
        }
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
      uint32_t p01, p23;  // the weights as the second product's operand rounds them
      if constexpr (F8) {
        // V's row scales go into the weights: O^T += codes^T . (P scale), one multiply per
        // (token, head) instead of one per value.  kPScale (a power of two) keeps the scaled
        // weights near the range of the weights themselves in fp16, and the sum carries the
        // same factor, so it cancels in the output.  A row outside the loaded range gets
        // scale 0 (its smem scale is not data).
        const float* vsp = sScale + (size_t)s * (C::kScaleBytes / 4) + kBlock;
        const float sa = (ra >= inf.lo && ra < inf.hi) ? vsp[ra] * kPScale : 0.f;
        const float sb = (rb >= inf.lo && rb < inf.hi) ? vsp[rb] * kPScale : 0.f;
        const float e0 = fast_exp2(s0 - base0), e1 = fast_exp2(s1 - base1);
        const float e2 = fast_exp2(s2 - base0), e3 = fast_exp2(s3 - base1);
        p01 = pack_f16(e0 * sa, e1 * sa);
        p23 = pack_f16(e2 * sb, e3 * sb);
        st.l[0] = st.l[0] * alpha0 + (e0 + e2) * kPScale;
        st.l[1] = st.l[1] * alpha1 + (e1 + e3) * kPScale;
      } else {
        p01 = pack_bf16(fast_exp2(s0 - base0), fast_exp2(s1 - base1));
        p23 = pack_bf16(fast_exp2(s2 - base0), fast_exp2(s3 - base1));
        st.l[0] = st.l[0] * alpha0 + bf16_lo(p01) + bf16_lo(p23);
        st.l[1] = st.l[1] * alpha1 + bf16_hi(p01) + bf16_hi(p23);
      }
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
      const int trow[4] = {row0 + tile_token(2 * ln.t), row0 + tile_token(2 * ln.t + 1),
                           row0 + tile_token(2 * ln.t + 8), row0 + tile_token(2 * ln.t + 9)};
      if constexpr (F8) {
        // O^T += codes^T . (P scale): m-tile i takes d = 16 g + 2 i (row g) and 16 g + 2 i + 1
        // (row g + 8) from the lane's chunk g of the four token rows; a byte permute pairs the
        // two tokens of each product row, widened to fp16 (exact).  Rows outside the loaded
        // range load as zero codes (their smem bytes are not data).
        int4 vq[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const bool in = trow[x] >= inf.lo && trow[x] < inf.hi;
          vq[x] = in ? lds128(v + swz(trow[x], ln.g)) : make_int4(0, 0, 0, 0);
        }
        auto word = [](const int4& x, int w) -> uint32_t {
          return (uint32_t)(w == 0 ? x.x : w == 1 ? x.y : w == 2 ? x.z : x.w);
        };
#pragma unroll
        for (int i = 0; i < C::MT; ++i) {
          const int wi = i >> 1, bo = 2 * (i & 1);
          // bytes (token a, d0), (token b, d0), (token a, d1), (token b, d1)
          const uint32_t sel =
              (uint32_t)(bo | ((4 + bo) << 4) | ((bo + 1) << 8) | ((5 + bo) << 12));
          const uint32_t x01 = __byte_perm(word(vq[0], wi), word(vq[1], wi), sel);
          const uint32_t x23 = __byte_perm(word(vq[2], wi), word(vq[3], wi), sel);
          mma_16816_f16(st.acc[i], e4m3x2_to_f16x2(x01), e4m3x2_to_f16x2(x01 >> 16),
                        e4m3x2_to_f16x2(x23), e4m3x2_to_f16x2(x23 >> 16), b0, b1);
        }
      } else {
        int4 vt[4][C::NCH];
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
    }
    // release the stage
    warp_arrive(&empty[s]);

    if (inf.flags & kSegEnd) {
      close_segment(inf);
      if (abort) {
        if (lane == 0) raise_flags(a.error_flags, SRKV_EFLAG_TIMEOUT);
        break;
      }
    }
  }
}

// Barrier setup of the stage ring (one thread; fenced for the async proxy and the cluster).
template <int D, bool F8 = false>
__device__ __forceinline__ void init_ring(unsigned char* smem) {
  using C = Cfg<D, F8>;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;
  uint64_t* mb_w1 = empty + C::kStages;
  for (int s = 0; s < C::kStages; ++s) {
    mbar_init(&full[s], 1);
    mbar_init(&full_v[s], 1);
    mbar_init(&empty[s], kConsumerWarps);  // one arrival per consumer warp
  }
  mbar_init(mb_w1, 4);
  mbar_init(mb_w1 + 1, 3);
  mbar_init(mb_w1 + 2, 1);
  fence_mbar_init();
}

// Host: tensor map of a cache [num_pages][Hkv * 128][d] of bf16 (64-column x 128-row boxes)
// or of E4M3 bytes (128-column boxes), 128-byte swizzle; false if it cannot be encoded.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_pages, int32_t Hkv,
                      int32_t d, bool e4m3);

}  // namespace srkv
