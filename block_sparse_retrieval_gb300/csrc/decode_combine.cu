// decode_combine.cu -- merge of the split partials into the attention output.
//
// KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV cache共享": partial
// attention results over disjoint KV subsets are merged the Flash-Decoding way.  With
// partial i = (m_i, l_i, acc_i) in the log2 domain:
//   out = sum_i 2^(m_i - m*) acc_i / sum_i 2^(m_i - m*) l_i,   m* = max_i m_i.
// One CTA of 4 warps per (request, q head).  The partials of a unit are those of the CTAs
// whose position ranges meet the unit's two lists (decode_plan.cuh).  For batches of at most
// 64 units the CTA derives those ranges from the lengths and selection counts before it
// waits for the split grid, so that after the wait a single round of independent loads
// fetches every partial (16 per warp, vector loads of d); larger batches read the unit
// offsets the split kernel left in the workspace first.  A unit with no positions (L = 0)
// gets a zero output.  Launched as a programmatic dependent of the split kernel.
#include "decode_plan.cuh"

namespace srkv {
namespace {


constexpr int kWarps = 4;
constexpr int kPartsPerWarp = 16;
constexpr int kRound = kWarps * kPartsPerWarp;  // partials fetched per round of loads
constexpr int32_t kDirectUnits = 64;            // up to here the offsets are derived

// Where the partials of unit u in one list are: the list has T positions, the unit's are
// [P, P + n).
struct ListParts {
  int64_t T, C, c_first, slot0;  // C: CTAs sharing the list
  int32_t parts;
};

__device__ __forceinline__ ListParts list_parts(int64_t C, int64_t T, int64_t P, int64_t n,
                                                int64_t bank, int32_t u) {
  ListParts lp;
  lp.T = T;
  lp.C = C;
  lp.c_first = 0;
  lp.parts = 0;
  if (n > 0 && T > 0) {
    lp.c_first = cta_of(P, T, C);
    lp.parts = (int32_t)(cta_of(P + n - 1, T, C) - lp.c_first + 1);
  }
  lp.slot0 = bank + u + lp.c_first;
  return lp;
}

__device__ __forceinline__ int32_t warp_inclusive_scan(int32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Offsets of unit u in one list from the counts of all U <= 64 units (lane l counts units l
// and l + 32); every lane returns the same.
__device__ __forceinline__ ListParts direct_parts(const DecodeArgs& a, int list, int64_t bank,
                                                  int32_t u) {
  const int lane = threadIdx.x & 31;
  const int32_t U = a.batch * a.Hkv;
  uint32_t dummy = 0;
  const int32_t c0 = lane < U ? list_count(a, list, lane, dummy) : 0;
  const int32_t c1 = lane + 32 < U ? list_count(a, list, lane + 32, dummy) : 0;
  const int32_t s0 = warp_inclusive_scan(c0, lane), s1 = warp_inclusive_scan(c1, lane);
  const int32_t t0 = __shfl_sync(0xffffffffu, s0, 31), t1 = __shfl_sync(0xffffffffu, s1, 31);
  const int src = u & 31;
  const int32_t b0 = __shfl_sync(0xffffffffu, s0 - c0, src);
  const int32_t n0 = __shfl_sync(0xffffffffu, c0, src);
  const int32_t b1 = __shfl_sync(0xffffffffu, s1 - c1, src);
  const int32_t n1 = __shfl_sync(0xffffffffu, c1, src);
  const int64_t P = u < 32 ? (int64_t)b0 : (int64_t)t0 + b1;
  return list_parts(list_ctas(a, list), (int64_t)t0 + t1, P, u < 32 ? n0 : n1, bank, u);
}

// Offsets of unit u from those the split kernel's CTA 0 left in the workspace.
__device__ __forceinline__ ListParts stored_parts(const DecodeArgs& a, int list, int64_t bank,
                                                  int32_t u) {
  const int64_t* o = reinterpret_cast<const int64_t*>(
      a.ws + (list == kListA ? a.lay.off_a : a.lay.off_b));
  const int32_t U = a.batch * a.Hkv;
  return list_parts(list_ctas(a, list), o[U], o[u], o[u + 1] - o[u], bank, u);
}

// Slot of part i of a list, or -1 when that CTA owns no position of the list.
__device__ __forceinline__ int64_t part_slot(const ListParts& lp, int32_t i) {
  if (lp.T < lp.C) {  // only then can a CTA's range be empty
    const int64_t c = lp.c_first + i;
    if (cta_begin(c, lp.T, lp.C) == cta_begin(c + 1, lp.T, lp.C)) return -1;
  }
  return lp.slot0 + i;
}

// Slot of part p of unit u: list A's parts, then list B's, then the unit's shared-prefix
// partials (one per block range of the cascade kernel), or -1 for a part that is absent.
__device__ __forceinline__ int64_t unit_part_slot(const DecodeArgs& a, const ListParts& la,
                                                  const ListParts& lb, int32_t u, int32_t p) {
  if (p < la.parts) return part_slot(la, p);
  p -= la.parts;
  if (p < lb.parts) return part_slot(lb, p);
  return a.lay.cascade + (int64_t)u * a.prefix_ranges + (p - lb.parts);
}

template <typename TOut>
__device__ __forceinline__ void store_vec(TOut* p, const float (&v)[4], int n);
template <>
__device__ __forceinline__ void store_vec<float>(float* p, const float (&v)[4], int n) {
  if (n == 4)
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4],
                                                         int n) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  if (n == 4) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(p) = a;
  }
}

// One CTA per (unit, query head).  Warp w merges parts [64 i + 16 w, 64 i + 16 w + 16) of
// every round i: lane l owns d elements [l V, l V + V) (V = d / 32) of each part, lanes
// 0..15 hold the parts' (m, l) pairs and the weights go round by shuffles.  The four warp
// results are merged through shared memory by warp 0.
template <typename TOut, int D>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const DecodeArgs a) {
  constexpr int V = D / 32;  // 4 (d 128) or 2 (d 64)
  __shared__ float s_acc[kWarps][D];
  __shared__ float s_ml[kWarps][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t G = a.G;
  const int32_t u = blockIdx.x / G, j = blockIdx.x % G;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  const int32_t U = a.batch * a.Hkv;
  const bool direct = U <= kDirectUnits;
  ListParts la, lb;
  if (direct) {  // inputs only: readable before the split grid finishes
    la = direct_parts(a, kListA, 0, u);
    lb = direct_parts(a, kListB, a.lay.bank, u);
  }
  griddep_wait();
  if (!direct) {
    la = stored_parts(a, kListA, 0, u);
    lb = stored_parts(a, kListB, a.lay.bank, u);
  }
  const float* accw = reinterpret_cast<const float*>(a.ws + a.lay.acc);
  const float* mlw = reinterpret_cast<const float*>(a.ws + a.lay.ml);
  const int32_t total = la.parts + lb.parts + a.prefix_ranges;
  float m_run = -INFINITY, l_run = 0.f, acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int32_t p0 = warp * kPartsPerWarp; p0 < total; p0 += kRound) {
    // every load of this warp's 16 parts is issued before any is used
    const int32_t p = p0 + lane;
    int64_t slot = -1;
    if (lane < kPartsPerWarp && p < total) slot = unit_part_slot(a, la, lb, u, p);
    float m = -INFINITY, l = 0.f;
    if (slot >= 0) {
      m = mlw[(slot * G + j) * 2];
      l = mlw[(slot * G + j) * 2 + 1];
    }
    float xs[kPartsPerWarp][V];
#pragma unroll
    for (int t = 0; t < kPartsPerWarp; ++t) {
      const int64_t st = __shfl_sync(0xffffffffu, slot, t);
#pragma unroll
      for (int e = 0; e < V; ++e) xs[t][e] = 0.f;
      if (st >= 0) {
        const float* src = accw + (st * G + j) * D + lane * V;
        if constexpr (V == 4) {
          const float4 v4 = *reinterpret_cast<const float4*>(src);
          xs[t][0] = v4.x;
          xs[t][1] = v4.y;
          xs[t][2] = v4.z;
          xs[t][3] = v4.w;
        } else {
          const float2 v2 = *reinterpret_cast<const float2*>(src);
          xs[t][0] = v2.x;
          xs[t][1] = v2.y;
        }
      }
    }
    float mx = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mx = fmaxf(mx, m_run);
    if (mx == -INFINITY) continue;
    const float f_run = fast_exp2(m_run - mx);
    const float w = fast_exp2(m - mx);  // 0 for an absent part
    float lw = w * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    l_run = l_run * f_run + lw;
    m_run = mx;
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] *= f_run;
#pragma unroll
    for (int t = 0; t < kPartsPerWarp; ++t) {
      const float wt = __shfl_sync(0xffffffffu, w, t);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += wt * xs[t][e];
    }
  }
  // merge the warps
#pragma unroll
  for (int e = 0; e < V; ++e) s_acc[warp][lane * V + e] = acc[e];
  if (lane == 0) {
    s_ml[warp][0] = m_run;
    s_ml[warp][1] = l_run;
  }
  __syncthreads();
  if (warp != 0) return;
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, s_ml[w][0]);
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (mx != -INFINITY) {
    float lsum = 0.f, o[V];
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = fast_exp2(s_ml[w][0] - mx);  // 0 for a warp without parts
      lsum += f * s_ml[w][1];
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] += f * s_acc[w][lane * V + e];
    }
#pragma unroll
    for (int e = 0; e < V; ++e) v[e] = lsum > 0.f ? o[e] / lsum : 0.f;
  }
  TOut* out = static_cast<TOut*>(a.out) + ((int64_t)r * a.Hq + (int64_t)h * G + j) * D + lane * V;
  store_vec<TOut>(out, v, V);
}

}  // namespace

// Batches with more units than split CTAs: a unit's positions meet few CTAs (a handful of
// partials per head), so one CTA per unit with one warp per query head (G warps) merges them,
// 16 partials per round of loads, with no cross-warp merge; the unit's offsets are found once
// per CTA.  (The kernel above spends 4 warps per head, for heads with many partials.)
template <typename TOut, int D>
__global__ void __launch_bounds__(256) combine_unit_kernel(const DecodeArgs a) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31, j = threadIdx.x >> 5;  // warp j: query head j
  const int32_t G = a.G;
  const int32_t u = blockIdx.x;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  griddep_wait();
  const ListParts la = stored_parts(a, kListA, 0, u);
  const ListParts lb = stored_parts(a, kListB, a.lay.bank, u);
  if (j >= G) return;
  const float* accw = reinterpret_cast<const float*>(a.ws + a.lay.acc);
  const float* mlw = reinterpret_cast<const float*>(a.ws + a.lay.ml);
  const int32_t total = la.parts + lb.parts + a.prefix_ranges;
  float m_run = -INFINITY, l_run = 0.f, acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int32_t p0 = 0; p0 < total; p0 += kPartsPerWarp) {
    const int32_t p = p0 + lane;
    int64_t slot = -1;
    if (lane < kPartsPerWarp && p < total) slot = unit_part_slot(a, la, lb, u, p);
    float m = -INFINITY, l = 0.f;
    if (slot >= 0) {
      m = mlw[(slot * G + j) * 2];
      l = mlw[(slot * G + j) * 2 + 1];
    }
    float xs[kPartsPerWarp][V];
#pragma unroll
    for (int t = 0; t < kPartsPerWarp; ++t) {
      const int64_t st = __shfl_sync(0xffffffffu, slot, t);
#pragma unroll
      for (int e = 0; e < V; ++e) xs[t][e] = 0.f;
      if (st >= 0) {
        const float* src = accw + (st * G + j) * D + lane * V;
        if constexpr (V == 4) {
          const float4 v4 = *reinterpret_cast<const float4*>(src);
          xs[t][0] = v4.x;
          xs[t][1] = v4.y;
          xs[t][2] = v4.z;
          xs[t][3] = v4.w;
        } else {
          const float2 v2 = *reinterpret_cast<const float2*>(src);
          xs[t][0] = v2.x;
          xs[t][1] = v2.y;
        }
      }
    }
    float mx = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mx = fmaxf(mx, m_run);
    if (mx == -INFINITY) continue;
    const float f_run = fast_exp2(m_run - mx);
    const float w = fast_exp2(m - mx);  // 0 for an absent part
    float lw = w * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    l_run = l_run * f_run + lw;
    m_run = mx;
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] *= f_run;
#pragma unroll
    for (int t = 0; t < kPartsPerWarp; ++t) {
      const float wt = __shfl_sync(0xffffffffu, w, t);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += wt * xs[t][e];
    }
  }
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < V; ++e) v[e] = l_run > 0.f ? acc[e] / l_run : 0.f;
  TOut* out = static_cast<TOut*>(a.out) + ((int64_t)r * a.Hq + (int64_t)h * G + j) * D + lane * V;
  store_vec<TOut>(out, v, V);
}

cudaError_t launch_combine(const DecodeArgs& a, int32_t dtype, cudaStream_t stream) {
  const int64_t units = (int64_t)a.batch * a.Hkv;
  if (units > kDirectUnits && units >= a.ctas && a.G <= 8) {
    const dim3 grid((unsigned)units), block((unsigned)(a.G * 32));
    if (dtype == SRKV_BF16)
      return a.d == 128 ? launch_pdl(combine_unit_kernel<__nv_bfloat16, 128>, grid, block, 0, stream, a)
                        : launch_pdl(combine_unit_kernel<__nv_bfloat16, 64>, grid, block, 0, stream, a);
    return a.d == 128 ? launch_pdl(combine_unit_kernel<float, 128>, grid, block, 0, stream, a)
                      : launch_pdl(combine_unit_kernel<float, 64>, grid, block, 0, stream, a);
  }
  const int64_t heads = (int64_t)a.batch * a.Hkv * a.G;
  if (heads == 0) return cudaSuccess;
  if (heads > INT32_MAX) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)heads);
  if (dtype == SRKV_BF16)
    return a.d == 128 ? launch_pdl(combine_kernel<__nv_bfloat16, 128>, grid, dim3(kWarps * 32), 0, stream, a)
                      : launch_pdl(combine_kernel<__nv_bfloat16, 64>, grid, dim3(kWarps * 32), 0, stream, a);
  return a.d == 128 ? launch_pdl(combine_kernel<float, 128>, grid, dim3(kWarps * 32), 0, stream, a)
                    : launch_pdl(combine_kernel<float, 64>, grid, dim3(kWarps * 32), 0, stream, a);
}

}  // namespace srkv
