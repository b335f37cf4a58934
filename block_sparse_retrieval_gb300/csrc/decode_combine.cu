// decode_combine.cu -- merge of the split partials into the attention output.
//
// KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV cache共享": partial
// attention results over disjoint KV subsets are merged the Flash-Decoding way.  With
// partial i = (m_i, l_i, acc_i) in the log2 domain:
//   out = sum_i 2^(m_i - m*) acc_i / sum_i 2^(m_i - m*) l_i,   m* = max_i m_i.
// One warp per (request, q head).  The partials of a unit are those of the CTAs whose
// position ranges meet the unit's two lists (decode_plan.cuh); the warp merges them online,
// 32 partials per round of independent loads (vector loads of d), so the kernel costs a few
// memory latencies, not one per partial, and spreads over as many SMs as there are heads.  A unit with no positions (L = 0) gets a zero
// output.  Launched as a programmatic dependent of the split kernel: it waits for that grid
// before reading.
#include "decode_plan.cuh"

namespace srkv {
namespace {


// Where the partials of unit u in one list are.
struct ListParts {
  int64_t T, c_first, slot0;
  int32_t parts;
};

__device__ __forceinline__ ListParts list_parts(const DecodeArgs& a, const int64_t* off,
                                                int64_t bank, int32_t u) {
  const int32_t U = a.batch * a.Hkv;
  ListParts lp;
  lp.T = off[U];
  const int64_t P = off[u], n = off[u + 1] - off[u];
  lp.c_first = 0;
  lp.parts = 0;
  if (n > 0 && lp.T > 0) {
    lp.c_first = cta_of(P, lp.T, a.ctas);
    lp.parts = (int32_t)(cta_of(P + n - 1, lp.T, a.ctas) - lp.c_first + 1);
  }
  lp.slot0 = bank + u + lp.c_first;
  return lp;
}

// Slot of part i of a list, or -1 when that CTA owns no position of the list.
__device__ __forceinline__ int64_t part_slot(const ListParts& lp, int32_t i, int64_t C) {
  if (lp.T < C) {  // only then can a CTA's range be empty
    const int64_t c = lp.c_first + i;
    if (cta_begin(c, lp.T, C) == cta_begin(c + 1, lp.T, C)) return -1;
  }
  return lp.slot0 + i;
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

// One warp per (unit, query head): lane l owns d elements [l*V, l*V + V) (V = d / 32), the
// partials' (m, l) pairs are spread over the lanes and their weights broadcast by shuffles.
template <typename TOut, int D>
__global__ void __launch_bounds__(32) combine_kernel(const DecodeArgs a) {
  constexpr int V = D / 32;  // 4 (d 128) or 2 (d 64)
  griddep_wait();
  const int lane = threadIdx.x;
  const int32_t G = a.G;
  const int32_t u = blockIdx.x / G, j = blockIdx.x % G;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  TOut* out = static_cast<TOut*>(a.out) + ((int64_t)r * a.Hq + (int64_t)h * G + j) * D + lane * V;
  const ListParts la = list_parts(a, reinterpret_cast<const int64_t*>(a.ws + a.lay.off_a), 0, u);
  const ListParts lb =
      list_parts(a, reinterpret_cast<const int64_t*>(a.ws + a.lay.off_b), a.lay.bank, u);
  const float* accw = reinterpret_cast<const float*>(a.ws + a.lay.acc);
  const float* mlw = reinterpret_cast<const float*>(a.ws + a.lay.ml);
  const int32_t total = la.parts + lb.parts;
  float m_run = -INFINITY, l_run = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int32_t p0 = 0; p0 < total; p0 += 32) {
    // (m, l) of parts p0 .. p0+31, one per lane; every slot is a valid address
    const int32_t p = p0 + lane;
    int64_t slot = -1;
    if (p < total) slot = p < la.parts ? part_slot(la, p, a.ctas) : part_slot(lb, p - la.parts, a.ctas);
    float m = -INFINITY, l = 0.f;
    if (slot >= 0) {
      m = mlw[(slot * G + j) * 2];
      l = mlw[(slot * G + j) * 2 + 1];
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
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] *= f_run;
    m_run = mx;
    // accumulators of the chunk's parts: all loads issued before any is used
    const int32_t cnt = total - p0 < 32 ? total - p0 : 32;
    const int64_t my_slot = slot >= 0 ? slot : 0;
    float xs[32][V];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int64_t st = __shfl_sync(0xffffffffu, my_slot, t);
      if (t < cnt) {
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
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float wt = __shfl_sync(0xffffffffu, w, t);
      if (t < cnt && wt != 0.f)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += wt * xs[t][e];
    }
  }
  float v[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = (e < V && l_run > 0.f) ? acc[e] / l_run : 0.f;
  store_vec<TOut>(out, v, V);
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int32_t dtype, cudaStream_t stream) {
  const int64_t warps = (int64_t)a.batch * a.Hkv * a.G;
  if (warps == 0) return cudaSuccess;
  if (warps > INT32_MAX) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)warps);
  if (dtype == SRKV_BF16)
    return a.d == 128 ? launch_pdl(combine_kernel<__nv_bfloat16, 128>, grid, dim3(32), 0, stream, a)
                      : launch_pdl(combine_kernel<__nv_bfloat16, 64>, grid, dim3(32), 0, stream, a);
  return a.d == 128 ? launch_pdl(combine_kernel<float, 128>, grid, dim3(32), 0, stream, a)
                    : launch_pdl(combine_kernel<float, 64>, grid, dim3(32), 0, stream, a);
}

}  // namespace srkv
