// decode_combine.cu -- merge of the split partials into the attention output.
//
// KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV cache共享": partial
// attention results over disjoint KV subsets are merged the Flash-Decoding way.  With
// partial i = (m_i, l_i, acc_i) in the log2 domain:
//   out = sum_i 2^(m_i - m*) acc_i / sum_i 2^(m_i - m*) l_i,   m* = max_i m_i.
// One CTA per (request, kv head) unit, one thread per head-dim element; the partials of a
// unit are those of the CTAs whose position range meets the unit's list (decode_plan.cuh).
// A unit with no positions (L = 0) gets a zero output.
#include "decode_plan.cuh"

namespace srkv {
namespace {

template <typename TOut>
__device__ __forceinline__ void store_out(TOut* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename TOut>
__global__ void combine_kernel(const DecodeArgs a) {
  const int32_t U = a.batch * a.Hkv;
  const int32_t u = blockIdx.x;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  const int32_t* unit_n = reinterpret_cast<const int32_t*>(a.ws + a.lay.unit_n);
  const int64_t* unit_off = reinterpret_cast<const int64_t*>(a.ws + a.lay.unit_off);
  const float* accw = reinterpret_cast<const float*>(a.ws + a.lay.acc);
  const float* mlw = reinterpret_cast<const float*>(a.ws + a.lay.ml);
  TOut* out = static_cast<TOut*>(a.out) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * a.d;

  const int64_t T = unit_off[U];
  const int64_t P = unit_off[u];
  const int32_t n = unit_n[u];
  const int64_t C = a.ctas;
  int64_t c_first = 0, c_last = -1;
  if (n > 0 && T > 0) {
    c_first = cta_of(P, T, C);
    c_last = cta_of(P + n - 1, T, C);
  }
  for (int32_t e = threadIdx.x; e < a.d; e += blockDim.x) {
    for (int32_t j = 0; j < a.G; ++j) {
      float mx = -INFINITY;
      for (int64_t c = c_first; c <= c_last; ++c) {
        if (cta_begin(c, T, C) == cta_begin(c + 1, T, C)) continue;  // empty range
        mx = fmaxf(mx, mlw[((u + c) * a.G + j) * 2]);
      }
      const float base = mx == -INFINITY ? 0.f : mx;
      float num = 0.f, den = 0.f;
      for (int64_t c = c_first; c <= c_last; ++c) {
        if (cta_begin(c, T, C) == cta_begin(c + 1, T, C)) continue;
        const int64_t slot = u + c;
        const float f = exp2f(mlw[(slot * a.G + j) * 2] - base);
        den += f * mlw[(slot * a.G + j) * 2 + 1];
        num += f * accw[(slot * a.G + j) * a.d + e];
      }
      store_out<TOut>(out + (int64_t)j * a.d + e, den > 0.f ? num / den : 0.f);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int32_t dtype, cudaStream_t stream) {
  const int32_t U = a.batch * a.Hkv;
  if (U == 0) return cudaSuccess;
  if (dtype == SRKV_BF16)
    combine_kernel<__nv_bfloat16><<<U, a.d, 0, stream>>>(a);
  else
    combine_kernel<float><<<U, a.d, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace srkv
