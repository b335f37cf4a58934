// decode_combine.cu -- merge of the split partials into the attention output.
//
// KV-cache survey "大模型推理百倍加速之KV cache篇", section "Share--KV cache共享": partial
// attention results over disjoint KV subsets are merged the Flash-Decoding way.  With
// partial i = (m_i, l_i, acc_i) in the log2 domain:
//   out = sum_i 2^(m_i - m*) acc_i / sum_i 2^(m_i - m*) l_i,   m* = max_i m_i.
// One thread per (request, q head, d).  The partials of a unit are those of the CTAs whose
// position range meets the unit's list (decode_plan.cuh); a thread merges them online,
// loading 16 partials' (m, l, acc) per round of independent loads, so the kernel costs a
// few memory latencies, not one per partial.  A unit with no positions (L = 0) gets a zero
// output.  Launched as a programmatic dependent of the split kernel: it waits for that grid
// before reading.
#include "decode_plan.cuh"

namespace srkv {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxG = 16;
constexpr int kChunk = 16;  // partials loaded per round

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
__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeArgs a) {
  griddep_wait();
  const int32_t U = a.batch * a.Hkv;
  const int32_t G = a.G, D = a.d;
  const int32_t GD = G * D;
  const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;  // (unit, head, d)
  if (idx >= (int64_t)U * GD) return;
  const int32_t u = (int32_t)(idx / GD);
  const int32_t je = (int32_t)(idx % GD);
  const int32_t j = je / D;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  const int32_t* unit_n = reinterpret_cast<const int32_t*>(a.ws + a.lay.unit_n);
  const int64_t* unit_off = reinterpret_cast<const int64_t*>(a.ws + a.lay.unit_off);
  TOut* out = static_cast<TOut*>(a.out) + ((int64_t)r * a.Hq + (int64_t)h * G) * D + je;

  const int64_t T = unit_off[U];
  const int64_t P = unit_off[u];
  const int32_t n = unit_n[u];
  const int64_t C = a.ctas;
  if (n <= 0 || T <= 0) {
    store_out<TOut>(out, 0.f);
    return;
  }
  const int64_t c_first = cta_of(P, T, C);
  const int32_t parts = (int32_t)(cta_of(P + n - 1, T, C) - c_first + 1);
  // With T >= C every CTA owns at least one position; otherwise skip empty ranges.
  const bool maybe_empty = T < C;
  const float* accp = reinterpret_cast<const float*>(a.ws + a.lay.acc) +
                      ((u + c_first) * G) * (int64_t)D + je;
  const float* mlp = reinterpret_cast<const float*>(a.ws + a.lay.ml) + (u + c_first) * G * 2 +
                     j * 2;
  // Online merge, kChunk partials per round of independent loads.
  float m_run = -INFINITY, l_run = 0.f, acc_run = 0.f;
  for (int32_t i0 = 0; i0 < parts; i0 += kChunk) {
    float m[kChunk], l[kChunk], x[kChunk];
#pragma unroll
    for (int32_t t = 0; t < kChunk; ++t) {
      const int32_t i = i0 + t;
      bool has = i < parts;
      if (has && maybe_empty)
        has = cta_begin(c_first + i, T, C) < cta_begin(c_first + i + 1, T, C);
      m[t] = has ? mlp[(int64_t)i * G * 2] : -INFINITY;
      l[t] = has ? mlp[(int64_t)i * G * 2 + 1] : 0.f;
      x[t] = has ? accp[(int64_t)i * GD] : 0.f;
    }
    float mx = m_run;
#pragma unroll
    for (int32_t t = 0; t < kChunk; ++t) mx = fmaxf(mx, m[t]);
    if (mx == -INFINITY) continue;
    const float f_run = exp2f(m_run - mx);
    l_run *= f_run;
    acc_run *= f_run;
#pragma unroll
    for (int32_t t = 0; t < kChunk; ++t) {
      const float f = exp2f(m[t] - mx);  // 0 for m = -inf
      l_run += f * l[t];
      acc_run += f * x[t];
    }
    m_run = mx;
  }
  store_out<TOut>(out, l_run > 0.f ? acc_run / l_run : 0.f);
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int32_t dtype, cudaStream_t stream) {
  const int64_t total = (int64_t)a.batch * a.Hkv * a.G * a.d;
  if (total == 0) return cudaSuccess;
  if (a.G > kMaxG) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((total + kThreads - 1) / kThreads));
  if (dtype == SRKV_BF16)
    return launch_pdl(combine_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, stream, a);
  return launch_pdl(combine_kernel<float>, grid, dim3(kThreads), 0, stream, a);
}

}  // namespace srkv
