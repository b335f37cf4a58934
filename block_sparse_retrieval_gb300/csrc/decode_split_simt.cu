// decode_split_simt.cu -- split phase of sparse paged decode on CUDA cores.
//
// Same page lists, CTA ranges and partial format as the tensor-core kernel
// (decode_split_mma.cu), for the cases it does not cover: fp32 caches (whose 1e-5 output
// tolerance rules out bf16 tensor-core inputs) and groups of more than 8 query heads.
// Attention is softmax(q K^T / sqrt(d)) V over the attended rows of each page (ATB reuse
// article, §1.1), accumulated in fp32 with an online max in the log2 domain.
//
// CTA = 4 warps.  Warp 0 plans each list, thread 0 resolves its positions one by one; every
// warp takes rows w, w+4, ...
// of the page, a lane holds d/32 elements of q (every head of the group), K and V, and one
// warp reduction per head gives each logit.  At the end of a unit's segment the warps merge
// through shared memory and warp 0 writes the partial to slot unit + CTA.
#include "decode_plan.cuh"

namespace srkv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kGMax = 16;

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) split_simt_kernel(const DecodeArgs a) {
  constexpr int E = D / 32;  // elements per lane
  __shared__ ListRange s_rg;
  __shared__ PageTask s_task;
  __shared__ int32_t s_unit;
  __shared__ uint32_t s_flags;
  __shared__ float s_m[kWarps][kGMax], s_l[kWarps][kGMax];
  __shared__ float s_acc[kWarps][kGMax][D];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();  // then the combine may be scheduled: it reads the inputs before its wait
  griddep_launch_dependents();
  const int G = a.G;
  uint32_t eflags = 0;
  float q[kGMax][E], acc[kGMax][E], m[kGMax], l[kGMax];

  for (int list = kListA; list <= kListB; ++list) {
    if (warp == 0) {
      int64_t* offsets = blockIdx.x == 0
                             ? reinterpret_cast<int64_t*>(a.ws + (list == kListA ? a.lay.off_a
                                                                                 : a.lay.off_b))
                             : nullptr;
      const ListRange rg = warp_plan(a, list, blockIdx.x, list_ctas(a, list), offsets, nullptr,
                                     eflags);
      if (lane == 0) s_rg = rg;
    }
    __syncthreads();
    const ListRange rg = s_rg;
    const int64_t npos = rg.end - rg.begin;
    int32_t cu = rg.u0;
    int64_t cj = rg.begin - rg.base0;
    uint32_t dummy = 0;
    Geom cg;
    int32_t cn = 0;
    if (tid == 0 && npos > 0) {
      cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
      cn = list == kListA ? list_a_count(cg) : cg.ns;
    }
    for (int64_t it = 0; it < npos; ++it) {
      __syncthreads();  // previous position fully consumed
      if (tid == 0) {
        while (cj >= cn) {
          ++cu;
          cj = 0;
          cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
          cn = list == kListA ? list_a_count(cg) : cg.ns;
        }
        const int64_t p = rg.begin + it;
        s_unit = cu;
        s_flags = ((cj == 0 || p == rg.begin) ? 1u : 0u) |
                  ((cj == cn - 1 || p == rg.end - 1) ? 2u : 0u);
        const int32_t* bt_r = a.block_table + (int64_t)(cu / a.Hkv) * a.max_blocks;
        s_task = list == kListA
                     ? resolve_a(cg, (int32_t)cj, bt_r, a.num_pages, eflags)
                     : resolve_b(cg, (int32_t)cj, a.sel + (int64_t)cu * a.kmax, bt_r,
                                 a.num_pages, a.init_tokens, eflags);
        ++cj;
      }
      __syncthreads();
      const int32_t u = s_unit;
      const uint32_t flags = s_flags;
      const PageTask task = s_task;
      const int32_t r = u / a.Hkv, h = u % a.Hkv;

      if (flags & 1u) {  // new segment: queries of the group, fresh state
        const T* qp = static_cast<const T*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * G) * D;
#pragma unroll
        for (int j = 0; j < kGMax; ++j) {
          m[j] = -INFINITY;
          l[j] = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            acc[j][e] = 0.f;
            q[j][e] = j < G ? ld_elem<T>(qp + (int64_t)j * D + lane + 32 * e) : 0.f;
          }
        }
      }
      if (task.page >= 0) {
        const int64_t slab = ((int64_t)task.page * a.Hkv + h) * kBlock * D;
        const T* kp = static_cast<const T*>(a.k_cache) + slab;
        const T* vp = static_cast<const T*>(a.v_cache) + slab;
        for (int row = task.lo + warp; row < task.hi; row += kWarps) {
          if (!(row < task.ie || row >= task.ws)) continue;
          float kv[E];
#pragma unroll
          for (int e = 0; e < E; ++e) kv[e] = ld_elem<T>(kp + (int64_t)row * D + lane + 32 * e);
          float vv[E];
#pragma unroll
          for (int e = 0; e < E; ++e) vv[e] = ld_elem<T>(vp + (int64_t)row * D + lane + 32 * e);
#pragma unroll
          for (int j = 0; j < kGMax; ++j) {
            if (j >= G) break;
            float sc = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) sc += q[j][e] * kv[e];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
            sc *= a.scale_log2;
            const float mn = fmaxf(m[j], sc);
            const float alpha = exp2f(m[j] - mn);
            const float p = exp2f(sc - mn);
            m[j] = mn;
            l[j] = l[j] * alpha + p;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[j][e] = acc[j][e] * alpha + p * vv[e];
          }
        }
      }
      if (flags & 2u) {  // end of the unit's segment: merge the warps, write the partial
        if (lane == 0)
          for (int j = 0; j < G; ++j) {
            s_m[warp][j] = m[j];
            s_l[warp][j] = l[j];
          }
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int e = 0; e < E; ++e) s_acc[warp][j][lane + 32 * e] = acc[j][e];
        __syncthreads();
        const int64_t slot = (list == kListB ? (int64_t)a.lay.bank : 0) + u + blockIdx.x;
        float* accp = reinterpret_cast<float*>(a.ws + a.lay.acc) + slot * G * D;
        float* mlp = reinterpret_cast<float*>(a.ws + a.lay.ml) + slot * G * 2;
        for (int idx = tid; idx < G * D; idx += kThreads) {
          const int j = idx / D, e = idx % D;
          float mx = -INFINITY;
          for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, s_m[w][j]);
          const float base = mx == -INFINITY ? 0.f : mx;
          float num = 0.f, den = 0.f;
          for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(s_m[w][j] - base);
            num += f * s_acc[w][j][e];
            den += f * s_l[w][j];
          }
          accp[idx] = num;
          if (e == 0) {
            mlp[j * 2 + 0] = mx;
            mlp[j * 2 + 1] = den;
          }
        }
      }
    }
    __syncthreads();
  }
  eflags = __reduce_or_sync(0xffffffffu, eflags);
  if (lane == 0) raise_flags(a.error_flags, eflags);
}

template <typename T, int D>
cudaError_t launch(const DecodeArgs& a, cudaStream_t s) {
  return launch_pdl(split_simt_kernel<T, D>, dim3(a.ctas), dim3(kThreads), 0, s, a);
}

}  // namespace

int32_t simt_split_ctas(int32_t sm_count) { return sm_count * 4; }

cudaError_t launch_split_simt(const DecodeArgs& a, int32_t dtype, cudaStream_t stream) {
  if (a.G > kGMax) return cudaErrorInvalidValue;
  if (dtype == SRKV_BF16)
    return a.d == 128 ? launch<__nv_bfloat16, 128>(a, stream) : launch<__nv_bfloat16, 64>(a, stream);
  return a.d == 128 ? launch<float, 128>(a, stream) : launch<float, 64>(a, stream);
}

}  // namespace srkv
