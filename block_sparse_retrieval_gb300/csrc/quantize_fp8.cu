// quantize_fp8.cu -- compressed K/V pages: E4M3 codes with one fp32 scale per row.
//
// KV-cache survey "大模型推理百倍加速之KV cache篇" lists quantisation of the cache among the
// ways to shrink it; the format here is the 8-bit floating point E4M3 of the OCP 8-bit
// floating point specification (largest finite value 448).  One (page, kv head, token) row
// of d values x gets scale = max|x| / 448 (1 for an all-zero row) and codes
// E4M3(x / scale): the quotient in fp32, then rounded to the nearest E4M3 value, ties to
// even, saturating at +-448.  The scale makes the row's largest magnitude land on 448, so
// the codes use the format's whole range; per row (not per page) so that a token appended
// later needs no re-quantisation of its page.
//
// One warp per row: each lane loads d / 32 consecutive bf16 values (8 bytes for d = 128),
// the warp reduces the maximum, and each lane writes its codes (4 bytes) and lane 0 the
// scale.  Bytes per row: 2d read + d + 4 written.
#include <cuda_fp8.h>

#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kQuantWarps = 8;

template <int D>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_fp8_kernel(const __nv_bfloat16* k_src, const __nv_bfloat16* v_src,
                        int64_t num_pages, const int32_t* page_ids, int32_t n_pages, int32_t Hkv,
                        uint8_t* k8, uint8_t* v8, float* k_scale, float* v_scale,
                        int32_t* error_flags) {
  constexpr int V = D / 32;  // values per lane
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)n_pages * Hkv * kBlock;
  const int64_t gw = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (gw >= 2 * rows) return;
  const int which = gw >= rows ? 1 : 0;  // 0: K, 1: V
  const int64_t rr = gw - which * rows;
  const int64_t i = rr / (Hkv * kBlock), hr = rr % (Hkv * kBlock);
  const int32_t page = page_ids[i];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (lane == 0 && hr == 0 && which == 0) raise_flags(error_flags, SRKV_EFLAG_PAGE_RANGE);
    return;
  }
  const int64_t row = (int64_t)page * Hkv * kBlock + hr;  // the same row in the destination
  const __nv_bfloat16* src = (which ? v_src : k_src) + row * D + lane * V;
  float x[V];
  if constexpr (V == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    x[0] = bf16_lo(w.x);
    x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y);
    x[3] = bf16_hi(w.y);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    x[0] = bf16_lo(w);
    x[1] = bf16_hi(w);
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < V; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < V; ++e) {
    const __nv_fp8_storage_t c =
        __nv_cvt_float_to_fp8(__fdiv_rn(x[e], scale), __NV_SATFINITE, __NV_E4M3);
    packed |= (uint32_t)c << (8 * e);
  }
  uint8_t* dst = (which ? v8 : k8) + row * D + lane * V;
  if constexpr (V == 4)
    *reinterpret_cast<uint32_t*>(dst) = packed;
  else
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
  if (lane == 0) (which ? v_scale : k_scale)[row] = scale;
}

}  // namespace

cudaError_t launch_quantize_fp8(const srkv_config& cfg, const void* k_src, const void* v_src,
                                int64_t num_pages, const int32_t* page_ids, int32_t n_pages,
                                void* k8, void* v8, float* k_scale, float* v_scale,
                                int32_t* error_flags, cudaStream_t stream) {
  const int64_t warps = 2 * (int64_t)n_pages * cfg.num_kv_heads * kBlock;
  const int64_t grid = (warps + kQuantWarps - 1) / kQuantWarps;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  const auto* ks = static_cast<const __nv_bfloat16*>(k_src);
  const auto* vs = static_cast<const __nv_bfloat16*>(v_src);
  auto* kd = static_cast<uint8_t*>(k8);
  auto* vd = static_cast<uint8_t*>(v8);
  if (cfg.head_dim == 128)
    quantize_fp8_kernel<128><<<(unsigned)grid, kQuantWarps * 32, 0, stream>>>(
        ks, vs, num_pages, page_ids, n_pages, cfg.num_kv_heads, kd, vd, k_scale, v_scale,
        error_flags);
  else
    quantize_fp8_kernel<64><<<(unsigned)grid, kQuantWarps * 32, 0, stream>>>(
        ks, vs, num_pages, page_ids, n_pages, cfg.num_kv_heads, kd, vd, k_scale, v_scale,
        error_flags);
  return cudaGetLastError();
}

}  // namespace srkv
