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
// A warp takes kRowsPerWarp consecutive rows of one (page, kv head) slab: d / 8 lanes per
// row, each with 8 consecutive bf16 values (16 bytes), so every load of the warp is
// contiguous and all of its rows' loads are in flight before the first is used.  The row's
// maximum is reduced over its lanes; each lane writes 8 codes (8 bytes) and the row's first
// lane the scale.  Bytes per row: 2d read + d + 4 written.
#include <cuda_fp8.h>

#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kQuantWarps = 8;
constexpr int kRowsPerWarp = 8;  // divides the 128 rows of a slab
static_assert(kBlock % kRowsPerWarp == 0, "a warp's rows lie in one slab");

template <int D>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_fp8_kernel(const __nv_bfloat16* k_src, const __nv_bfloat16* v_src,
                        int64_t num_pages, const int32_t* page_ids, int32_t n_pages, int32_t Hkv,
                        uint8_t* k8, uint8_t* v8, float* k_scale, float* v_scale,
                        int32_t* error_flags) {
  constexpr int LPR = D / 8;              // lanes per row (16 bytes of bf16 each)
  constexpr int RPL = 32 / LPR;           // rows per warp-wide load
  constexpr int LOADS = kRowsPerWarp / RPL;
  static_assert(LOADS * RPL == kRowsPerWarp, "whole loads per warp");
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)n_pages * Hkv * kBlock;
  const int64_t gw = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  const int64_t r0 = gw * kRowsPerWarp;  // the warp's first row over K then V
  if (r0 >= 2 * rows) return;
  const int which = r0 >= rows ? 1 : 0;  // 0: K, 1: V (rows never straddle: rows % 8 == 0)
  const int64_t rr = r0 - which * rows;
  const int64_t i = rr / (Hkv * kBlock), hr = rr % (Hkv * kBlock);
  const int32_t page = page_ids[i];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (lane == 0 && hr == 0 && which == 0) raise_flags(error_flags, SRKV_EFLAG_PAGE_RANGE);
    return;
  }
  const int64_t row0 = (int64_t)page * Hkv * kBlock + hr;  // the same rows in the destination
  const int sub = lane / LPR, col = (lane % LPR) * 8;        // row within a load, first value
  const __nv_bfloat16* src = (which ? v_src : k_src) + row0 * D;
  int4 w[LOADS];
#pragma unroll
  for (int l = 0; l < LOADS; ++l)
    w[l] = *reinterpret_cast<const int4*>(src + (int64_t)(l * RPL + sub) * D + col);
  uint8_t* dst8 = (which ? v8 : k8) + row0 * D;
  float* dscale = (which ? v_scale : k_scale) + row0;
#pragma unroll
  for (int l = 0; l < LOADS; ++l) {
    const uint32_t u[4] = {(uint32_t)w[l].x, (uint32_t)w[l].y, (uint32_t)w[l].z,
                           (uint32_t)w[l].w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_lo(u[e]);
      x[2 * e + 1] = bf16_hi(u[e]);
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)  // within the row's lanes
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[e], scale), __fdiv_rn(x[e + 1], scale)), __NV_SATFINITE,
          __NV_E4M3);
      packed[e / 4] |= (uint32_t)c << (8 * (e % 4));
    }
    const int row = l * RPL + sub;
    *reinterpret_cast<uint2*>(dst8 + (int64_t)row * D + col) = make_uint2(packed[0], packed[1]);
    if (lane % LPR == 0) dscale[row] = scale;
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const srkv_config& cfg, const void* k_src, const void* v_src,
                                int64_t num_pages, const int32_t* page_ids, int32_t n_pages,
                                void* k8, void* v8, float* k_scale, float* v_scale,
                                int32_t* error_flags, cudaStream_t stream) {
  const int64_t warps = 2 * (int64_t)n_pages * cfg.num_kv_heads * kBlock / kRowsPerWarp;
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
