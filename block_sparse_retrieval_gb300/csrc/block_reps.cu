// block_reps.cu -- representation vectors: the fp32 mean of each page's keys per kv head.
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Feature Description": at prefill, representation vectors are extracted block by block.
// The pages do not define the vector; it is the mean of the block's keys per kv head,
// over the tokens the page holds.
//
// Pure streaming: each CTA reads one contiguous (page, kv head) slab of S x d values with
// 16-byte loads, all issued before any is used, and writes d floats.  Bytes per unit:
// S*d*elem read + 4d written (bf16, d = 128: 32 KiB + 512 B).
#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kRepThreads = 256;

template <typename T>
struct Vec16;  // 16 bytes of T, widened to float
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void widen(const int4& v, float (&f)[8]) {
    const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_lo(w[i]);
      f[2 * i + 1] = bf16_hi(w[i]);
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void widen(const int4& v, float (&f)[4]) {
    f[0] = __int_as_float(v.x);
    f[1] = __int_as_float(v.y);
    f[2] = __int_as_float(v.z);
    f[3] = __int_as_float(v.w);
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(kRepThreads)
    block_reps_kernel(const T* __restrict__ k_cache, int64_t num_pages, int32_t Hkv,
                      const int32_t* __restrict__ page_ids,
                      const int32_t* __restrict__ valid, int32_t n, float* __restrict__ reps,
                      int32_t* error_flags) {
  constexpr int EPV = Vec16<T>::N;        // elements per 16-byte vector
  constexpr int VPR = D / EPV;            // vectors per row
  constexpr int RPP = kRepThreads / VPR;  // rows per pass
  constexpr int PASSES = kBlock / RPP;
  __shared__ float partial[RPP][D];

  const int32_t i = blockIdx.x / Hkv;
  const int32_t h = blockIdx.x % Hkv;
  if (i >= n) return;
  const int32_t page = page_ids[i];
  const int32_t v = valid[i];
  if (page < 0 || (int64_t)page >= num_pages || v < 0 || v > kBlock) {
    if (threadIdx.x == 0) raise_flags(error_flags, SRKV_EFLAG_PAGE_RANGE);
    return;
  }
  const int col = threadIdx.x % VPR;
  const int row0 = threadIdx.x / VPR;
  const int4* slab = reinterpret_cast<const int4*>(
      k_cache + ((int64_t)page * Hkv + h) * (int64_t)kBlock * D);

  int4 raw[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = row0 + p * RPP;
    raw[p] = row < v ? __ldg(slab + row * VPR + col) : make_int4(0, 0, 0, 0);
  }
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    float f[EPV];
    Vec16<T>::widen(raw[p], f);
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) partial[row0][col * EPV + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < RPP; ++r) s += partial[r][threadIdx.x];
    reps[((int64_t)page * Hkv + h) * D + threadIdx.x] = v > 0 ? s / (float)v : 0.f;
  }
}

template <typename T, int D>
cudaError_t launch(const void* k, int64_t P, int32_t Hkv, const int32_t* ids,
                   const int32_t* valid, int32_t n, float* reps, int32_t* flags,
                   cudaStream_t s) {
  const int64_t grid = (int64_t)n * Hkv;
  if (grid == 0) return cudaSuccess;
  block_reps_kernel<T, D><<<(unsigned)grid, kRepThreads, 0, s>>>(
      static_cast<const T*>(k), P, Hkv, ids, valid, n, reps, flags);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_reps(const srkv_config& cfg, const void* k_cache, int64_t num_pages,
                              const int32_t* page_ids, const int32_t* valid, int32_t n,
                              float* reps, int32_t* error_flags, cudaStream_t stream) {
  const int32_t Hkv = cfg.num_kv_heads;
  if (cfg.dtype == SRKV_BF16) {
    if (cfg.head_dim == 128)
      return launch<__nv_bfloat16, 128>(k_cache, num_pages, Hkv, page_ids, valid, n, reps,
                                        error_flags, stream);
    return launch<__nv_bfloat16, 64>(k_cache, num_pages, Hkv, page_ids, valid, n, reps,
                                     error_flags, stream);
  }
  if (cfg.head_dim == 128)
    return launch<float, 128>(k_cache, num_pages, Hkv, page_ids, valid, n, reps, error_flags,
                              stream);
  return launch<float, 64>(k_cache, num_pages, Hkv, page_ids, valid, n, reps, error_flags,
                           stream);
}

}  // namespace srkv
