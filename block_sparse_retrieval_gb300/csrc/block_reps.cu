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
//
// At decode the same mean keeps the store current: appending a token rewrites one row of its
// page and recomputes that page's vector with the same code, so it equals a fresh build.
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

// Mean of the first v rows of one contiguous (page, kv head) slab, written to out[0, D):
// every 16-byte load issued before any is used, fixed-order sums (per thread over rows,
// then over the thread rows in shared memory).  kFresh: the slab was written by this CTA
// (plain coherent loads instead of the read-only path).
template <typename T, int D, bool kFresh>
__device__ __forceinline__ void slab_mean(const T* slab_p, int32_t v, float* out,
                                          float (*partial)[D]) {
  constexpr int EPV = Vec16<T>::N;        // elements per 16-byte vector
  constexpr int VPR = D / EPV;            // vectors per row
  constexpr int RPP = kRepThreads / VPR;  // rows per pass
  constexpr int PASSES = kBlock / RPP;
  const int col = threadIdx.x % VPR;
  const int row0 = threadIdx.x / VPR;
  const int4* slab = reinterpret_cast<const int4*>(slab_p);
  int4 raw[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = row0 + p * RPP;
    raw[p] = row < v ? (kFresh ? slab[row * VPR + col] : __ldg(slab + row * VPR + col))
                     : make_int4(0, 0, 0, 0);
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
    out[threadIdx.x] = v > 0 ? s / (float)v : 0.f;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kRepThreads)
    block_reps_kernel(const T* __restrict__ k_cache, int64_t num_pages, int32_t Hkv,
                      const int32_t* __restrict__ page_ids,
                      const int32_t* __restrict__ valid, int32_t n, float* __restrict__ reps,
                      int32_t* error_flags) {
  constexpr int RPP = kRepThreads / (D / Vec16<T>::N);
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
  const int64_t slab = ((int64_t)page * Hkv + h) * (int64_t)kBlock * D;
  slab_mean<T, D, false>(k_cache + slab, v, reps + ((int64_t)page * Hkv + h) * D, partial);
}

// Decode-time maintenance: CTA (request r, kv head h) writes the new token's key and value
// at position L = seq_lens[r] (page block_table[r][L / 128], row L % 128) and recomputes the
// page's representation vector over its rows [0, L % 128].
template <typename T, int D>
__global__ void __launch_bounds__(kRepThreads)
    append_kv_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* k_cache,
                     T* v_cache, int64_t num_pages, const int32_t* __restrict__ block_table,
                     int32_t max_blocks, const int32_t* __restrict__ seq_lens, int32_t Hkv,
                     float* __restrict__ reps, int32_t* error_flags) {
  constexpr int VPR = D / Vec16<T>::N;
  constexpr int RPP = kRepThreads / VPR;
  __shared__ float partial[RPP][D];
  const int32_t r = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
  const int32_t L = seq_lens[r];
  if (L < 0 || (int64_t)L >= (int64_t)max_blocks * kBlock) {
    if (threadIdx.x == 0) raise_flags(error_flags, SRKV_EFLAG_SEQ_LEN);
    return;
  }
  const int32_t page = block_table[(int64_t)r * max_blocks + L / kBlock];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (threadIdx.x == 0) raise_flags(error_flags, SRKV_EFLAG_PAGE_RANGE);
    return;
  }
  const int32_t row = L % kBlock;
  const int64_t slab = ((int64_t)page * Hkv + h) * (int64_t)kBlock * D;
  const int64_t src = ((int64_t)r * Hkv + h) * D;
  if (threadIdx.x < VPR) {
    reinterpret_cast<int4*>(k_cache + slab + (int64_t)row * D)[threadIdx.x] =
        reinterpret_cast<const int4*>(k_new + src)[threadIdx.x];
    reinterpret_cast<int4*>(v_cache + slab + (int64_t)row * D)[threadIdx.x] =
        reinterpret_cast<const int4*>(v_new + src)[threadIdx.x];
  }
  __syncthreads();  // the new row is visible to the CTA's own (coherent) loads
  slab_mean<T, D, true>(k_cache + slab, row + 1, reps + ((int64_t)page * Hkv + h) * D, partial);
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

template <typename T, int D>
cudaError_t launch_append(const void* kn, const void* vn, void* k, void* v, int64_t P,
                          const int32_t* bt, int32_t max_blocks, const int32_t* seq_lens,
                          int32_t batch, int32_t Hkv, float* reps, int32_t* flags,
                          cudaStream_t s) {
  const int64_t grid = (int64_t)batch * Hkv;
  if (grid == 0) return cudaSuccess;
  append_kv_kernel<T, D><<<(unsigned)grid, kRepThreads, 0, s>>>(
      static_cast<const T*>(kn), static_cast<const T*>(vn), static_cast<T*>(k),
      static_cast<T*>(v), P, bt, max_blocks, seq_lens, Hkv, reps, flags);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_kv(const srkv_config& cfg, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, int64_t num_pages,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t batch, float* reps,
                             int32_t* error_flags, cudaStream_t stream) {
  const int32_t Hkv = cfg.num_kv_heads;
  if (cfg.dtype == SRKV_BF16) {
    if (cfg.head_dim == 128)
      return launch_append<__nv_bfloat16, 128>(k_new, v_new, k_cache, v_cache, num_pages,
                                               block_table, max_blocks, seq_lens, batch, Hkv,
                                               reps, error_flags, stream);
    return launch_append<__nv_bfloat16, 64>(k_new, v_new, k_cache, v_cache, num_pages,
                                            block_table, max_blocks, seq_lens, batch, Hkv, reps,
                                            error_flags, stream);
  }
  if (cfg.head_dim == 128)
    return launch_append<float, 128>(k_new, v_new, k_cache, v_cache, num_pages, block_table,
                                     max_blocks, seq_lens, batch, Hkv, reps, error_flags,
                                     stream);
  return launch_append<float, 64>(k_new, v_new, k_cache, v_cache, num_pages, block_table,
                                  max_blocks, seq_lens, batch, Hkv, reps, error_flags, stream);
}

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
