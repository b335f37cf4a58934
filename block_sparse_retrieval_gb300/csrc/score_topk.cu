// score_topk.cu -- inner-product scoring of the offload blocks and top-k selection.
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Overall Solution": sparse retrieval computes the inner product of the current query
// with every representation vector and keeps the topK closest blocks; "Configuration
// Parameters": TOPK_PERCENT is the ratio kept, and a prompt shorter than DENSE_BOUNDARY is
// attended densely.  The KV-cache survey ("Share--KV cache共享") has a group of query heads
// share one K/V head: here a block's score for a kv head is the inner product with the sum
// of the group's queries, and selection is per (request, kv head).
//
// One CTA per (request, kv head) unit:
//   1. block-table entries of the candidates -> shared memory (one round of loads);
//   2. group query sum q_bar (fp32);
//   3. one warp per candidate: s_b = q_bar . rep (fp32, fixed lane order), turned into an
//      order-preserving 32-bit key (NaN and out-of-range pages rank lowest);
//   4. MSB-first radix select (4 passes of 8 bits) finds the k-th largest key exactly;
//   5. ties on that key go to the lower block index (an exclusive count in block order),
//      and a second count writes the kept blocks ascending.
// Bytes per unit: n * (4 + 4d) read (block table + reps), k * 4 written.
#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

struct ScoreArgs {
  const void* q;
  const float* reps;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* prompt_lens;
  int32_t* sel;
  int32_t kmax;
  int32_t* nsel;
  int32_t* error_flags;
  int32_t Hq, Hkv, G;
  int32_t init_tokens, local_tokens, dense_boundary;
  double topk_percent;
};

// k = min(n, ceil(p*n - 1e-9)) with separately rounded operations (no contraction), so
// that the host and the device agree on every n.
__device__ __forceinline__ int32_t device_topk_count(int32_t n, double p) {
  if (n <= 0) return 0;
  const double x = ceil(__dadd_rn(__dmul_rn(p, (double)n), -1e-9));
  if (!(x > 0.0)) return 0;
  if (x > (double)n) return n;
  return (int32_t)x;
}

__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;            // NaN ranks below everything
  if (s == 0.0f) s = 0.0f;          // -0 and +0 tie
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the CTA of one int per thread; returns the prefix, *total the sum.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* scratch,
                                                        int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) scratch[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int32_t before = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_topk_kernel(ScoreArgs a) {
  extern __shared__ uint32_t smem[];
  uint32_t* keys = smem;                                        // [max_blocks]
  int32_t* pages = reinterpret_cast<int32_t*>(smem + a.max_blocks);  // [max_blocks]
  __shared__ float qbar[D];
  __shared__ int32_t hist[256];
  __shared__ int32_t scratch[32];
  __shared__ int32_t digit_out, remaining_out;
  __shared__ uint32_t flags_out;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t u = blockIdx.x;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  if (tid == 0) flags_out = 0;

  int32_t L = a.seq_lens[r];
  const int32_t Lmax = a.max_blocks * kBlock;
  uint32_t eflags = 0;
  if (L < 0 || L > Lmax) {
    eflags |= SRKV_EFLAG_SEQ_LEN;
    L = L < 0 ? 0 : Lmax;
  }
  const int32_t prompt = a.prompt_lens ? a.prompt_lens[r] : L;
  const int32_t W = L - a.local_tokens;
  int32_t b_lo = 0, n = 0;
  if (W > a.init_tokens) {
    b_lo = a.init_tokens / kBlock;
    n = (W + kBlock - 1) / kBlock - b_lo;
  }
  const bool dense = prompt < a.dense_boundary;
  int32_t k = dense ? n : device_topk_count(n, a.topk_percent);
  if (k > a.kmax) {
    eflags |= SRKV_EFLAG_SELECTION;
    k = a.kmax;
  }
  int32_t* sel_u = a.sel + (int64_t)u * a.kmax;

  if (k == n && n <= a.kmax) {  // every candidate is kept: no scoring needed
    for (int32_t i = tid; i < n; i += kThreads) sel_u[i] = b_lo + i;
    if (tid == 0) {
      a.nsel[u] = n;
      raise_flags(a.error_flags, eflags);
    }
    return;
  }
  if (k == 0) {
    if (tid == 0) {
      a.nsel[u] = 0;
      raise_flags(a.error_flags, eflags);
    }
    return;
  }

  // 1. physical pages of the candidates.
  const int32_t* bt_r = a.block_table + (int64_t)r * a.max_blocks;
  for (int32_t i = tid; i < n; i += kThreads) pages[i] = bt_r[b_lo + i];
  // 2. group query sum.
  const T* q = static_cast<const T*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * D;
  for (int e = tid; e < D; e += kThreads) {
    float s = 0.f;
    for (int j = 0; j < a.G; ++j) s += static_cast<float>(q[(int64_t)j * D + e]);
    qbar[e] = s;
  }
  __syncthreads();

  // 3. scores, one warp per candidate, lanes over d.
  constexpr int EPL = D / 32;  // elements per lane: 4 (d 128) or 2 (d 64)
  float qv[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] = qbar[lane * EPL + e];
  constexpr int UNROLL = 8;
  for (int32_t i0 = warp; i0 < n; i0 += kWarps * UNROLL) {
    float part[UNROLL];
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {
      const int32_t i = i0 + x * kWarps;
      part[x] = 0.f;
      if (i < n) {
        const int32_t page = pages[i];
        if (page >= 0 && (int64_t)page < a.num_pages) {
          const float* rep = a.reps + ((int64_t)page * a.Hkv + h) * D + lane * EPL;
          if constexpr (EPL == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(rep));
            part[x] = qv[0] * v.x + qv[1] * v.y + qv[2] * v.z + qv[3] * v.w;
          } else {
            const float2 v = __ldg(reinterpret_cast<const float2*>(rep));
            part[x] = qv[0] * v.x + qv[1] * v.y;
          }
        }
      }
    }
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {
      float s = part[x];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const int32_t i = i0 + x * kWarps;
      if (lane == 0 && i < n) {
        const int32_t page = pages[i];
        if (page >= 0 && (int64_t)page < a.num_pages) {
          keys[i] = score_key(s);
        } else {
          keys[i] = 0u;
          atomicOr(&flags_out, SRKV_EFLAG_PAGE_RANGE);
        }
      }
    }
  }
  __syncthreads();

  // 4. radix select of the k-th largest key.
  uint32_t prefix = 0, pmask = 0;
  int32_t remaining = k;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int32_t i = tid; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      int32_t c[8], local = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hist[lane * 8 + b];
        local += c[b];
      }
      // suffix sums over lanes (higher digits first)
      int32_t suffix = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_down_sync(0xffffffffu, suffix, o);
        if (lane + o < 32) suffix += y;
      }
      int32_t above = suffix - local;  // keys whose digit lies in higher lanes
#pragma unroll
      for (int b = 7; b >= 0; --b) {
        if (above < remaining && above + c[b] >= remaining) {
          digit_out = lane * 8 + b;
          remaining_out = remaining - above;
        }
        above += c[b];
      }
    }
    __syncthreads();
    prefix |= (uint32_t)digit_out << shift;
    pmask |= 0xffu << shift;
    remaining = remaining_out;
    __syncthreads();
  }
  const uint32_t kth = prefix;
  const int32_t need_equal = remaining;  // keys equal to kth that are kept (lowest blocks)

  // 5. keep key > kth, and the first need_equal keys == kth in block order; write ascending.
  const int32_t chunk = (n + kThreads - 1) / kThreads;
  const int32_t c0 = min(n, tid * chunk), c1 = min(n, c0 + chunk);
  int32_t n_eq = 0;
  for (int32_t i = c0; i < c1; ++i) n_eq += keys[i] == kth;
  int32_t total;
  int32_t eq_rank = block_exclusive_scan(n_eq, scratch, &total);
  int32_t n_take = 0;
  for (int32_t i = c0; i < c1; ++i) {
    const uint32_t key = keys[i];
    bool take = key > kth;
    if (key == kth) take = eq_rank++ < need_equal;
    n_take += take;
  }
  int32_t pos = block_exclusive_scan(n_take, scratch, &total);
  eq_rank -= n_eq;
  for (int32_t i = c0; i < c1; ++i) {
    const uint32_t key = keys[i];
    bool take = key > kth;
    if (key == kth) take = eq_rank++ < need_equal;
    if (take) sel_u[pos++] = b_lo + i;
  }
  if (tid == 0) {
    a.nsel[u] = total;
    raise_flags(a.error_flags, eflags | flags_out);
  }
}

template <typename T, int D>
cudaError_t launch(const ScoreArgs& a, int32_t units, cudaStream_t s) {
  const size_t smem = sizeof(uint32_t) * 2 * (size_t)a.max_blocks;
  auto kernel = score_topk_kernel<T, D>;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kernel<<<units, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_topk(const srkv_config& cfg, const void* q, const float* reps,
                              int64_t num_pages, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* seq_lens,
                              const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                              int32_t kmax, int32_t* nsel, int32_t* error_flags,
                              cudaStream_t stream) {
  ScoreArgs a;
  a.q = q;
  a.reps = reps;
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.prompt_lens = prompt_lens;
  a.sel = sel;
  a.kmax = kmax;
  a.nsel = nsel;
  a.error_flags = error_flags;
  a.Hq = cfg.num_q_heads;
  a.Hkv = cfg.num_kv_heads;
  a.G = cfg.num_q_heads / cfg.num_kv_heads;
  a.init_tokens = cfg.init_tokens;
  a.local_tokens = cfg.local_tokens;
  a.dense_boundary = cfg.dense_boundary;
  a.topk_percent = cfg.topk_percent;
  const int32_t units = batch * cfg.num_kv_heads;
  if (units == 0) return cudaSuccess;
  if (cfg.dtype == SRKV_BF16)
    return cfg.head_dim == 128 ? launch<__nv_bfloat16, 128>(a, units, stream)
                               : launch<__nv_bfloat16, 64>(a, units, stream);
  return cfg.head_dim == 128 ? launch<float, 128>(a, units, stream)
                             : launch<float, 64>(a, units, stream);
}

}  // namespace srkv
