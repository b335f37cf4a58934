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
// One thread-block cluster (up to 8 CTAs) per (request, kv head) unit:
//   1. one round of independent loads: the sequence and prompt lengths, the block-table
//      entries of this CTA's fixed share of the longest possible candidate range, and the
//      group's queries (summed into q_bar, fp32);
//   2. one warp per candidate below the request's own count n: s_b = q_bar . rep (fp32,
//      fixed lane order), turned into an order-preserving 32-bit key (NaN and out-of-range
//      pages rank lowest) and stored into the leader CTA's shared memory through
//      distributed shared memory; one cluster barrier gathers them;
//   3. the leader runs an MSB-first radix select, 8 bits a pass, until the bin holding the
//      k-th largest key has at most 32 keys; one warp then ranks that bin exactly (score,
//      then lower block index).  If four passes are needed the k-th key is known exactly
//      and its equal keys go to the lowest block indices;
//   4. kept blocks are written ascending (one exclusive count in block order).
// Bytes per unit: n * (4 + 4d) read (block table + reps), k * 4 written.
#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kThreads = 256;  // a decode CTA (48K registers) still fits beside one
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDynamicSmem = 200 * 1024;  // keys + pages of up to 25600 blocks

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
  int32_t nmax;  // candidates of a request as long as the block table allows
  double topk_percent;
};

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

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Store to the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_u32(uint32_t* local, uint32_t rank, uint32_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Every warp finds the digit holding the remaining-th largest key from a 256-bin histogram.
__device__ __forceinline__ void find_digit(const int32_t* hist, int lane, int32_t remaining,
                                           int32_t* digit, int32_t* rem_out, int32_t* cnt_out) {
  int32_t c[8], local = 0;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    c[b] = hist[lane * 8 + b];
    local += c[b];
  }
  int32_t suffix = local;  // keys in this lane's bins and above
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_down_sync(0xffffffffu, suffix, o);
    if (lane + o < 32) suffix += y;
  }
  int32_t above = suffix - local, dg = -1, rm = 0, cn = 0;
#pragma unroll
  for (int b = 7; b >= 0; --b) {
    if (above < remaining && above + c[b] >= remaining) {
      dg = lane * 8 + b;
      rm = remaining - above;
      cn = c[b];
    }
    above += c[b];
  }
  const uint32_t who = __ballot_sync(0xffffffffu, dg >= 0);
  const int src = __ffs(who) - 1;
  *digit = __shfl_sync(0xffffffffu, dg, src);
  *rem_out = __shfl_sync(0xffffffffu, rm, src);
  *cnt_out = __shfl_sync(0xffffffffu, cn, src);
}

// Grid: one cluster of `cluster_size()` CTAs per (request, kv head) unit.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_topk_kernel(ScoreArgs a) {
  extern __shared__ uint32_t smem[];
  uint32_t* keys = smem;                                             // [max_blocks], leader
  int32_t* pages = reinterpret_cast<int32_t*>(smem + a.max_blocks);  // [max_blocks]
  __shared__ float qbar[D];
  __shared__ int32_t hist[3][256];
  __shared__ int32_t scratch[32];
  __shared__ int32_t bnd_idx[32];
  __shared__ int32_t bnd_cnt;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the decode may be scheduled now; it waits for this grid
  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int32_t u = blockIdx.x / csize;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;

  // 1. independent loads.  The share of block-table entries is fixed by the longest
  // candidate range the table allows (nmax), so it does not wait for the length.
  const int32_t L_in = a.seq_lens[r];
  const int32_t prompt_in = a.prompt_lens ? a.prompt_lens[r] : 0;
  const int32_t b_lo = a.init_tokens / kBlock;
  const int32_t s_lo = (int32_t)((int64_t)a.nmax * crank / csize);
  const int32_t s_hi = (int32_t)((int64_t)a.nmax * (crank + 1) / csize);
  const int32_t* bt_r = a.block_table + (int64_t)r * a.max_blocks + b_lo;
  for (int32_t i = s_lo + tid; i < s_hi; i += kThreads) pages[i - s_lo] = bt_r[i];
  const T* q = static_cast<const T*>(a.q) + ((int64_t)r * a.Hq + (int64_t)h * a.G) * D;
  for (int e = tid; e < D; e += kThreads) {
    float s = 0.f;
    int j = 0;
    for (; j + 4 <= a.G; j += 4) {  // four independent loads in flight
      const float x0 = static_cast<float>(q[(int64_t)(j + 0) * D + e]);
      const float x1 = static_cast<float>(q[(int64_t)(j + 1) * D + e]);
      const float x2 = static_cast<float>(q[(int64_t)(j + 2) * D + e]);
      const float x3 = static_cast<float>(q[(int64_t)(j + 3) * D + e]);
      s += x0;
      s += x1;
      s += x2;
      s += x3;
    }
    for (; j < a.G; ++j) s += static_cast<float>(q[(int64_t)j * D + e]);
    qbar[e] = s;
  }

  int32_t L = L_in;
  const int32_t prompt = a.prompt_lens ? prompt_in : L_in;
  const int32_t Lmax = a.max_blocks * kBlock;
  uint32_t eflags = 0;
  if (L < 0 || L > Lmax) {
    eflags |= SRKV_EFLAG_SEQ_LEN;
    L = L < 0 ? 0 : Lmax;
  }
  const int32_t W = L - a.local_tokens;
  const int32_t n = W > a.init_tokens ? (W + kBlock - 1) / kBlock - b_lo : 0;  // <= nmax
  const bool dense = prompt < a.dense_boundary;
  int32_t k = dense ? n : device_topk_count(n, a.topk_percent);
  if (k > a.kmax) {
    eflags |= SRKV_EFLAG_SELECTION;
    k = a.kmax;
  }
  int32_t* sel_u = a.sel + (int64_t)u * a.kmax;

  // Uniform over the cluster: every CTA takes the same branch.
  if ((k == n && n <= a.kmax) || k == 0) {  // all candidates, or none: no scoring
    if (crank == 0) {
      for (int32_t i = tid; i < k; i += kThreads) sel_u[i] = b_lo + i;
      if (tid == 0) {
        a.nsel[u] = k;
        raise_flags(a.error_flags, eflags);
      }
    }
    return;
  }
  __syncthreads();  // pages and qbar

  // 2. scores of the share, one warp per candidate; keys go to the leader's shared memory
  constexpr int EPL = D / 32;  // elements per lane: 4 (d 128) or 2 (d 64)
  float qv[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] = qbar[lane * EPL + e];
  const int32_t i_hi = min(s_hi, n);
  constexpr int UNROLL = 4;
  for (int32_t i0 = s_lo + warp; i0 < i_hi; i0 += kWarps * UNROLL) {
    float part[UNROLL];
    bool ok[UNROLL];
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {
      const int32_t i = i0 + x * kWarps;
      part[x] = 0.f;
      ok[x] = false;
      if (i < i_hi) {
        const int32_t page = pages[i - s_lo];
        ok[x] = page >= 0 && (int64_t)page < a.num_pages;
        if (ok[x]) {
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
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int x = 0; x < UNROLL; ++x) part[x] += __shfl_xor_sync(0xffffffffu, part[x], o);
#pragma unroll
    for (int x = 0; x < UNROLL; ++x) {
      const int32_t i = i0 + x * kWarps;
      if (lane == 0 && i < i_hi) {
        if (!ok[x]) eflags |= SRKV_EFLAG_PAGE_RANGE;
        st_cluster_u32(&keys[i], 0, ok[x] ? score_key(part[x]) : 0u);
      }
    }
  }
  if (lane == 0 && eflags) raise_flags(a.error_flags, eflags);
  cluster_sync();  // every key is in the leader's shared memory
  if (crank != 0) return;

  // 3. radix select (one barrier per pass, triple-buffered bins) until the boundary bin is
  // small enough for one warp to rank
  for (int i = tid; i < 2 * 256; i += kThreads) hist[i >> 8][i & 255] = 0;
  if (tid == 0) bnd_cnt = 0;
  __syncthreads();
  uint32_t prefix = 0, pmask = 0;
  int32_t remaining = k;
  bool ranked = false;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int32_t* hcur = hist[pass % 3];
    for (int i = tid; i < 256; i += kThreads) hist[(pass + 1) % 3][i] = 0;
    for (int32_t i0 = warp * 32; i0 < n; i0 += kThreads) {
      // Scores cluster in a few digits; lanes with equal digits add once (one leader).
      const int32_t i = i0 + lane;
      const uint32_t key = i < n ? keys[i] : 0u;
      const bool in = i < n && (key & pmask) == prefix;
      const uint32_t digit = in ? (key >> shift) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hcur[digit], __popc(peers));
    }
    __syncthreads();
    int32_t dg, rm, cnt;
    find_digit(hcur, lane, remaining, &dg, &rm, &cnt);
    prefix |= (uint32_t)dg << shift;
    pmask |= 0xffu << shift;
    remaining = rm;
    if (pass < 3 && cnt <= 32) {  // uniform: every warp read the same histogram
      ranked = true;
      break;
    }
  }
  int32_t* mark = pages;  // the leader's page share is no longer needed
  if (ranked) {
    // The <= 32 keys of the boundary bin, ranked by (key desc, block asc); the first
    // `remaining` of them are kept.
    for (int32_t i = tid; i < n; i += kThreads)
      if ((keys[i] & pmask) == prefix) bnd_idx[atomicAdd(&bnd_cnt, 1)] = i;
    __syncthreads();
    if (warp == 0) {
      const int32_t m = bnd_cnt;
      const int32_t idx = lane < m ? bnd_idx[lane] : INT32_MAX;
      const uint32_t key = lane < m ? keys[idx] : 0u;
      int32_t rank = 0;
      for (int32_t j = 0; j < m; ++j) {
        const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
        const int32_t ij = __shfl_sync(0xffffffffu, idx, j);
        rank += kj > key || (kj == key && ij < idx);
      }
      if (lane < m) mark[idx] = rank < remaining;
    }
    __syncthreads();
  }

  // 4. keep a key above the boundary bin; inside it, the ranked ones (or, after four
  // passes, the first `remaining` equal keys in block order).  Written ascending.
  const int32_t chunk = (n + kThreads - 1) / kThreads;
  const int32_t c0 = min(n, tid * chunk), c1 = min(n, c0 + chunk);
  int32_t total, eq_rank = 0, n_eq = 0;
  if (!ranked) {
    for (int32_t i = c0; i < c1; ++i) n_eq += keys[i] == prefix;
    eq_rank = block_exclusive_scan(n_eq, scratch, &total);
  }
  int32_t n_take = 0;
  for (int32_t i = c0; i < c1; ++i) {
    const uint32_t hi = keys[i] & pmask;
    n_take += hi > prefix || (hi == prefix && (ranked ? mark[i] != 0 : eq_rank++ < remaining));
  }
  int32_t pos = block_exclusive_scan(n_take, scratch, &total);
  eq_rank -= n_eq;
  for (int32_t i = c0; i < c1; ++i) {
    const uint32_t hi = keys[i] & pmask;
    if (hi > prefix || (hi == prefix && (ranked ? mark[i] != 0 : eq_rank++ < remaining)))
      sel_u[pos++] = b_lo + i;
  }
  if (tid == 0) a.nsel[u] = total;
}

template <typename T, int D>
cudaError_t launch(const ScoreArgs& a, int32_t units, int32_t cluster, cudaStream_t s) {
  const size_t smem = sizeof(uint32_t) * 2 * (size_t)a.max_blocks;
  auto kernel = score_topk_kernel<T, D>;
  // Once per device: the largest dynamic shared memory the host checks allow, and the full
  // shared-memory carveout, so that an SM running this kernel keeps room for a decode CTA
  // launched early behind it (programmatic launch).
  static bool configured[128] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxDynamicSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(units * cluster));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, a);
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
  // Candidates of the longest request the block table allows -> CTAs per unit (<= 8,
  // about 64 candidates each).
  int64_t W = (int64_t)max_blocks * kBlock - cfg.local_tokens;
  int64_t nmax = W > cfg.init_tokens ? (W + kBlock - 1) / kBlock - cfg.init_tokens / kBlock : 0;
  if (nmax > INT32_MAX) return cudaErrorInvalidValue;
  a.nmax = (int32_t)nmax;
  int32_t cluster = (int32_t)((nmax + 63) / 64);
  cluster = cluster < 1 ? 1 : (cluster > 8 ? 8 : cluster);
  if ((int64_t)units * cluster > INT32_MAX) return cudaErrorInvalidValue;
  if (cfg.dtype == SRKV_BF16)
    return cfg.head_dim == 128 ? launch<__nv_bfloat16, 128>(a, units, cluster, stream)
                               : launch<__nv_bfloat16, 64>(a, units, cluster, stream);
  return cfg.head_dim == 128 ? launch<float, 128>(a, units, cluster, stream)
                             : launch<float, 64>(a, units, cluster, stream);
}

}  // namespace srkv
