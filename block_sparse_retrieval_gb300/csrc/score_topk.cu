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
//      pages rank lowest), stored into the leader CTA's shared memory and counted into its
//      histogram of the top 8 key bits through distributed shared memory; one cluster
//      barrier gathers them;
//   3. the leader runs an MSB-first radix select, 8 bits a pass (the first from that
//      histogram), until the bin holding the k-th largest key has at most 32 keys; one warp
//      then ranks that bin exactly (score, then lower block index).  If four passes are
//      needed the k-th key is known exactly and its equal keys go to the lowest blocks;
//   4. the kept blocks are written ascending: a kept key's slot is the number of kept keys
//      before it in block order, from ballot counts per warp.
// Bytes per unit: n * (4 + 4d) read (block table + reps), k * 4 written.
#include "select.cuh"

namespace srkv {
namespace {

constexpr int kThreads = 256;
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

// Grid: one cluster of `cluster_size()` CTAs per (request, kv head) unit.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 4) score_topk_kernel(ScoreArgs a) {
  extern __shared__ uint32_t smem[];
  uint32_t* keys = smem;                                             // [max_blocks], leader
  int32_t* pages = reinterpret_cast<int32_t*>(smem + a.max_blocks);  // [max_blocks]
  __shared__ float qbar[D];
  __shared__ int32_t hist[3][256];  // leader: radix histograms (pass 0 filled by the cluster)
  __shared__ FinishShared<kThreads> fin;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the decode may be scheduled now; it waits for this grid
  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int32_t u = blockIdx.x / csize;
  const int32_t r = u / a.Hkv, h = u % a.Hkv;
  for (int i = tid; i < 3 * 256; i += kThreads) (&hist[0][0])[i] = 0;
  cluster_arrive();  // the leader's histograms are zero before any CTA adds to them

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

  const int32_t prompt = a.prompt_lens ? prompt_in : L_in;
  const SelCount sc = selection_count(L_in, prompt, a.max_blocks, a.kmax, a.init_tokens,
                                      a.local_tokens, a.dense_boundary, a.topk_percent);
  const int32_t n = sc.n, k = sc.k;  // n <= nmax
  uint32_t eflags = sc.flags;
  int32_t* sel_u = a.sel + (int64_t)u * a.kmax;

  // Uniform over the cluster: every CTA takes the same branch (and none waits at the
  // cluster barrier it arrived at).
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

  // 2. scores of the share, one warp per candidate, into the leader's keys and histogram
  cluster_wait();
  eflags |= score_share<D, kWarps>(qbar, pages, s_lo, min(s_hi, n), a.reps, a.num_pages, a.Hkv,
                                   h, keys, &hist[0][0], nullptr, nullptr, warp, lane, [] {},
                                   [](uint32_t) {});
  if (lane == 0 && eflags) raise_flags(a.error_flags, eflags);
  cluster_sync();  // every key and the pass-0 histogram are in the leader
  if (crank != 0) return;

  // 3. radix select until the boundary bin is small enough for one warp to rank
  auto bar = [] { __syncthreads(); };
  const RadixState rs = radix_narrow<kThreads>(keys, n, k, hist, tid, bar);

  // 4. kept blocks written ascending
  if (n <= kFastRounds * kThreads) {
    const int32_t kept = finish_fast<kThreads>(keys, n, rs, fin, tid, bar,
                                               [&](int32_t pos, int32_t i) { sel_u[pos] = b_lo + i; });
    if (tid == 0) a.nsel[u] = kept;
    return;
  }
  const uint32_t prefix = rs.prefix, pmask = rs.pmask;
  const int32_t remaining = rs.remaining;
  const bool ranked = rs.ranked;
  int32_t* bnd_idx = fin.bnd_idx;

  // Longer candidate lists: one warp walks the keys, lane l taking [l c, l c + c).
  if (warp != 0) return;
  const int32_t chunk = (n + 31) / 32;
  const int32_t c0 = min(n, lane * chunk), c1 = min(n, c0 + chunk);
  int32_t in_bin = 0;
  for (int32_t i = c0; i < c1; ++i) in_bin += (keys[i] & pmask) == prefix;
  int32_t bin_total;
  const int32_t bin0 = warp_exclusive_scan(in_bin, lane, &bin_total);
  uint32_t take_mask = 0;  // ranked: bit t set = the bin's t-th key in block order is kept
  if (ranked) {            // bin_total <= 32
    int32_t t = bin0;
    for (int32_t i = c0; i < c1; ++i)
      if ((keys[i] & pmask) == prefix) bnd_idx[t++] = i;
    __syncwarp();
    const uint32_t key = lane < bin_total ? keys[bnd_idx[lane]] : 0u;
    int32_t rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
      rank += j < bin_total && (kj > key || (kj == key && j < lane));
    }
    take_mask = __ballot_sync(0xffffffffu, lane < bin_total && rank < remaining);
  }
  int32_t n_take = 0;
  {
    int32_t t = bin0;
    for (int32_t i = c0; i < c1; ++i) {
      const uint32_t hi = keys[i] & pmask;
      if (hi > prefix) {
        ++n_take;
      } else if (hi == prefix) {
        n_take += ranked ? (int32_t)((take_mask >> t) & 1u) : (t < remaining);
        ++t;
      }
    }
  }
  int32_t total;
  int32_t pos = warp_exclusive_scan(n_take, lane, &total);
  {
    int32_t t = bin0;
    for (int32_t i = c0; i < c1; ++i) {
      const uint32_t hi = keys[i] & pmask;
      bool take = hi > prefix;
      if (hi == prefix) {
        take = ranked ? ((take_mask >> t) & 1u) != 0 : t < remaining;
        ++t;
      }
      if (take) sel_u[pos++] = b_lo + i;
    }
  }
  if (lane == 0) a.nsel[u] = total;
}

template <typename T, int D>
cudaError_t launch(const ScoreArgs& a, int32_t units, int32_t cluster, cudaStream_t s) {
  size_t smem = sizeof(uint32_t) * 2 * (size_t)a.max_blocks;
  if (smem < (size_t)kScoreExclusiveSmem) smem = kScoreExclusiveSmem;
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // One CTA of a cluster per SM, so that every SM keeps room for a decode CTA.
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicySpread;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, kernel, a);
}

// Candidates of the longest request the block table allows.
int64_t max_candidates(const srkv_config& cfg, int32_t max_blocks) {
  const int64_t W = (int64_t)max_blocks * kBlock - cfg.local_tokens;
  return W > cfg.init_tokens ? (W + kBlock - 1) / kBlock - cfg.init_tokens / kBlock : 0;
}

// CTAs per unit: about 64 candidates each, at most 8 (a portable cluster).
int32_t cluster_for(int64_t nmax) {
  const int64_t c = (nmax + 63) / 64;
  return (int32_t)(c < 1 ? 1 : (c > 8 ? 8 : c));
}

// CTAs per unit for a batch of `units`: cluster_for, but when at least two CTAs per unit
// still fit in half of a 152-SM GPU, no more than that, so that the other half of the SMs
// streams the initial and window pages while the scoring runs (a scoring CTA keeps its SM
// to itself); each CTA then scores more candidates, in more rounds of loads.  Not for
// compressed (E4M3) pages: their consumers are bound by the code conversions rather than
// by bytes, so half of the SMs cannot take all of list A, and the scoring keeps its grid.
int32_t cluster_for_batch(int64_t nmax, int64_t units, bool compressed) {
  const int32_t c = cluster_for(nmax);
  const int64_t u = units > 0 ? units : 1;
  const int64_t fit = 76 / u;
  if (fit >= 2 && fit < c) return compressed ? c : (int32_t)fit;
  // larger batches: no more CTAs than one wave on 152 SMs needs (at least one per unit)
  if (fit < 2 && u * c > 152) return (int32_t)(152 / u > 1 ? 152 / u : 1);
  return c;
}

}  // namespace

int64_t score_topk_ctas(const srkv_config& cfg, int32_t max_blocks, int32_t batch,
                        bool compressed) {
  const int64_t units = (int64_t)batch * cfg.num_kv_heads;
  return units * cluster_for_batch(max_candidates(cfg, max_blocks), units, compressed);
}

cudaError_t launch_score_topk(const srkv_config& cfg, const void* q, const float* reps,
                              int64_t num_pages, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* seq_lens,
                              const int32_t* prompt_lens, int32_t batch, int32_t* sel,
                              int32_t kmax, int32_t* nsel, int32_t* error_flags,
                              cudaStream_t stream, bool compressed) {
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
  const int64_t nmax = max_candidates(cfg, max_blocks);
  if (nmax > INT32_MAX) return cudaErrorInvalidValue;
  a.nmax = (int32_t)nmax;
  const int32_t cluster = cluster_for_batch(nmax, units, compressed);
  if ((int64_t)units * cluster > INT32_MAX) return cudaErrorInvalidValue;
  if (cfg.dtype == SRKV_BF16)
    return cfg.head_dim == 128 ? launch<__nv_bfloat16, 128>(a, units, cluster, stream)
                               : launch<__nv_bfloat16, 64>(a, units, cluster, stream);
  return cfg.head_dim == 128 ? launch<float, 128>(a, units, cluster, stream)
                             : launch<float, 64>(a, units, cluster, stream);
}

}  // namespace srkv
