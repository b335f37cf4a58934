// block_reps.cu -- representation vectors: the fp32 mean of each page's keys per kv head.
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Feature Description": at prefill, representation vectors are extracted block by block.
// The pages do not define the vector; it is the mean of the block's keys per kv head,
// over the tokens the page holds.
//
// Pure streaming: every (page, kv head) slab of S x d keys is contiguous, so one bulk copy
// (the TMA engine, 1-D) moves it into shared memory.  A persistent grid of one CTA per SM
// walks the slabs with a ring of stages in flight: a producer warp resolves 32 slabs' page
// ids at once and keeps every free stage filled, while 8 consumer warps reduce the slab in
// the oldest full stage.  Bytes per unit: S*d*elem read + 4d written (bf16, d = 128: 32 KiB
// + 512 B).
//
// The reduction has one fixed order, shared with the decode-time maintenance below so that
// both give the same bits: warp w sums its 16 rows [16w, 16w + 16) per 16-byte column chunk
// (a lane over the rows of its chunk, then warp shuffles across the lanes that hold the same
// chunk), and the 8 warp sums of a column are added in warp order.
//
// At decode the same mean keeps the store current: appending a token rewrites one row of its
// page and recomputes that page's vector with the same arithmetic, so it equals a fresh build.
#include "srkv_internal.cuh"

namespace srkv {
namespace {

constexpr int kRepWarps = 8;                    // consumer warps (and the append kernel's)
constexpr int kRepThreads = kRepWarps * 32;     // the append kernel's block
constexpr int kRepKernelThreads = kRepThreads + 32;  // + the producer warp
constexpr int kRepRingBytes = 192 * 1024;

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

// Geometry of one slab's reduction.
template <typename T, int D>
struct RepGeom {
  static constexpr int EPV = Vec16<T>::N;                  // elements per 16-byte chunk
  static constexpr int LPR = D / EPV;                      // chunks (lanes) per row
  static constexpr int RPI = 32 / LPR;                     // rows per warp-wide load
  static constexpr int RPW = kBlock / kRepWarps;           // rows per warp
  static constexpr int IPW = RPW / RPI;                    // loads per lane per slab
  static constexpr int CPW = D / kRepWarps;                // columns each warp finishes
  static constexpr int kSlab = kBlock * D * (int)sizeof(T);
  static constexpr int kStages = kRepRingBytes / kSlab;
  static_assert(LPR <= 32 && RPW % RPI == 0 && CPW <= 32, "slab geometry");
  // shared memory of the streaming kernel
  static constexpr size_t kOffPart = (size_t)kStages * kSlab;           // [stage][warp][D]
  static constexpr size_t kOffInfo = kOffPart + sizeof(float) * kStages * kRepWarps * D;
  static constexpr size_t kOffBar = kOffInfo + sizeof(int4) * kStages;  // full, ready, empty
  static constexpr size_t kSmem = kOffBar + sizeof(uint64_t) * 3 * kStages;
  static constexpr size_t kSmemAlloc = kSmem + 128;  // the ring starts 128-byte aligned
  static_assert(kSmemAlloc <= 232448, "shared memory opt-in limit");
};

// Warp `warp`'s sum over its rows r < v of the lane's column chunk: on return, lanes
// [0, LPR) hold the sums of columns [lane * EPV, lane * EPV + EPV) (the other lanes hold
// copies).  load(row, chunk) gives the 16 bytes of that chunk of that row.
template <typename T, int D, typename Load>
__device__ __forceinline__ void warp_column_sums(Load&& load, int warp, int lane, int32_t v,
                                                 float (&acc)[RepGeom<T, D>::EPV]) {
  using R = RepGeom<T, D>;
  const int chunk = lane % R::LPR, sub = lane / R::LPR;
  int4 raw[R::IPW];
#pragma unroll
  for (int i = 0; i < R::IPW; ++i) {
    const int row = warp * R::RPW + sub + i * R::RPI;
    raw[i] = row < v ? load(row, chunk) : make_int4(0, 0, 0, 0);
  }
#pragma unroll
  for (int e = 0; e < R::EPV; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < R::IPW; ++i) {
    float f[R::EPV];
    Vec16<T>::widen(raw[i], f);
#pragma unroll
    for (int e = 0; e < R::EPV; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int o = R::LPR; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < R::EPV; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
}

// part[w][c] = warp w's column sums; lanes [0, CPW) of warp `warp` finish columns
// [warp * CPW, warp * CPW + CPW): the 8 warp sums in warp order, divided by v.
template <typename T, int D>
__device__ __forceinline__ void finish_columns(const float* part, int warp, int lane, int32_t v,
                                               float* out) {
  using R = RepGeom<T, D>;
  if (lane < R::CPW) {
    const int c = warp * R::CPW + lane;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kRepWarps; ++w) s += part[w * D + c];
    out[c] = v > 0 ? s / (float)v : 0.f;
  }
}

template <typename T, int D>
__device__ __forceinline__ void store_column_sums(float* part, int warp, int lane,
                                                  const float (&acc)[RepGeom<T, D>::EPV]) {
  using R = RepGeom<T, D>;
  if (lane < R::LPR) {
#pragma unroll
    for (int e = 0; e < R::EPV; ++e) part[warp * D + lane * R::EPV + e] = acc[e];
  }
}

// What a stage holds: x, y = the slab index page * Hkv + h (its low 31 bits, the rest),
// z = the valid rows, w = -1 for the sentinel.
__device__ __forceinline__ int4 rep_stage(int64_t slab, int32_t v) {
  return make_int4((int32_t)(slab & 0x7fffffff), (int32_t)(slab >> 31), v, 0);
}

// Grid: persistent, at most one CTA per SM; CTA c takes units c, c + gridDim.x, ... where
// unit j is (listed page j / Hkv, kv head j % Hkv).  Warp 8 produces, warps 0..7 consume.
template <typename T, int D>
__global__ void __launch_bounds__(kRepKernelThreads, 1)
    block_reps_kernel(const T* __restrict__ k_cache, int64_t num_pages, int32_t Hkv,
                      const int32_t* __restrict__ page_ids,
                      const int32_t* __restrict__ valid, int32_t n, float* __restrict__ reps,
                      int32_t* error_flags) {
  using R = RepGeom<T, D>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  float* part = reinterpret_cast<float*>(smem + R::kOffPart);
  int4* info = reinterpret_cast<int4*>(smem + R::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + R::kOffBar);
  uint64_t* ready = full + R::kStages;   // the stage's 8 warp sums are in `part`
  uint64_t* empty = ready + R::kStages;  // the stage (slab and sums) may be refilled
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < R::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], kRepWarps);
      mbar_init(&empty[s], kRepWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // Launched behind the previous kernel of the stream (programmatic launch): the set-up above
  // touches shared memory only; the inputs may be that kernel's outputs.
  griddep_wait();
  griddep_launch_dependents();
  const int64_t units = (int64_t)n * Hkv;

  if (warp == kRepWarps) {
    // ---------------------------------------------------------------- producer
    uint32_t eflags = 0;
    bool abort = false;
    int64_t it = 0;
    const uint64_t once = l2_policy_evict_first();  // keys are read once here
    for (int64_t j0 = blockIdx.x; j0 < units && !abort; j0 += 32 * (int64_t)gridDim.x) {
      // lane l resolves unit j0 + l * gridDim.x
      const int64_t j = j0 + (int64_t)lane * gridDim.x;
      int64_t slab = -1;
      int32_t v = 0;
      if (j < units) {
        const int32_t i = (int32_t)(j / Hkv), h = (int32_t)(j % Hkv);
        const int32_t page = page_ids[i];
        v = valid[i];
        if (page < 0 || (int64_t)page >= num_pages || v < 0 || v > kBlock)
          eflags |= SRKV_EFLAG_PAGE_RANGE;
        else
          slab = (int64_t)page * Hkv + h;
      }
      const uint32_t todo = __ballot_sync(0xffffffffu, slab >= 0);
      // hand the valid units out in lane order (every lane takes part in the shuffles)
      for (uint32_t m = todo; m && !abort; m &= m - 1) {
        const int l = __ffs(m) - 1;
        const int64_t sl = __shfl_sync(0xffffffffu, slab, l);
        const int32_t vl = __shfl_sync(0xffffffffu, v, l);
        if (lane == 0) {
          const int s = (int)(it % R::kStages);
          if (it >= R::kStages && !mbar_wait(&empty[s], (uint32_t)((it / R::kStages - 1) & 1))) {
            abort = true;
            eflags |= SRKV_EFLAG_TIMEOUT;
          } else {
            info[s] = rep_stage(sl, vl);
            if (vl > 0) {
              mbar_arrive_expect_tx(&full[s], (uint32_t)R::kSlab);
              bulk_load_hint(smem + (size_t)s * R::kSlab, k_cache + sl * (int64_t)kBlock * D,
                             (uint32_t)R::kSlab, &full[s], once);
            } else {
              mbar_arrive(&full[s]);  // nothing to copy: the vector is zero
            }
          }
        }
        abort = __shfl_sync(0xffffffffu, abort, 0);
        if (abort) break;  // the stage was not armed
        ++it;
      }
    }
    if (lane == 0) {
      // the sentinel ends the consumers' loop (unless the ring is stuck)
      const int s = (int)(it % R::kStages);
      if (!abort &&
          (it < R::kStages || mbar_wait(&empty[s], (uint32_t)((it / R::kStages - 1) & 1)))) {
        info[s] = make_int4(0, 0, 0, -1);
        mbar_arrive(&full[s]);
        ++it;  // the drain below then skips this stage's earlier use, whose phase has passed
      } else if (!abort) {
        eflags |= SRKV_EFLAG_TIMEOUT;
      }
      // every copy lands before the CTA exits (also on the abort path): the last kStages
      // stages handed out are the latest use of each stage, so their phases are the ones to
      // wait for
      const int64_t first = it > R::kStages ? it - R::kStages : 0;
      for (int64_t i = first; i < it; ++i)
        if (!mbar_wait(&full[i % R::kStages], (uint32_t)((i / R::kStages) & 1))) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          break;
        }
    }
    eflags = __reduce_or_sync(0xffffffffu, eflags);
    if (lane == 0) raise_flags(error_flags, eflags);
    return;
  }

  // ------------------------------------------------------------------ consumers
  for (int64_t it = 0;; ++it) {
    const int s = (int)(it % R::kStages);
    const uint32_t ph = (uint32_t)((it / R::kStages) & 1);
    if (!mbar_wait(&full[s], ph)) {
      if (lane == 0) raise_flags(error_flags, SRKV_EFLAG_TIMEOUT);
      break;
    }
    const int4 inf = info[s];
    if (inf.w < 0) break;  // the sentinel
    const int64_t slab = (int64_t)(uint32_t)inf.x | ((int64_t)inf.y << 31);
    const int32_t v = inf.z;
    const unsigned char* st = smem + (size_t)s * R::kSlab;
    float acc[R::EPV];
    warp_column_sums<T, D>(
        [&](int row, int chunk) {
          return lds128(st + (size_t)row * (D * sizeof(T)) + (size_t)chunk * 16);
        },
        warp, lane, v, acc);
    float* ps = part + (size_t)s * kRepWarps * D;
    store_column_sums<T, D>(ps, warp, lane, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&ready[s]);
    if (!mbar_wait(&ready[s], ph)) {
      if (lane == 0) raise_flags(error_flags, SRKV_EFLAG_TIMEOUT);
      break;
    }
    finish_columns<T, D>(ps, warp, lane, v, reps + slab * D);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// Decode-time maintenance: CTA (request r, kv head h) writes the new token's key and value
// at position L = seq_lens[r] (page block_table[r][L / 128], row L % 128) and recomputes the
// page's representation vector over its rows [0, L % 128] with the arithmetic of
// block_reps_kernel.
template <typename T, int D>
__global__ void __launch_bounds__(kRepThreads)
    append_kv_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* k_cache,
                     T* v_cache, int64_t num_pages, const int32_t* __restrict__ block_table,
                     int32_t max_blocks, const int32_t* __restrict__ seq_lens, int32_t Hkv,
                     float* __restrict__ reps, int32_t* error_flags) {
  using R = RepGeom<T, D>;
  __shared__ float part[kRepWarps * D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t r = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
  griddep_wait();  // programmatic launch: the inputs may be the previous kernel's outputs
  griddep_launch_dependents();
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
  if (threadIdx.x < R::LPR) {
    reinterpret_cast<int4*>(k_cache + slab + (int64_t)row * D)[threadIdx.x] =
        reinterpret_cast<const int4*>(k_new + src)[threadIdx.x];
    reinterpret_cast<int4*>(v_cache + slab + (int64_t)row * D)[threadIdx.x] =
        reinterpret_cast<const int4*>(v_new + src)[threadIdx.x];
  }
  __syncthreads();  // the new row is visible to the CTA's own (coherent) loads
  const int4* rows = reinterpret_cast<const int4*>(k_cache + slab);
  float acc[R::EPV];
  warp_column_sums<T, D>([&](int rr, int chunk) { return rows[rr * R::LPR + chunk]; }, warp,
                         lane, row + 1, acc);
  store_column_sums<T, D>(part, warp, lane, acc);
  __syncthreads();
  finish_columns<T, D>(part, warp, lane, row + 1, reps + ((int64_t)page * Hkv + h) * D);
}

int32_t device_sms() {
  static int32_t cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

// Launch as a programmatic dependent of the previous kernel in the stream (the kernel waits
// for it before reading its inputs), so that consecutive launches overlap their start-up.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(block);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<Params>(args)...);
}

template <typename T, int D>
cudaError_t launch(const void* k, int64_t P, int32_t Hkv, const int32_t* ids,
                   const int32_t* valid, int32_t n, float* reps, int32_t* flags,
                   cudaStream_t s) {
  using R = RepGeom<T, D>;
  const int64_t units = (int64_t)n * Hkv;
  if (units == 0) return cudaSuccess;
  const int32_t sms = device_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // The shared-memory opt-in is set once per device (not during graph capture).
  static bool configured[128] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(block_reps_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)R::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int64_t grid = units < sms ? units : sms;
  return launch_pdl(block_reps_kernel<T, D>, (unsigned)grid, kRepKernelThreads, R::kSmemAlloc,
                    s, static_cast<const T*>(k), P, Hkv, ids, valid, n, reps, flags);
}

template <typename T, int D>
cudaError_t launch_append(const void* kn, const void* vn, void* k, void* v, int64_t P,
                          const int32_t* bt, int32_t max_blocks, const int32_t* seq_lens,
                          int32_t batch, int32_t Hkv, float* reps, int32_t* flags,
                          cudaStream_t s) {
  const int64_t grid = (int64_t)batch * Hkv;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(append_kv_kernel<T, D>, (unsigned)grid, kRepThreads, 0, s,
                    static_cast<const T*>(kn), static_cast<const T*>(vn), static_cast<T*>(k),
                    static_cast<T*>(v), P, bt, max_blocks, seq_lens, Hkv, reps, flags);
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
