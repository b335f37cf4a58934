// decode_split_mma.cu -- split phase of sparse paged decode on tensor cores (bf16).
//
// openGauss DataVec "KV Cache Query-Based Computation Inference Acceleration", section
// "Overall Solution": the selected blocks are concatenated with the initial tokens and the
// sliding window and take part in attention; the ATB reuse article (§1.1) gives
// softmax(QK^T/sqrt(d_k))V and (§2.2, §3.1) reads K/V page by page through a page table
// staged on chip.  Each (page, kv head) slab of K or V is contiguous (S*d*2 bytes) and is
// moved by tiled TMA copies into shared memory (decode_mma.cuh).
//
// CTA = 1 producer warp + 8 consumer warps, one CTA per SM (persistent), each CTA owning
// an equal share of all units' page lists (see decode_plan.cuh).
//   producer: plans list A (initial + window pages) and list B (selected pages) with
//             warp-level scans, resolves 32 list positions at once (one per lane), and lane 0
//             streams the pages through the ring.  When the previous kernel is the scoring
//             kernel, list A is streamed before that kernel finishes (programmatic launch)
//             and the producer waits for the selection only before list B; a sentinel stage
//             ends the consumers' loop;
//   consumers: consumer_loop (decode_mma.cuh); at the end of a unit's segment the 8 warps
//             merge and warp 0 writes the partial to slot unit + CTA of the workspace.
// Every wait is bounded (SRKV_EFLAG_TIMEOUT).
#include "decode_mma.cuh"

namespace srkv {
namespace {

// 128 registers: a quarter-SM register file (16K) then holds this CTA's three warps on one
// sub-partition (12K) beside one warp of a combine CTA, so the combine is resident and
// waiting when the last partial is written.
template <int D, bool F8>
__global__ void __maxnreg__(128) split_mma_kernel(const DecodeArgs a,
                                                  const __grid_constant__ TmaMaps maps) {
  using C = Cfg<D, F8>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  StageInfo* sInfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_v = full + C::kStages;
  uint64_t* empty = full_v + C::kStages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The combine may be scheduled once every CTA has passed this point (it waits for this
  // grid before reading partials).  Without the early mode the inputs are only read after
  // the previous kernel in the stream has finished, and the combine reads them too.
  if (!a.early && !a.wait_late) griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) init_ring<D, F8>(smem);
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    uint32_t eflags = 0;
    bool abort = false;
    int64_t it = 0;     // stages handed out so far (uniform over the warp)
    int64_t armed = 0;  // stages lane 0 armed
    // Both lists are planned first: list B's counts are the selection counts, known from
    // the lengths alone in the early mode.  CTA 0 leaves each list's unit offsets for the
    // combine kernel.
    ListRange rgs[2];
#pragma unroll
    for (int list = kListA; list <= kListB; ++list) {
      int64_t* offsets = blockIdx.x == 0
                             ? reinterpret_cast<int64_t*>(a.ws + (list == kListA ? a.lay.off_a
                                                                                 : a.lay.off_b))
                             : nullptr;
      rgs[list] = warp_plan(a, list, blockIdx.x, list_ctas(a, list), offsets, nullptr, eflags);
    }
    for (int list = kListA; list <= kListB && !abort; ++list) {
      // the selection (or, behind the shared-prefix kernel, that kernel's partials) must
      // exist from here on
      if (list == kListB && (a.early || a.wait_late)) griddep_wait();
      const ListRange rg = rgs[list];
      const int64_t npos = rg.end - rg.begin;
      if (npos <= 0) continue;
      const uint32_t bank = list == kListB ? kBankB : 0u;
      int32_t cu = rg.u0;  // walk state: unit and position within its list
      int64_t cj = rg.begin - rg.base0;
      uint32_t dummy = 0;
      Geom cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
      int32_t cn = list == kListA ? list_a_count(cg) : cg.ns;
      for (int64_t done = 0; done < npos && !abort; done += 32) {
        const int cnt = npos - done < 32 ? (int)(npos - done) : 32;
        // Assign positions done .. done+cnt-1 to lanes (uniform walk over the units).
        int32_t my_u = 0, my_j = 0;
        Geom my_g = cg;
        uint32_t my_flags = 0;
        for (int l = 0; l < cnt; ++l) {
          while (cj >= cn) {
            ++cu;
            cj = 0;
            cg = list == kListA ? unit_geom_a(a, cu, dummy) : unit_geom(a, cu, dummy);
            cn = list == kListA ? list_a_count(cg) : cg.ns;
          }
          const int64_t p = rg.begin + done + l;
          if (lane == l) {
            my_u = cu;
            my_j = (int32_t)cj;
            my_g = cg;
            my_flags = bank | ((cj == 0 || p == rg.begin) ? kNewUnit : 0u) |
                       ((cj == cn - 1 || p == rg.end - 1) ? kSegEnd : 0u);
          }
          ++cj;
        }
        PageTask task;
        task.page = -1;
        task.lo = task.hi = task.ie = task.ws = 0;
        if (lane < cnt) {
          const int32_t* bt_r = a.block_table + (int64_t)(my_u / a.Hkv) * a.max_blocks;
          // Early mode: the count the plan assumed must be the one the scoring wrote.
          const int32_t written = list == kListB && a.early ? a.nsel[my_u] : my_g.ns;
          task = list == kListA
                     ? resolve_a(my_g, my_j, bt_r, total_pages(a), eflags)
                     : resolve_b(my_g, my_j, a.sel + (int64_t)my_u * a.kmax, bt_r, total_pages(a),
                                 a.init_tokens, eflags);
          if (list == kListB && (my_j >= written || (my_j == 0 && written != my_g.ns))) {
            eflags |= SRKV_EFLAG_SELECTION;
            if (my_j >= written) task.page = -1;
          }
        }
        for (int l = 0; l < cnt; ++l) {
          PageTask t;
          const int32_t u = __shfl_sync(0xffffffffu, my_u, l);
          const uint32_t fl = __shfl_sync(0xffffffffu, my_flags, l);
          t.page = __shfl_sync(0xffffffffu, task.page, l);
          t.lo = __shfl_sync(0xffffffffu, task.lo, l);
          t.hi = __shfl_sync(0xffffffffu, task.hi, l);
          t.ie = __shfl_sync(0xffffffffu, task.ie, l);
          t.ws = __shfl_sync(0xffffffffu, task.ws, l);
          // A selected shared-prefix block loads nothing here (the cascade kernel attends
          // it); it takes a stage only when it opens or closes the unit's segment.
          if (a.prefix_blocks > 0 && t.page < 0 && !(fl & (kNewUnit | kSegEnd))) continue;
          issue_stage_warp<D, F8>(a, maps, smem, it, u, fl, t, armed, abort, eflags, lane);
          ++it;
        }
      }
    }
    if (lane == 0) {
      PageTask none;
      none.page = -1;
      none.lo = none.hi = none.ie = none.ws = 0;
      issue_stage<D, F8>(a, maps, smem, it, -1, kLast, none, armed, abort, eflags);  // sentinel
      // Drain: every copy this CTA issued must land before the CTA exits.
      const int64_t first = armed > C::kStages ? armed - C::kStages : 0;
      for (int64_t i = first; i < armed; ++i)
        if (!mbar_wait(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1)) ||
            !mbar_wait(&full_v[i % C::kStages], (uint32_t)((i / C::kStages) & 1))) {
          eflags |= SRKV_EFLAG_TIMEOUT;
          break;
        }
    }
    eflags = __reduce_or_sync(0xffffffffu, eflags);
    if (lane == 0) raise_flags(a.error_flags, eflags);
    return;
  }

  // -------------------------------------------------------------------- consumers
  // warp 0 writes the partial of (unit, this CTA) into the list's bank
  consumer_loop<D, F8>(a, smem, lane, warp, [&](const SoftmaxState<D>& st, const StageInfo& inf,
                                            Lane ln) {
    const int64_t slot =
        ((inf.flags & kBankB) ? (int64_t)a.lay.bank : 0) + inf.unit + blockIdx.x;
    store_partial<D, F8>(reinterpret_cast<float*>(a.ws + a.lay.acc) + slot * a.G * D,
                     reinterpret_cast<float*>(a.ws + a.lay.ml) + slot * a.G * 2, st, ln, a.G);
  });
}

}  // namespace

bool mma_split_supported(const srkv_config& cfg) {
  const int32_t G = cfg.num_q_heads / cfg.num_kv_heads;
  return cfg.dtype == SRKV_BF16 && (cfg.head_dim == 128 || cfg.head_dim == 64) && G >= 1 &&
         G <= 8;
}

int32_t mma_split_ctas(int32_t sm_count) { return sm_count; }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiled encode_tiled() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [num_pages][Hkv * 128][d] of bf16 (boxes of 64 columns) or E4M3 bytes (boxes of 128
// columns): 128-byte-wide boxes of 128 rows, 128-byte swizzle.
// The maps of the last few caches this host thread encoded are kept (a map is a function of
// these arguments alone), so a decode loop over the same caches encodes none per call.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_pages, int32_t Hkv,
                      int32_t d, bool e4m3) {
  struct Entry {
    const void* base;
    int64_t num_pages;
    int32_t Hkv, d;
    bool e4m3, used;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i) {
    const Entry& c = cache[i];
    if (c.used && c.base == base && c.num_pages == num_pages && c.Hkv == Hkv && c.d == d &&
        c.e4m3 == e4m3) {
      *map = c.map;
      return true;
    }
  }
  const EncodeTiled fn = encode_tiled();
  if (!fn || num_pages > INT32_MAX || (int64_t)Hkv * kBlock > INT32_MAX) return false;
  const cuuint64_t elem = e4m3 ? 1 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hkv * kBlock, (cuuint64_t)num_pages};
  const cuuint64_t strides[2] = {(cuuint64_t)d * elem, (cuuint64_t)Hkv * kBlock * d * elem};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / elem), (cuuint32_t)kBlock, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& c = cache[next];
  next = (next + 1) % kEntries;
  c = Entry{base, num_pages, Hkv, d, e4m3, true, *map};
  return true;
}

template <int D, bool F8>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t stream) {
  // The shared-memory opt-in is set once per device (not during graph capture).
  static bool configured[128] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(split_mma_kernel<D, F8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg<D, F8>::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  TmaMaps maps;
  if (!encode_cache_map(&maps.k, a.k_cache, a.num_pages, a.Hkv, D, F8) ||
      !encode_cache_map(&maps.v, a.v_cache, a.num_pages, a.Hkv, D, F8))
    return cudaErrorInvalidValue;
  return launch_pdl(split_mma_kernel<D, F8>, dim3(a.ctas), dim3(kThreads),
                    Cfg<D, F8>::kSmemAlloc, stream, a, maps);
}

cudaError_t launch_split_mma(const DecodeArgs& a, cudaStream_t stream) {
  if (a.k_scale) return launch_d<128, true>(a, stream);  // compressed pages (d 128)
  return a.d == 128 ? launch_d<128, false>(a, stream) : launch_d<64, false>(a, stream);
}

}  // namespace srkv
