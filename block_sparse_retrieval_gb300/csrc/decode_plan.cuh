// decode_plan.cuh -- how the split grid divides the attended pages of all units.
//
// Flash-decoding style split (KV-cache survey "大模型推理百倍加速之KV cache篇", section
// "Share--KV cache共享": partial attention results are merged like Flash-Decoding).  The
// page lists of all (request, kv head) units are concatenated in unit order, T positions in
// total, and CTA c of C takes positions [c*T/C, (c+1)*T/C).  Every CTA therefore gets the
// same number of pages whatever the lengths of the requests (ragged batches balance by
// construction).  A CTA writes one partial (max, sum, unnormalised output) per unit its
// range touches, into slot u + c: along the staircase of (unit, CTA) pairs each step raises
// u or c, so the slot is unique and at most U + C - 1 slots are used.
#pragma once

#include "srkv_internal.cuh"

namespace srkv {

template <int NT>
__device__ __forceinline__ int64_t block_exclusive_scan64(int64_t v, int64_t* scratch,
                                                          int64_t* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < NW ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) scratch[lane] = w;
  }
  __syncthreads();
  const int64_t before = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[NW - 1];
  __syncthreads();
  return before + x - v;
}

struct CtaRange {
  int64_t T;      // positions of all units
  int64_t begin;  // this CTA's first position
  int64_t end;    // one past its last
  int32_t u0;     // unit holding `begin`
  int64_t base0;  // first position of unit u0
};

// Shared-memory scratch of the planner: NT/32 int64 + 2 int64.
template <int NT>
__device__ CtaRange plan_cta_range(const DecodeArgs& a, int64_t* scratch) {
  const int32_t U = a.batch * a.Hkv;
  const int32_t chunk = (U + NT - 1) / NT;
  const int32_t u_lo = min(U, (int32_t)threadIdx.x * chunk);
  const int32_t u_hi = min(U, u_lo + chunk);
  uint32_t eflags = 0;
  int64_t local = 0;
  for (int32_t u = u_lo; u < u_hi; ++u) {
    const Geom g = make_geom(a.seq_lens[u / a.Hkv], a.nsel[u], a.max_blocks, a.kmax,
                             a.init_tokens, a.local_tokens, eflags);
    local += g.npos();
  }
  int64_t T;
  const int64_t excl = block_exclusive_scan64<NT>(local, scratch, &T);
  CtaRange rg;
  rg.T = T;
  rg.begin = cta_begin(blockIdx.x, T, gridDim.x);
  rg.end = cta_begin(blockIdx.x + 1, T, gridDim.x);
  int64_t* s_found = scratch + NT / 32;  // [0] = u0, [1] = base0
  if (rg.begin < rg.end && excl <= rg.begin && rg.begin < excl + local) {
    int64_t pos = excl;
    uint32_t dummy = 0;
    for (int32_t u = u_lo; u < u_hi; ++u) {
      const Geom g = make_geom(a.seq_lens[u / a.Hkv], a.nsel[u], a.max_blocks, a.kmax,
                               a.init_tokens, a.local_tokens, dummy);
      if (rg.begin < pos + g.npos()) {
        s_found[0] = u;
        s_found[1] = pos;
        break;
      }
      pos += g.npos();
    }
  }
  if (blockIdx.x == 0) {  // unit tables for the combine pass
    int32_t* unit_n = reinterpret_cast<int32_t*>(a.ws + a.lay.unit_n);
    int64_t* unit_off = reinterpret_cast<int64_t*>(a.ws + a.lay.unit_off);
    int64_t pos = excl;
    uint32_t dummy = 0;
    for (int32_t u = u_lo; u < u_hi; ++u) {
      const Geom g = make_geom(a.seq_lens[u / a.Hkv], a.nsel[u], a.max_blocks, a.kmax,
                               a.init_tokens, a.local_tokens, dummy);
      unit_n[u] = g.npos();
      unit_off[u] = pos;
      pos += g.npos();
    }
    if (threadIdx.x == 0) unit_off[U] = T;
    raise_flags(a.error_flags, eflags);
  }
  __syncthreads();
  if (rg.begin < rg.end) {
    rg.u0 = (int32_t)s_found[0];
    rg.base0 = s_found[1];
  } else {
    rg.u0 = 0;
    rg.base0 = 0;
  }
  return rg;
}

}  // namespace srkv
