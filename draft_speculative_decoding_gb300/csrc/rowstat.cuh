// rowstat.cuh -- statistics of target-logit rows: running (max, argmax, sum of
// exp((z - max) / T)), combinable across threads and chunks. Used by the standalone
// reduction kernel and by the spare warps of the LM-head kernel.
#pragma once

#include "common.cuh"

namespace dfs {

constexpr int kIntMaxRs = 0x7fffffff;

// (max, argmax, sum of exp((z - max) * inv_T)); ties keep the lower index.
struct RowStat {
  float m;
  int i;
  float s;
};

__device__ __forceinline__ RowStat rowstat_empty() { return RowStat{-INFINITY, kIntMaxRs, 0.f}; }

__device__ __forceinline__ RowStat combine(RowStat a, RowStat b, float inv_T) {
  if (b.m == -INFINITY) return a;
  if (a.m == -INFINITY) return b;
  RowStat r;
  const bool take_b = ranks_before(b.m, b.i, a.m, a.i);
  r.m = take_b ? b.m : a.m;
  r.i = take_b ? b.i : a.i;
  r.s = a.s * expf((a.m - r.m) * inv_T) + b.s * expf((b.m - r.m) * inv_T);
  return r;
}

__device__ __forceinline__ RowStat warp_combine(RowStat v, float inv_T) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    RowStat o;
    o.m = __shfl_xor_sync(0xffffffffu, v.m, off);
    o.i = __shfl_xor_sync(0xffffffffu, v.i, off);
    o.s = __shfl_xor_sync(0xffffffffu, v.s, off);
    v = combine(v, o, inv_T);
  }
  return v;
}

// 8 consecutive elements (16-byte aligned) of a bf16 or fp32 row, streamed (read once).
__device__ __forceinline__ void load8_stream(const void* base, int is_bf16, size_t idx,
                                             float (&x)[8]) {
  if (is_bf16) {
    const uint4 q = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
      x[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = __ldcs(p), b = __ldcs(p + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Fold NG groups of 8 elements (element v0[g] + j) into a running statistic: the group
// maximum first, then one exp per element relative to the updated maximum. Elements at or
// beyond V are skipped; indices within a thread increase, so ties keep the lower index.
template <int NG, bool kSoft>
__device__ __forceinline__ void rowstat_fold(RowStat& st, const float (&x)[NG][8],
                                             const int (&v0)[NG], int V, float inv_T) {
  float bm = -INFINITY;
  int bi = kIntMaxRs;
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (v0[g] < V && x[g][j] > bm) {
        bm = x[g][j];
        bi = v0[g] + j;
      }
  if (bm == -INFINITY) return;
  if (kSoft) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (v0[g] < V) s += expf((x[g][j] - bm) * inv_T);
    st = combine(st, RowStat{bm, bi, s}, inv_T);
  } else {
    if (bm > st.m) {
      st.m = bm;
      st.i = bi;
    }
  }
}

}  // namespace dfs
