// rowstat.cuh -- statistics of target-logit rows: running (max, argmax, sum of
// exp((z - max) / T)), combinable across threads and chunks. Used by the standalone
// reduction kernel and by the spare warps of the LM-head kernel.
#pragma once

#include "common.cuh"

namespace dfs {

constexpr int kIntMaxRs = 0x7fffffff;
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(y) = 2^(y log2 e)

// 2^x on the special-function unit (ex2.approx.ftz.f32, relative error about 2^-22): one
// instruction per term of the target rows' sums of exponentials.
__device__ __forceinline__ float exp2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// The same statistics over NG groups of 8 bf16 elements still packed as loaded (16 bytes
// per group), so twice as many loads fit in the registers a thread keeps in flight. One
// pass, one group unpacked at a time: the running maximum is raised group by group and the
// running sum rescaled by exp((old max - new max) / T) when it rises (the online form of
// the same sum). Indices within a thread increase, so ties keep the lower index.
template <int NG, bool kSoft>
__device__ __forceinline__ void rowstat_fold_bf16(RowStat& st, const uint4 (&q)[NG],
                                                  const int (&v0)[NG], int V, float inv_T) {
  float m = -INFINITY, s = 0.f;
  int mi = kIntMaxRs;
  const float c = inv_T * kLog2e;  // exp((x - m) / T) = 2^(x c - m c)
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    if (v0[g] >= V) continue;
    const uint32_t w[4] = {q[g].x, q[g].y, q[g].z, q[g].w};
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      x[j] = bf16_bits_to_float((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
    float gm = x[0];
    int gj = 0;
#pragma unroll
    for (int j = 1; j < 8; ++j)
      if (x[j] > gm) {
        gm = x[j];
        gj = j;
      }
    if (gm > m) {
      if (kSoft) s *= exp2_sfu((m - gm) * c);
      m = gm;
      mi = v0[g] + gj;
    }
    if (kSoft && m != -INFINITY) {
      const float mc = m * c;
#pragma unroll
      for (int j = 0; j < 8; ++j) s += exp2_sfu(fmaf(x[j], c, -mc));
    }
  }
  if (m == -INFINITY) return;
  if (kSoft) {
    st = combine(st, RowStat{m, mi, s}, inv_T);
  } else if (m > st.m) {
    st.m = m;
    st.i = mi;
  }
}

// Statistics of one kZChunk-element chunk of one target row by one warp: every lane's loads
// are issued together (16 x 16 bytes for bf16), then folded and combined across the warp.
__device__ __forceinline__ RowStat zchunk_stat_warp(const void* Z, int is_bf16, size_t rbase,
                                                    int chunk, int V, float inv_T, int lane) {
  RowStat st = rowstat_empty();
  if (is_bf16) {
    uint4 q[16];
    int v0[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      v0[g] = chunk * 4096 + g * 256 + lane * 8;
      if (v0[g] < V)
        q[g] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(Z) + rbase + v0[g]));
    }
    if (inv_T > 0.f)
      rowstat_fold_bf16<16, true>(st, q, v0, V, inv_T);
    else
      rowstat_fold_bf16<16, false>(st, q, v0, V, 0.f);
  } else {
#pragma unroll 1
    for (int bt = 0; bt < 2; ++bt) {
      float x[8][8];
      int v0[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        v0[g] = chunk * 4096 + (bt * 8 + g) * 256 + lane * 8;
        if (v0[g] < V) load8_stream(Z, 0, rbase + v0[g], x[g]);
      }
      if (inv_T > 0.f)
        rowstat_fold<8, true>(st, x, v0, V, inv_T);
      else
        rowstat_fold<8, false>(st, x, v0, V, 0.f);
    }
  }
  return warp_combine(st, inv_T);
}

}  // namespace dfs
