// select_tail.cu -- everything after the LM head: target-logit row statistics, the merge
// of partial top-16 lists, bilinear pair scores, greedy / Viterbi paths, greedy and
// rejection-sampling verification with the redraw.
//
// Sources:
//   "DFlash 2: Keep Drafting Parallel", section "A lightweight path selector":
//     S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>, all adjacent pairs scored at once;
//     the only sequential work is one traversal from the last verified token following
//     the best successor; rejection sampling recovers the target distribution.
//   "DFlash 2 讓 Qwen3.8-27B 快了兩倍", section 2 (Viterbi dynamic programming over the
//     candidate lattice) and section "The output is exactly the same" (greedy output
//     equals autoregressive decoding; sampling keeps the target distribution).
//   Table 1 caption of the blog: the verify length counts the verifier's next token.
//
// The work here is small and latency-bound, so it is organised around round trips: one
// block per (request, position) merges, scores and hands its 16 x 16 scores to the last
// block of its request (an atomic counter, no spinning), which selects the path and
// verifies it. Every global-to-shared copy issues all of a thread's loads before any
// store, so a phase costs one memory round trip.
#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"
#include "rowstat.cuh"

namespace dfs {

namespace {

constexpr int kTailThreads = 256;
constexpr int kIntMax = 0x7fffffff;

// ------------------------------------------------------------------ loads
__device__ __forceinline__ void load8(const void* base, int is_bf16, size_t idx, float (&x)[8]) {
  if (is_bf16) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
      x[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

__device__ __forceinline__ float load1(const void* base, int is_bf16, size_t idx) {
  return is_bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx])
                 : static_cast<const float*>(base)[idx];
}

// A contiguous run of 16-byte chunks to copy from global to shared memory.
struct Seg {
  const uint4* src;
  uint4* dst;
  int n;
};

// Chunk j of the concatenated segments: its source and destination (static indexing only,
// so the segment table stays in registers).
template <int kNSeg>
__device__ __forceinline__ void seg_locate(const Seg (&seg)[kNSeg], int j, const uint4*& src,
                                           uint4*& dst) {
  src = nullptr;
  dst = nullptr;
#pragma unroll
  for (int q = 0; q < kNSeg; ++q) {
    if (src == nullptr) {
      if (j < seg[q].n) {
        src = seg[q].src + j;
        dst = seg[q].dst + j;
      } else {
        j -= seg[q].n;
      }
    }
  }
}

// Copies the segments with every thread's loads issued before its stores (one round trip).
template <int kMaxPer, int kNSeg>
__device__ __forceinline__ void staged_copy(const Seg (&seg)[kNSeg]) {
  int total = 0;
#pragma unroll
  for (int q = 0; q < kNSeg; ++q) total += seg[q].n;
  uint4 r[kMaxPer];
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int j = threadIdx.x + k * blockDim.x;
    if (j < total) {
      const uint4* src;
      uint4* dst;
      seg_locate(seg, j, src, dst);
      r[k] = __ldcg(src);
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int j = threadIdx.x + k * blockDim.x;
    if (j < total) {
      const uint4* src;
      uint4* dst;
      seg_locate(seg, j, src, dst);
      *dst = r[k];
    }
  }
}

// Device-scope acquire-release add (returns the old value).
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ------------------------------------------------------------------ packed keys
// (value desc, id asc) as one unsigned 64-bit key: larger key = ranks first.
__device__ __forceinline__ unsigned long long pack_key(float v, int id) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0, so equal values compare equal
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}


// ------------------------------------------------------------------ target rows
// One block of 128 threads reduces kZChunk (4096) elements of one row of Z: each thread
// holds 4 groups of 8 consecutive elements, the groups 1024 elements apart. Block (c, y)
// takes chunk c of row y; with kStrided, of rows y, y + gridDim.y, ... (more rows than the
// 65535 blocks of the second grid dimension; the one-row form measured faster where it fits).
template <bool kSoft, bool kStrided>
__global__ void __launch_bounds__(128) k_zreduce(const void* Z, int is_bf16, int rows, int V,
                                                 int nchunk, float inv_T, float* zmax, int* zarg,
                                                 float* zsum, int* zero_ptr, int zero_count) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && zero_ptr != nullptr)
    for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_ptr[i] = 0;
  const int chunk = blockIdx.x;
  __shared__ RowStat ws[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int row = blockIdx.y; row < rows; row += gridDim.y) {
    const size_t rbase = static_cast<size_t>(row) * V;
    float x[4][8];
    int v0[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      v0[g] = chunk * kZChunk + g * 1024 + threadIdx.x * 8;
      if (v0[g] < V) load8_stream(Z, is_bf16, rbase + v0[g], x[g]);
    }
    RowStat st = rowstat_empty();
    rowstat_fold<4, kSoft>(st, x, v0, V, inv_T);
    st = warp_combine(st, inv_T);
    if (lane == 0) ws[warp] = st;
    __syncthreads();
    if (warp == 0) {
      st = lane < 4 ? ws[lane] : rowstat_empty();
      st = warp_combine(st, inv_T);
      if (lane == 0) {
        const size_t o = static_cast<size_t>(row) * nchunk + chunk;
        zmax[o] = st.m;
        zarg[o] = st.i;
        if (kSoft) zsum[o] = st.s;
      }
    }
    if (!kStrided) break;
    __syncthreads();  // ws is rewritten by the next row
  }
}

// Merged statistics of one target row, computed by one warp (a lane's chunk loads are
// issued together).
__device__ RowStat row_stat_warp(const TailLaunch& a, int row) {
  RowStat st = rowstat_empty();
  const bool soft = a.T > 0.f;
  const float inv_T = soft ? 1.0f / a.T : 0.f;
  const int lane = threadIdx.x & 31;
  for (int c0 = 0; c0 < a.nchunk; c0 += 128) {
    float m[4], s[4];
    int ix[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = c0 + lane + 32 * k;
      const size_t o = static_cast<size_t>(row) * a.nchunk + c;
      const bool in = c < a.nchunk;
      m[k] = in ? __ldcg(a.zmax + o) : -INFINITY;
      ix[k] = in ? __ldcg(a.zarg + o) : kIntMax;
      s[k] = (in && soft) ? __ldcg(a.zsum + o) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) st = combine(st, RowStat{m[k], ix[k], s[k]}, inv_T);
  }
  return warp_combine(st, inv_T);
}

// ------------------------------------------------------------------ top-16 merge
// A float as an unsigned key with the same order (larger float -> larger key; -0 == +0).
__device__ __forceinline__ uint32_t ord_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The lane holding the warp's best (value desc, id asc) candidate, among lanes with
// `has`; ties on both (only possible for empty-list sentinels) go to the lowest lane.
// Returns -1 when no lane has a candidate. Two single-instruction warp reductions.
__device__ __forceinline__ int warp_best_lane(bool has, float v, int id) {
  const uint32_t key = has ? ord_key(v) : 0u;
  const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
  if (mx == 0u) return -1;
  const bool top = has && key == mx;
  const uint32_t mid = __reduce_min_sync(0xffffffffu, top ? static_cast<uint32_t>(id) : 0xffffffffu);
  const unsigned w = __ballot_sync(0xffffffffu, top && static_cast<uint32_t>(id) == mid);
  return __ffs(w) - 1;
}

// Top 16 (value desc, id asc) of a set of G <= 256 sorted lists of 16, by warps m and m + 2
// (set m). The lists are staged as they are written: entry n of list j at place j * 16 + n.
// Ids are unique across lists (the vocabulary tiles partition V); the only repeated entries
// are the (-inf, INT_MAX) fillers, which merge_key tells apart by their place, below every
// real entry of equal value. So the keys of a set are distinct.
// 1. The lists are taken in groups of 2^lg consecutive lists, at most kMaxGroups groups (one
//    per lane of the two warps); a group's head is its best list head. Group heads are ranked
//    by counting (broadcast shared-memory loads). Only the 16 groups with the best heads can
//    hold a top-16 entry (each of those heads ranks before any other group's head, which
//    ranks before every other entry of that group), and theta, the 16th best group head, is
//    a lower bound on the 16th best key overall (16 distinct entries reach it).
// 2. Candidates, by warp m alone: the entries >= theta of those groups' lists (no other
//    entry reaches theta; in a sorted list they are a prefix), placed by a warp scan of the
//    prefix lengths, with their values and ids. The top 16 are among them. Logits without order across the vocabulary
//    tiles leave a few more than 16; logits that rise or fall with the id can leave hundreds.
// 3. Up to kCandMax candidates: each one's rank among them by counting; ranks 0..15 are the
//    result. More: merge_exact, by warps 0..3, takes over.
constexpr int kCandMax = 64;
constexpr int kMaxGroups = 40;
struct MergeSmem {
  unsigned long long gk[2][kMaxGroups];  // group heads
  unsigned long long ck[2][kCandMax + 2];  // candidate keys (one zero pad)
  unsigned long long theta[2];           // 16th best group head
  float cv[2][kCandMax];                // candidate values
  int ci[2][kCandMax];                  // candidate ids
  int gsel[2][kK];                     // groups by head rank
  int ncand[2];
  // merge_exact
  unsigned long long hk[2][kMaxLists];  // head keys
  int sel[2][kK];                       // lists by head rank
  float v1[16][kK];                     // tree levels: 16, 4 lists (both sets)
  int i1[16][kK];
  float v2[8][kK];                      // 8 lists
  int i2[8][kK];
};

__device__ __forceinline__ void bar_sync_warps0to3() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// warps m and m + 2, the two warps of set m
__device__ __forceinline__ void bar_sync_set(int m) {
  if (m == 0)
    asm volatile("bar.sync 3, 64;" ::: "memory");
  else
    asm volatile("bar.sync 4, 64;" ::: "memory");
}

// pack_key, except that a filler (id INT_MAX) takes the low word 0x7fffffff - pos: distinct
// for every place pos, and below the low word ~id of any real entry.
__device__ __forceinline__ unsigned long long merge_key(float v, int id, int pos) {
  const unsigned long long k = pack_key(v, id);
  return id == kIntMax ? ((k & 0xffffffff00000000ull) | static_cast<uint32_t>(0x7fffffff - pos)) : k;
}

// Set m's step 1, by its two warps (h = 0: warp m, h = 1: warp m + 2), each taking half of
// the groups, one per lane; ends with gsel and theta in shared memory for warp m. The heads
// are read from the lists gv/gi [G][16] in global memory (through L2), so that the fused
// kernel ranks them while the lists' bulk copy to shared memory is still in flight.
__device__ __forceinline__ void merge_rank_groups(const float* gv, const int* gi, int m, int h, int G,
                                                  MergeSmem& ms) {
  const int lane = threadIdx.x & 31;
  int lg = 0;
  while ((kMaxGroups << lg) < G) ++lg;
  const int gs = 1 << lg, ng = (G + gs - 1) >> lg, half = (ng + 1) >> 1;
  const int g = h * half + lane;
  const bool valid = lane < half && g < ng;
  unsigned long long k = 0;  // zero (below every key) past the last group
  if (valid) {
    // four heads' loads in flight at once (one L2 round trip for groups of up to four lists)
    for (int d0 = 0; d0 < gs; d0 += 4) {
      float hv[4];
      int hi[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = (g << lg) + d0 + e;
        const bool in = d0 + e < gs && j < G;
        hv[e] = in ? __ldcg(gv + j * kK) : 0.f;
        hi[e] = in ? __ldcg(gi + j * kK) : 0;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = (g << lg) + d0 + e;
        if (d0 + e < gs && j < G) {
          const unsigned long long x = merge_key(hv[e], hi[e], j * kK);
          k = x > k ? x : k;
        }
      }
    }
  }
  if (lane < half) ms.gk[m][g] = k;
  if (h == 0 && lane < kK) ms.gsel[m][lane] = -1;
  if (h == 0 && lane == 0) ms.theta[m] = 0;  // fewer than 16 groups: every entry is a candidate
  bar_sync_set(m);
  if (valid) {
    const ulonglong2* g2 = reinterpret_cast<const ulonglong2*>(ms.gk[m]);
    int rank = 0;
#pragma unroll 4
    for (int i = 0; i < half; ++i) {
      const ulonglong2 o = g2[i];  // broadcast
      rank += (o.x > k) + (o.y > k);
    }
    if (rank < kK) ms.gsel[m][rank] = g;
    if (rank == kK - 1) ms.theta[m] = k;
  }
  bar_sync_set(m);
}

// Set m's steps 2 and 3, by warp m alone. Returns the candidate count (the same in every
// lane); when it is at most kCandMax, outv/outi hold the top 16 and every lane of the warp
// sees them.
__device__ __forceinline__ int merge_candidates_warp(const float* sv, const int* si, int m, int G,
                                                     MergeSmem& ms, float* outv, int* outi) {
  const int lane = threadIdx.x & 31;
  int lg = 0;
  while ((kMaxGroups << lg) < G) ++lg;
  const int gs = 1 << lg;
  const unsigned long long theta = ms.theta[m];
  // 2. candidates: the lane takes selected lists lane, lane + 32, ... (16 * 2^lg <= 128); the
  // keys of the first four entries of its first list are kept for the writes
  const int nsl = kK << lg;
  int len[4], jl[4];
  unsigned long long kf[4];
  int total = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s = lane + 32 * i;
    len[i] = 0;
    jl[i] = 0;
    if (s < nsl) {
      const int g = ms.gsel[m][s >> lg];
      const int j = (g << lg) + (s & (gs - 1));
      jl[i] = j;
      if (g >= 0 && j < G) {  // the first four entries at once, the rest one by one
        int n = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const unsigned long long x = merge_key(sv[j * kK + e], si[j * kK + e], j * kK + e);
          if (i == 0) kf[e] = x;
          n += x >= theta;
        }
        if (n == 4)
          while (n < kK && merge_key(sv[j * kK + n], si[j * kK + n], j * kK + n) >= theta) ++n;
        len[i] = n;
      }
    }
    total += len[i];
  }
  int incl = total;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  const int c = __shfl_sync(0xffffffffu, incl, 31);
  if (c > kCandMax) return c;
  int q = incl - total;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = jl[i];
    for (int n = 0; n < len[i]; ++n, ++q) {
      const unsigned long long kn = n == 0 ? kf[0] : n == 1 ? kf[1] : n == 2 ? kf[2] : kf[3];
      ms.ck[m][q] = (i == 0 && n < 4) ? kn : merge_key(sv[j * kK + n], si[j * kK + n], j * kK + n);
      ms.cv[m][q] = sv[j * kK + n];
      ms.ci[m][q] = si[j * kK + n];
    }
  }
  if (lane == 0 && (c & 1)) ms.ck[m][c] = 0;  // pads the last pair: below every key
  __syncwarp();
  // 3. ranks among the candidates
  const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(ms.ck[m]);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int x = lane + 32 * h;
    if (x < c) {
      const unsigned long long k = ms.ck[m][x];
      int rank = 0;
#pragma unroll 4
      for (int i = 0; i < (c + 1) / 2; ++i) {
        const ulonglong2 o = c2[i];  // broadcast
        rank += (o.x > k) + (o.y > k);
      }
      if (rank < kK) {
        outv[rank] = ms.cv[m][x];
        outi[rank] = ms.ci[m][x];
      }
    }
  }
  __syncwarp();
  return c;
}

// Two sorted lists (element l16 of A and of B in lane l16 of this half-warp) merged into
// their top 16, sorted, in (av, ai). All 32 lanes of the warp call it.
__device__ __forceinline__ void merge2_halfwarp(float& av, int& ai, float bv, int bi) {
  const int l16 = threadIdx.x & 15;
  const float rv = __shfl_xor_sync(0xffffffffu, bv, 15);  // B[15 - l16]
  const int ri = __shfl_xor_sync(0xffffffffu, bi, 15);
  if (pack_key(rv, ri) > pack_key(av, ai)) {
    av = rv;
    ai = ri;
  }
#pragma unroll
  for (int d = 8; d > 0; d >>= 1) {
    const float pv = __shfl_xor_sync(0xffffffffu, av, d);
    const int pi = __shfl_xor_sync(0xffffffffu, ai, d);
    const bool lower = (l16 & d) == 0;  // the lower index keeps the better one
    if ((pack_key(pv, pi) > pack_key(av, ai)) == lower) {
      av = pv;
      ai = pi;
    }
  }
}

// The exact merge, for sets with more than kCandMax candidates, by warps 0..3 (they sync
// among themselves): every head ranked by counting, then a merge tree over the 16 lists with
// the best heads: a half-warp merges two sorted lists into their top 16 (the elementwise
// better of A[l] and B[15-l] is bitonic, four half-cleaner steps sort it), 16 -> 8 -> 4 -> 2
// -> 1 lists per set. Set m's top 16 go to outv[m]/outi[m] where wm (w0, w1) is set.
__device__ __noinline__ void merge_exact(const float* sv0, const int* si0, const float* sv1, const int* si1,
                                         int nm, int G, MergeSmem& ms, float* outv0, int* outi0,
                                         float* outv1, int* outi1, bool w0, bool w1) {
  const int tid = threadIdx.x;
  for (int x = tid; x < nm * G; x += 128) {
    const int m = x >= G, j = x - m * G;
    ms.hk[m][j] = merge_key((m ? sv1 : sv0)[j * kK], (m ? si1 : si0)[j * kK], j * kK);
  }
  if (tid < 2 * kK) ms.sel[tid >> 4][tid & 15] = -1;
  bar_sync_warps0to3();
  for (int x = tid; x < nm * G; x += 128) {
    const int m = x >= G, j = x - m * G;
    const unsigned long long k = ms.hk[m][j];
    int rank = 0;
    for (int i = 0; i < G; ++i) rank += ms.hk[m][i] > k;
    if (rank < kK) ms.sel[m][rank] = j;
  }
  bar_sync_warps0to3();
  const int warp = tid >> 5, lane = tid & 31, l16 = lane & 15;
  const int h = lane >> 4;
#pragma unroll 1
  for (int rep = 0; rep < 2; ++rep) {  // 16 -> 8 lists per set: merge q, lists 2p, 2p+1
    const int q = rep * 8 + warp * 2 + h, m = q >> 3, p = q & 7;
    const float* sv = m ? sv1 : sv0;
    const int* si = m ? si1 : si0;
    const int la = m < nm ? ms.sel[m][2 * p] : -1, lb = m < nm ? ms.sel[m][2 * p + 1] : -1;
    float av = la >= 0 ? sv[la * kK + l16] : -INFINITY;
    int ai = la >= 0 ? si[la * kK + l16] : kIntMax;
    const float bv = lb >= 0 ? sv[lb * kK + l16] : -INFINITY;
    const int bi = lb >= 0 ? si[lb * kK + l16] : kIntMax;
    merge2_halfwarp(av, ai, bv, bi);
    ms.v1[q][l16] = av;
    ms.i1[q][l16] = ai;
  }
  bar_sync_warps0to3();
  {  // 8 -> 4 lists per set: merge q = 2 warp + h (q < 8), set q >> 2
    const int q = warp * 2 + h, m = q >> 2, p = q & 3;
    float av = ms.v1[m * 8 + 2 * p][l16];
    int ai = ms.i1[m * 8 + 2 * p][l16];
    merge2_halfwarp(av, ai, ms.v1[m * 8 + 2 * p + 1][l16], ms.i1[m * 8 + 2 * p + 1][l16]);
    ms.v2[q][l16] = av;
    ms.i2[q][l16] = ai;
  }
  bar_sync_warps0to3();
  if (warp < 2) {  // 4 -> 2 lists per set: merge q = 2 warp + h (q < 4), set q >> 1
    const int q = warp * 2 + h, m = q >> 1, p = q & 1;
    float av = ms.v2[m * 4 + 2 * p][l16];
    int ai = ms.i2[m * 4 + 2 * p][l16];
    merge2_halfwarp(av, ai, ms.v2[m * 4 + 2 * p + 1][l16], ms.i2[m * 4 + 2 * p + 1][l16]);
    ms.v1[q][l16] = av;  // level 1's lists are all consumed
    ms.i1[q][l16] = ai;
  }
  bar_sync_warps0to3();
  if (warp == 0) {  // 2 -> 1 list per set: half h is set h
    float av = ms.v1[2 * h][l16];
    int ai = ms.i1[2 * h][l16];
    merge2_halfwarp(av, ai, ms.v1[2 * h + 1][l16], ms.i1[2 * h + 1][l16]);
    if (h < nm && (h ? w1 : w0)) {
      (h ? outv1 : outv0)[l16] = av;
      (h ? outi1 : outi0)[l16] = ai;
    }
  }
  bar_sync_warps0to3();
}

// ------------------------------------------------------------------ pair scores
// S_t(a, c) = U_t(c) + sum_j A(a)_j g_j B(c)_j for the 16 x 16 pairs of one position.
// bf16 tables with r a multiple of 16 take the tensor-core path (gather_rows_bulk,
// pair_dot_mma, below); the others the SIMT path: first one warp gathers 16 table rows into
// fp32 shared rows dst[16][r+4],
// the A rows of the predecessors scaled by the gate g (isA), or the B rows of the
// candidates; lane l takes the 16-byte chunks l, l + 32, ... of every row, eight rows'
// loads in flight at a time. tok == nullptr: every row is token tok_all (position 1, where
// every predecessor is the last verified token). A token outside the vocabulary reads as a
// zero row.
__device__ __forceinline__ void gather_rows_warp(const TailLaunch& a, const int* tok, int tok_all, bool isA,
                                              float* dst, const float* g) {
  const int lane = threadIdx.x & 31;
  const int r = a.r, rs = r + 4;
  const int is_bf16 = a.dtype == 0;
  const int per_row = r * (is_bf16 ? 2 : 4) / 16;  // 16-byte chunks per row: <= 128
  const size_t row_bytes = static_cast<size_t>(r) * (is_bf16 ? 2 : 4);
  const char* tab = static_cast<const char*>(isA ? a.A : a.Bt);
  for (int ch = lane; ch < per_row; ch += 32) {
#pragma unroll 1
    for (int i0 = 0; i0 < kK; i0 += 8) {  // eight rows' loads in flight at a time
      uint4 raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = tok ? tok[i0 + i] : tok_all;
        raw[i] = (t >= 0 && t < a.V)
                     ? __ldg(reinterpret_cast<const uint4*>(tab + static_cast<size_t>(t) * row_bytes) + ch)
                     : make_uint4(0u, 0u, 0u, 0u);
      }
      if (is_bf16) {
        const int e0 = ch * 8;
        float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
        if (isA) {
          g0 = *reinterpret_cast<const float4*>(g + e0);
          g1 = *reinterpret_cast<const float4*>(g + e0 + 4);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
          float x[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            x[2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
            x[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
          }
          float* d = dst + (i0 + i) * rs + e0;
          *reinterpret_cast<float4*>(d) = make_float4(x[0] * g0.x, x[1] * g0.y, x[2] * g0.z, x[3] * g0.w);
          *reinterpret_cast<float4*>(d + 4) = make_float4(x[4] * g1.x, x[5] * g1.y, x[6] * g1.z, x[7] * g1.w);
        }
      } else {
        const int e0 = ch * 4;
        float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
        if (isA) gg = *reinterpret_cast<const float4*>(g + e0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(dst + (i0 + i) * rs + e0) =
              make_float4(__uint_as_float(raw[i].x) * gg.x, __uint_as_float(raw[i].y) * gg.y,
                          __uint_as_float(raw[i].z) * gg.z, __uint_as_float(raw[i].w) * gg.w);
      }
    }
  }
}

// The rows for the tensor-core products (bf16 tables, r a multiple of 16): one warp gathers
// 16 rows of `table` as they are (bf16) into dst[16][r + 8] by bulk copies completing on
// the mbarrier bar (lane i copies row i; the 16-byte pad per row keeps the MMA fragment
// loads free of bank conflicts). tok == nullptr: every row is token tok_all. A token
// outside the vocabulary gets a zero row, written by its lane (visible after a block
// barrier). The barrier's one arrival is lane 0's, with the bytes of the copied rows.
__device__ __forceinline__ void gather_rows_bulk(const TailLaunch& a, const int* tok, int tok_all,
                                                 const void* table, uint16_t* dst, uint32_t bar) {
  const int lane = threadIdx.x & 31;
  const int rowb = a.r * 2, rsb = (a.r + 8) * 2;
  int t = -1;
  if (lane < kK) {
    const int x = tok ? tok[lane] : tok_all;
    t = (x >= 0 && x < a.V) ? x : -1;
  }
  const unsigned ok = __ballot_sync(0xffffffffu, t >= 0);
  if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(ok) * rowb));
  __syncwarp();
  char* row = reinterpret_cast<char*>(dst) + lane * rsb;
  if (t >= 0) {
    bulk_load(smem_u32(row), static_cast<const char*>(table) + static_cast<size_t>(t) * rowb,
              static_cast<uint32_t>(rowb), bar);
  } else if (lane < kK) {
    for (int o = 0; o < rowb; o += 16) *reinterpret_cast<uint4*>(row + o) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// D += A (16 x 16, bf16, row-major fragment) * B (16 x 8, bf16, column fragment), fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The products on the tensor cores: the 16 x 16 scores are one 16 x 16 x r product of the
// gated A rows (A g) and the B rows, both gathered as bf16 rows of stride r + 8. B enters
// the MMA as it is. Each A g value is formed in fp32 and split into bf16 hi + lo (hi =
// A g rounded, lo = the rest rounded), so (A g) B^T = hi B^T + lo B^T with about 16
// significant bits of A g (against the 24 of an fp32 product), every bf16 product exact
// and the sums in fp32. Warp w takes the k-steps of 16 w, w + 8, ...: two m16n8k16 MMAs
// (hi, lo) per step and half of the 16 candidates; the eight warps' partial tiles are summed
// through red[8][256] (shared memory). Returns the score of pair tid (a = tid / 16,
// c = tid % 16) in `pair`. Contains a block barrier.
__device__ float pair_dot_mma(int r, const uint16_t* Ab, const uint16_t* Bb, const float* g,
                              const float* cur_U, float* red, int& pair) {
  const int rsb = r + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int k0 = warp * 16; k0 < r; k0 += 8 * 16) {
    uint32_t ahi[4], alo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // a0..a3: rows gq, gq + 8; columns k0 + 2 tq, + 8
      const int col = k0 + 8 * (q >> 1) + 2 * tq;
      const uint32_t w = *reinterpret_cast<const uint32_t*>(Ab + (gq + 8 * (q & 1)) * rsb + col);
      const float2 gg = *reinterpret_cast<const float2*>(g + col);
      const float x0 = bf16_bits_to_float(w & 0xFFFFu) * gg.x, x1 = bf16_bits_to_float(w >> 16) * gg.y;
      const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
      const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
      ahi[q] = *reinterpret_cast<const uint32_t*>(&h);
      alo[q] = *reinterpret_cast<const uint32_t*>(&l);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {  // candidates 8 nt .. 8 nt + 7
      const uint16_t* brow = Bb + (8 * nt + gq) * rsb + k0 + 2 * tq;
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(brow);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(brow + 8);
      mma_bf16_16816(d[nt], ahi, b0, b1);
      mma_bf16_16816(d[nt], alo, b0, b1);
    }
  }
  // d[nt]: rows gq (0, 1) and gq + 8 (2, 3), columns 8 nt + 2 tq (+1)
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float* rw = red + warp * 256 + 8 * nt + 2 * tq;
    *reinterpret_cast<float2*>(rw + gq * 16) = make_float2(d[nt][0], d[nt][1]);
    *reinterpret_cast<float2*>(rw + (gq + 8) * 16) = make_float2(d[nt][2], d[nt][3]);
  }
  __syncthreads();
  const int t = threadIdx.x;
  float acc = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) acc += red[w * 256 + t];
  pair = t;
  return cur_U[t & 15] + acc;
}

// Then the SIMT products, by the whole block once P (the gated A rows) and Q (the B rows) are
// in place: thread (blk = tid / 16, ks = tid % 16) accumulates a 4 x 4 block of pairs (a in
// 4 (blk / 4) + 0..3, c in 4 (blk % 4) + 0..3) over the float4 chunks ks, ks + 16, ... of
// the rank, and the 16 lanes of each half-warp reduce-scatter the block so that lane ks ends
// with pair (4 (blk / 4) + ks / 4, 4 (blk % 4) + ks % 4). Returns that pair's score and its
// index a * 16 + c in `pair`.
__device__ float pair_dot_block(int r, const float* P, const float* Q, const float* cur_U, int& pair) {
  const int rs = r + 4;
  const int ks = threadIdx.x & 15, blk = threadIdx.x >> 4;
  const int a0 = 4 * (blk >> 2), c0 = 4 * (blk & 3);
  float acc[16];
#pragma unroll
  for (int o = 0; o < 16; ++o) acc[o] = 0.f;
  for (int kc = ks; kc < r / 4; kc += 16) {
    float4 pv[4], qv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pv[i] = reinterpret_cast<const float4*>(P + (a0 + i) * rs)[kc];
      qv[i] = reinterpret_cast<const float4*>(Q + (c0 + i) * rs)[kc];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float t = acc[i * 4 + j];
        t = fmaf(pv[i].x, qv[j].x, t);
        t = fmaf(pv[i].y, qv[j].y, t);
        t = fmaf(pv[i].z, qv[j].z, t);
        t = fmaf(pv[i].w, qv[j].w, t);
        acc[i * 4 + j] = t;
      }
  }
  // reduce-scatter over the 16 lanes: at step d the lane keeps the half of its outputs
  // selected by bit d of ks and adds its partner's copy of that half
#pragma unroll
  for (int d = 8, n = 16; d > 0; d >>= 1, n >>= 1) {
    const bool upper = (ks & d) != 0;
#pragma unroll
    for (int o = 0; o < n / 2; ++o) {
      const float send = upper ? acc[o] : acc[o + n / 2];
      const float keep = upper ? acc[o + n / 2] : acc[o];
      acc[o] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
  const int ai = a0 + (ks >> 2), ci = c0 + (ks & 3);
  pair = ai * kK + ci;
  return cur_U[ci] + acc[0];
}

// ------------------------------------------------------------------ path
// Sampled traversal (mode 2) by the whole block: from the last verified token, x_t is drawn
// from q_t(c) = softmax_c(S_t(x_{t-1}, c) / T) over the 16 candidates by one uniform (Philox
// stream 3, published by the position blocks in the row statistics: upub[p * 8 + 5] for
// position p + 1) against the cumulative q in candidate order; if rounding leaves no
// candidate above it, the last one with mass. With backward messages logb (the joint path
// draw, mode 3) the weights are S_t(x_{t-1}, c) / T + logb[t][c]. Every (position p,
// predecessor a) row's q and draw are computed first, one row per thread (the rows spread
// over all eight warps), the row's q kept in place of its scores; then thread 0 walks from
// predecessor 0 and the drawn rows' q are copied out. Writes path_tok[P], pidx[P] and
// q[P][16]; returns the path score in thread 0. Contains block barriers.
__device__ float path_sample_block(float* S, const int* ids, int P, float inv_T, const float* upub,
                                   int* path_tok, int* pidx, float* q, float* sdraw,
                                   unsigned char* draw, const float* logb = nullptr) {
  const int nrow = P * kK;  // at most 240: one pass of the 256 threads
  const int per_warp = (nrow + kTailThreads / 32 - 1) / (kTailThreads / 32);
  const int lane = threadIdx.x & 31, x = (threadIdx.x >> 5) * per_warp + lane;
  if (lane < per_warp && x < nrow) {
    float* row = S + x * kK;
    const float* lb = logb != nullptr ? logb + (x >> 4) * kK : nullptr;
    float v[kK], w[kK];
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < kK; ++c) {
      v[c] = row[c];
      w[c] = v[c] * inv_T + (lb != nullptr ? lb[c] : 0.f);
      m = fmaxf(m, w[c]);
    }
    float z = 0.f;
    float e[kK];
#pragma unroll
    for (int c = 0; c < kK; ++c) {
      e[c] = expf(w[c] - m);
      z += e[c];
    }
    const float rz = 1.0f / z;
    const float u = upub[(x >> 4) * 8 + 5];
    float cum = 0.f, v_pick = v[0], v_last = v[0];
    int pick = -1, last = 0;
#pragma unroll
    for (int c = 0; c < kK; ++c) {
      const float qc = e[c] * rz;
      cum += qc;
      if (qc > 0.f) {
        last = c;
        v_last = v[c];
      }
      if (pick < 0 && cum > u) {
        pick = c;
        v_pick = v[c];
      }
      row[c] = qc;
    }
    draw[x] = static_cast<unsigned char>(pick < 0 ? last : pick);
    sdraw[x] = pick < 0 ? v_last : v_pick;
  }
  __syncthreads();
  float total = 0.f;
  if (threadIdx.x == 0) {
    int a = 0;
    for (int p = 0; p < P; ++p) {
      const int c = draw[p * kK + a];
      total += sdraw[p * kK + a];
      path_tok[p] = ids[p * kK + c];
      pidx[p] = c;
      a = c;
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < P * kK; x += blockDim.x) {
    const int p = x >> 4, a = p == 0 ? 0 : pidx[p - 1];
    q[x] = S[(p * kK + a) * kK + (x & 15)];
  }
  __syncthreads();
  return total;
}

// Backward messages of the joint path draw (mode 3) by the whole block (256 threads):
// logb[P-1][c] = 0 and logb[p][a] = log sum_c exp(S_{p+1}(a, c) / T + logb[p+1][c]), one
// (a, c) term per thread, the log-sum-exp over c across a half-warp. Contains barriers.
__device__ void backward_messages_block(const float* S, int P, float inv_T, float* logb) {
  static_assert(kTailThreads == kK * kK, "one (a, c) term per thread");
  const int a = threadIdx.x >> 4, c = threadIdx.x & 15;
  if (threadIdx.x < kK) logb[(P - 1) * kK + threadIdx.x] = 0.f;
  __syncthreads();
  for (int p = P - 2; p >= 0; --p) {
    const float x = S[((p + 1) * kK + a) * kK + c] * inv_T + logb[(p + 1) * kK + c];
    float m = x;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float e = expf(x - m);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
    if (c == 0) logb[p * kK + a] = m + logf(e);
    __syncthreads();
  }
}

// Greedy traversal by one warp (dfs_path_select): x_t = argmax_c S_t(x_{t-1}, c) by (score
// desc, id asc). S [P][16][16] and ids [P][16] in shared memory; writes path_tok[P] (shared)
// and returns the path score in every lane.
__device__ float path_greedy_warp(const float* S, const int* ids, int P, int* path_tok) {
  const int lane = threadIdx.x & 31;
  const bool act = lane < kK;
  int a = 0;
  float total = 0.f;
#pragma unroll 1
  for (int p = 0; p < P; ++p) {
    const float v = act ? S[(p * kK + a) * kK + lane] : -INFINITY;
    int c = warp_best_lane(act, v, act ? ids[p * kK + lane] : kIntMax);
    c = c < 0 ? 0 : c;  // no orderable score at all (NaN row): take candidate 0
    total += __shfl_sync(0xffffffffu, v, c);
    if (lane == 0) path_tok[p] = ids[p * kK + c];
    a = c;
  }
  __syncwarp();
  return total;
}

// Viterbi by the whole block (256 threads): delta_1(c) = S_1(x0, c), delta_t(c) = max_a
// delta_{t-1}(a) + S_t(a, c), then the best final candidate (score desc, id asc) and the
// back-pointers. Thread (c, a) = (tid / 16, tid % 16) forms delta_{t-1}(a) + S_t(a, c), and
// the 16 threads of c (a half-warp) keep the best by (score desc, predecessor id asc) with a
// shuffle butterfly; of equal keys the lowest a wins. delta2 [2][16] alternates between
// positions, so one barrier per position suffices.
__device__ float path_viterbi_block(const float* S, const int* ids, int P, int* path_tok,
                                    unsigned char* bp, float* delta2, int* pidx) {
  const int tid = threadIdx.x, lane = tid & 31, c = tid >> 4, aa = tid & 15;
  if (tid < kK) delta2[tid] = S[tid];
  __syncthreads();
#pragma unroll 1
  for (int p = 1; p < P; ++p) {
    const float* dcur = delta2 + ((p - 1) & 1) * kK;
    float* dnext = delta2 + (p & 1) * kK;
    const float v = dcur[aa] + S[(p * kK + aa) * kK + c];
    const unsigned long long k = pack_key(v, ids[(p - 1) * kK + aa]);
    unsigned long long m = k;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
      m = o > m ? o : m;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, k == m) & (0xffffu << (lane & 16));
    if (lane == __ffs(hit) - 1) {
      dnext[c] = v;
      bp[p * kK + c] = static_cast<unsigned char>(aa);
    }
    __syncthreads();
  }
  float score = 0.f;
  if (tid < 32) {
    const bool act = lane < kK;
    const float* dl = delta2 + ((P - 1) & 1) * kK;
    const float v = act ? dl[lane] : -INFINITY;
    int cb = warp_best_lane(act, v, act ? ids[(P - 1) * kK + lane] : kIntMax);
    cb = cb < 0 ? 0 : cb;
    score = __shfl_sync(0xffffffffu, v, cb);
    if (lane == 0) {
      int cur = cb;
      for (int p = P - 1; p >= 0; --p) {
        path_tok[p] = ids[p * kK + cur];
        if (pidx) pidx[p] = cur;
        if (p > 0) cur = bp[p * kK + cur];
      }
    }
    __syncwarp();
  }
  return score;
}

// ------------------------------------------------------------------ verify
struct VerifySmem {
  float rm[kMaxL], rl[kMaxL], zx[kMaxL];
  int ry[kMaxL];
  int info[4];
  float ur[kMaxL];                 // the redraw uniform of each possible redraw row
  float frac;                      // the target's place within the chosen chunk's mass, [0, 1]
  float mass[kMaxZChunks];         // cumulative residual mass over chunks
  float wsum[kTailThreads / 32];   // in-chunk weight of each warp's tokens
  int wpick[kTailThreads / 32];    // each warp's first token past the target
  int wlast[kTailThreads / 32];    // each warp's last token with weight
  // sampled proposals: the rejected position's candidates in the chosen chunk
  uint32_t inchunk[kZChunk / 32];  // bit j: token lo + j is a candidate
  int cand[kK];                    // candidate ids
  float cfac[kK];                  // max(0, 1 - q/p): the candidate's residual weight factor
  float take[kK];                  // min(p, q) of each candidate on the chunk-mass scale
};

// Verification of request b given its path (shared memory), by the whole block: row
// statistics (one warp per row), the acceptance tests of all positions in parallel (one lane
// each), then for T > 0 the redraw: the first token of the row, in vocabulary order, whose
// cumulative residual weight exceeds one uniform times the row's total. It is found in two
// steps that take the same decision: the chunk whose cumulative mass first exceeds the
// target (from the per-chunk row statistics), then the token inside that chunk by its own
// cumulative weights, against the target's remainder past the earlier chunks.
// With a sampled proposal (prop_q != nullptr: q[P][16] over the candidates cand[P][16], the
// drawn one at pidx[t-1]) a draft is accepted when U < p(x_t) / q(x_t), and the redraw is
// from the residual max(0, p - q): a chunk's mass loses min(p, q) of each candidate in it,
// and a candidate's weight is scaled by max(0, 1 - q/p). Without one the proposal is the
// path itself (q = 1 on x_t).
// The statistics of target row `row` (b = row / L, n = row % L) for the request's last block,
// by one warp: dst[0..2] = max, argmax bits, log-sum-exp; at T > 0 also dst[3] = the
// acceptance uniform of the draft the row verifies (n < L - 1), dst[4] = the row's redraw
// uniform and, for the drawn paths (modes 2 and 3), dst[5] = the path uniform of position
// n + 1 (n < L - 1), all at counter position n + 1, so that the last block draws no Philox
// numbers itself.
__device__ void row_stat_publish(const TailLaunch& a, int row, float* dst) {
  const RowStat st = row_stat_warp(a, row);
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    dst[0] = st.m;
    dst[1] = __int_as_float(st.i);
    dst[2] = a.T > 0.f ? logf(st.s) : 0.f;
  }
  if (a.T > 0.f && lane < 3) {
    // lanes 0, 1, 2 side by side: the acceptance uniform (stream 0), the redraw uniform
    // (stream 1) and, for the drawn paths, the path uniform (stream 3) of position n + 1
    const int b = row / a.L, n = row - b * a.L;
    const bool drafted = n < a.L - 1;  // the bonus row verifies no draft and draws no path
    const bool drawn = a.path_mode == 2 || a.path_mode == 3;
    const float u = uniform_stream(a.seed, b, n + 1, lane == 2 ? 3ull : static_cast<uint64_t>(lane));
    if (lane == 0) dst[3] = drafted ? u : 0.f;
    if (lane == 1) dst[4] = u;
    if (lane == 2) dst[5] = drafted && drawn ? u : 0.f;
  }
}

// stats != nullptr: the request's L row statistics were published (rstat layout) and staged
// into shared memory already; otherwise they are computed here.
// zc (with stats): the target logit of every candidate in its verifying row, [P][16], and
// path_pidx [P] the path's candidate index at each position; then no target logit is read
// from Z here except the redraw's chunk.
__device__ void verify_block(const TailLaunch& a, int b, const int* path_tok, VerifySmem& vs,
                             const float* prop_q = nullptr, const int* prop_cand = nullptr,
                             const int* prop_pidx = nullptr, const float* stats = nullptr,
                             const float* zc = nullptr, const int* path_pidx = nullptr) {
  const int L = a.L, P = L - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool soft = a.T > 0.f;
  const float inv_T = soft ? 1.0f / a.T : 0.f;
  const int is_bf16 = a.zdtype == 0;
  if (stats != nullptr) {
    if (threadIdx.x < L) {
      vs.rm[threadIdx.x] = stats[threadIdx.x * 8];
      vs.ry[threadIdx.x] = __float_as_int(stats[threadIdx.x * 8 + 1]);
      vs.rl[threadIdx.x] = stats[threadIdx.x * 8 + 2];
    }
  } else {
    for (int i = warp; i < L; i += blockDim.x >> 5) {
      const RowStat st = row_stat_warp(a, b * L + i);
      if (lane == 0) {
        vs.rm[i] = st.m;
        vs.ry[i] = st.i;
        vs.rl[i] = soft ? logf(st.s) : 0.f;
      }
    }
  }
  __syncthreads();
  int* out = a.out_tokens + static_cast<size_t>(b) * L;
  if (warp == 0) {
    bool ok = false;
    if (lane < P) {
      const int x = path_tok[lane];  // the proposal for position lane + 1, verified by row lane
      if (!soft) {
        ok = x == vs.ry[lane];
      } else {
        const bool in_vocab = x >= 0 && x < a.V;  // an out-of-vocabulary proposal has p = 0
        const float z = zc != nullptr ? zc[lane * kK + path_pidx[lane]]  // -inf outside V
                                      : in_vocab ? load1(a.Z, is_bf16, (static_cast<size_t>(b) * L + lane) * a.V + x)
                                                 : -INFINITY;
        vs.zx[lane] = z;
        const float p = expf((z - vs.rm[lane]) * inv_T - vs.rl[lane]);
        const float qx = prop_q ? prop_q[lane * kK + prop_pidx[lane]] : 1.0f;
        const float ua = stats != nullptr ? stats[lane * 8 + 3] : uniform_accept(a.seed, b, lane + 1);
        ok = ua < p / qx;
      }
    }
    if (soft && lane < L) vs.ur[lane] = stats != nullptr ? stats[lane * 8 + 4] : uniform_redraw(a.seed, b, lane + 1);
    const unsigned fail = __ballot_sync(0xffffffffu, lane < P && !ok);
    const int n = fail ? __ffs(fail) - 1 : P;  // accepted drafts
    if (lane < L && (lane != n || !soft))
      out[lane] = lane < n ? path_tok[lane] : (lane == n ? vs.ry[n] : -1);
    if (lane == 0) {
      a.accept_len[b] = n + 1;
      vs.info[0] = n;
    }
  }
  if (!soft) return;
  __syncthreads();
  // redraw from row n (the rejected position's row, or the bonus row L-1 when n = P), with
  // the rejected proposal removed; the draw's counter position is n + 1
  const int n = vs.info[0];
  const bool sampled = prop_q != nullptr && n < P;  // residual against a sampled proposal
  const int excl = (n < P && !sampled) ? path_tok[n] : -1;
  const size_t grow = static_cast<size_t>(b) * L + n;
  if (warp == 0) {
    const float M = vs.rm[n];
    const bool ex_in = excl >= 0 && excl < a.V;
    const float ex_mass = ex_in ? expf((vs.zx[n] - M) * inv_T) : 0.f;
    // sampled: mass each candidate takes out of its chunk, min(p, q) on the chunk scale
    // (unnormalised exp((z - M)/T), whose row total is exp(rl)); lane k holds candidate k
    int ck = -1;
    float take = 0.f, cfac = 0.f;
    if (sampled && lane < kK) {
      ck = prop_cand[n * kK + lane];
      const float qk = prop_q[n * kK + lane];
      if (ck >= 0 && ck < a.V) {
        const float zk = zc != nullptr ? zc[n * kK + lane] : load1(a.Z, is_bf16, grow * a.V + ck);
        const float pk = expf((zk - M) * inv_T - vs.rl[n]);
        take = fminf(pk, qk) * expf(vs.rl[n]);
        cfac = qk < pk ? 1.f - qk / pk : 0.f;
      } else {
        ck = -1;  // an id outside the vocabulary carries no target mass
      }
      vs.cand[lane] = ck;
      vs.cfac[lane] = cfac;
      vs.take[lane] = take;
    }
    __syncwarp();
    // chunk masses, lane-parallel; the cumulative sum by warp scans in chunk order (its last
    // value is the total, so the pick below always finds a chunk when target < total)
    const int exc = ex_in ? excl / kZChunk : -1;
    float run = 0.f;
    int last_nonzero = 0;
    for (int c0 = 0; c0 < a.nchunk; c0 += 32) {
      const int c = c0 + lane;
      float m = 0.f;
      if (c < a.nchunk) {
        const size_t o = grow * a.nchunk + c;
        m = __ldcg(a.zsum + o) * expf((__ldcg(a.zmax + o) - M) * inv_T);
        if (c == exc) m = fmaxf(m - ex_mass, 0.f);
        if (sampled) {  // the candidates' mass, removed in candidate order
          bool hit = false;
          for (int k = 0; k < kK; ++k)
            if (vs.cand[k] >= 0 && vs.cand[k] / kZChunk == c) {
              m -= vs.take[k];
              hit = true;
            }
          if (hit) m = fmaxf(m, 0.f);
        }
      }
      const unsigned nz = __ballot_sync(0xffffffffu, m > 0.f);
      if (nz) last_nonzero = c0 + 31 - __clz(nz);
      float cum = m;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, cum, off);
        if (lane >= off) cum += o;
      }
      cum += run;
      if (c < a.nchunk) vs.mass[c] = cum;
      run = __shfl_sync(0xffffffffu, cum, 31);
    }
    __syncwarp();
    const float target = vs.ur[n] * run;
    int pick = -1;
    for (int c0 = 0; c0 < a.nchunk && pick < 0; c0 += 32) {
      const int c = c0 + lane;
      const unsigned above = __ballot_sync(0xffffffffu, c < a.nchunk && vs.mass[c] > target);
      if (above) pick = c0 + __ffs(above) - 1;
    }
    if (lane == 0) {
      vs.info[1] = pick < 0 ? last_nonzero : pick;
      // the target's remainder past the earlier chunks, as a fraction of the chunk's mass;
      // 1 when rounding left no chunk above the target (then the chunk's last token with
      // weight is drawn, as a whole-row scan would take the row's last)
      float frac = 1.f;
      if (pick >= 0) {
        const float before = pick > 0 ? vs.mass[pick - 1] : 0.f;
        const float mc = vs.mass[pick] - before;
        frac = mc > 0.f ? fminf(fmaxf((target - before) / mc, 0.f), 1.f) : 1.f;
      }
      vs.frac = frac;
    }
  }
  __syncthreads();
  const int lo = vs.info[1] * kZChunk;
  const int hi = min(a.V, lo + kZChunk);
  if (sampled) {
    if (threadIdx.x < kZChunk / 32) vs.inchunk[threadIdx.x] = 0u;
    __syncthreads();
    if (threadIdx.x < kK) {
      const int ck = vs.cand[threadIdx.x];
      if (ck >= lo && ck < hi) atomicOr(&vs.inchunk[(ck - lo) >> 5], 1u << ((ck - lo) & 31));
    }
    __syncthreads();
  }
  // the token within the chunk by inverse CDF: weights exp((z - M)/T) (times the residual
  // factor of a sampled proposal's candidates; 0 for the excluded token), cumulated in
  // vocabulary order, against the target's place within the chunk times their total
  const int v0 = lo + threadIdx.x * 16;  // kZChunk = 16 tokens x 256 threads
  const float M = vs.rm[n];
  float w[16];
  float tsum = 0.f;
  {
    float x[2][8] = {};
    if (v0 < hi) load8(a.Z, is_bf16, grow * a.V + v0, x[0]);
    if (v0 + 8 < hi) load8(a.Z, is_bf16, grow * a.V + v0 + 8, x[1]);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int v = v0 + j;
      float wt = 0.f;
      if (v < hi && v != excl) {
        float fac = 1.f;
        if (sampled && (vs.inchunk[(v - lo) >> 5] >> ((v - lo) & 31) & 1u))
          for (int k = 0; k < kK; ++k)
            if (vs.cand[k] == v) fac = vs.cfac[k];
        wt = expf((x[j >> 3][j & 7] - M) * inv_T) * fac;
      }
      w[j] = wt;
      tsum += wt;
    }
  }
  float incl = tsum;  // inclusive scan over the warp, then over the warps
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) vs.wsum[warp] = incl;
  __syncthreads();
  float before = 0.f, total = 0.f;
#pragma unroll
  for (int i = 0; i < kTailThreads / 32; ++i) {
    if (i < warp) before += vs.wsum[i];
    total += vs.wsum[i];
  }
  const float target = vs.frac * total;
  float cum = before + incl - tsum;
  int mine = kIntMax, last = -1;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (w[j] > 0.f) {
      cum += w[j];
      last = v0 + j;
      if (mine == kIntMax && cum > target) mine = v0 + j;
    }
  mine = __reduce_min_sync(0xffffffffu, mine);
  last = __reduce_max_sync(0xffffffffu, last);
  if (lane == 0) {
    vs.wpick[warp] = mine;
    vs.wlast[warp] = last;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int pick = kIntMax, lastw = -1;
    for (int i = 0; i < kTailThreads / 32; ++i) {
      pick = min(pick, vs.wpick[i]);
      lastw = max(lastw, vs.wlast[i]);
    }
    // rounding left no token past the target: the last with weight; no weight at all: lo
    out[n] = pick != kIntMax ? pick : (lastw >= 0 ? lastw : lo);
  }
}

// ------------------------------------------------------------------ shared memory plan
struct TailSmem {
  float* lv_cur; int* li_cur;    // staged partial lists of position t   [G*16]
  float* lv_prev; int* li_prev;  // staged partial lists of position t-1 [G*16]
  float* g;                      // gate row [r]
  float* cand_U; int* cand_id;   // merged candidates of t   [16]
  float* prev_U; int* prev_id;   // merged candidates of t-1 [16]
  float* P; float* Q;            // [16][r+4]
  float* S_all; int* ids_all;    // last block: [P][16][16], [P][16]
  unsigned char* bp;             // [16][16]
  float* delta;                  // [2][16] Viterbi scores, alternating between positions
  int* path_tok;                 // [16]
  int* flag;
  VerifySmem* vs;
  float* qprop;                  // sampled traversal: [P][16] proposal distributions
  float* sdraw;                  // [P][16] score of the drawn successor of each (p, a)
  float* logb;                   // joint path draw: [P][16] backward messages (log beta)
  int* pidx;                     // [16] drawn candidate indices
  float* rstat;                  // [L][8] the request's published row statistics and uniforms
  float* zc_all;                 // [P][16] the candidates' target logits (T > 0)
  MergeSmem* ms;                 // top-16 merge scratch
  uint64_t* bar;                 // bulk-copy completion: [0] the staged lists and gate row,
                                 // [1] set 0's B rows, [2] set 1's A rows (tensor-core path)
  int* abort;                    // set when a bounded wait gave up
};

__host__ __device__ inline size_t tail_smem_bytes(int G, int r) {
  size_t n = 0;
  n += 4 * (static_cast<size_t>(G) * kK * 4 + 16);
  n += static_cast<size_t>(r) * 4 + 16;
  n += 5 * 80;
  n += 2 * (16 * static_cast<size_t>(r + 4) * 4 + 16);
  n += static_cast<size_t>(kMaxL) * kK * kK * 4 + kMaxL * kK * 4 + 32;
  n += kMaxL * kK + 16 + 144 + 80 + 16;
  n += sizeof(VerifySmem) + 16;
  n += static_cast<size_t>(kMaxL) * kK * 4 + 16 + kMaxL * 4 + 16;
  n += static_cast<size_t>(kMaxL) * kK * 4 + 16;
  n += static_cast<size_t>(kMaxL) * kK * 4 + 16;
  n += kMaxL * 32 + 16 + kMaxL * kK * 4 + 16;
  n += sizeof(MergeSmem) + 16;
  n += 48;
  return n + 256;
}

__device__ TailSmem carve(uint8_t* base, int G, int r) {
  TailSmem s;
  uint8_t* p = base;
  auto take = [&](size_t bytes) {
    uint8_t* q = p;
    p += (bytes + 15) & ~static_cast<size_t>(15);
    return q;
  };
  const size_t lb = static_cast<size_t>(G) * kK * 4;
  s.lv_cur = reinterpret_cast<float*>(take(lb));
  s.li_cur = reinterpret_cast<int*>(take(lb));
  s.lv_prev = reinterpret_cast<float*>(take(lb));
  s.li_prev = reinterpret_cast<int*>(take(lb));
  s.g = reinterpret_cast<float*>(take(static_cast<size_t>(r) * 4));
  s.cand_U = reinterpret_cast<float*>(take(64));
  s.cand_id = reinterpret_cast<int*>(take(64));
  s.prev_U = reinterpret_cast<float*>(take(64));
  s.prev_id = reinterpret_cast<int*>(take(64));
  s.P = reinterpret_cast<float*>(take(16 * static_cast<size_t>(r + 4) * 4));
  s.Q = reinterpret_cast<float*>(take(16 * static_cast<size_t>(r + 4) * 4));
  s.S_all = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxL) * kK * kK * 4));
  s.ids_all = reinterpret_cast<int*>(take(kMaxL * kK * 4));
  s.bp = take(kMaxL * kK);
  s.delta = reinterpret_cast<float*>(take(128));
  s.path_tok = reinterpret_cast<int*>(take(64));
  s.flag = reinterpret_cast<int*>(take(16));
  s.vs = reinterpret_cast<VerifySmem*>(take(sizeof(VerifySmem)));
  s.qprop = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxL) * kK * 4));
  s.pidx = reinterpret_cast<int*>(take(kMaxL * 4));
  s.sdraw = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxL) * kK * 4));
  s.logb = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxL) * kK * 4));
  s.rstat = reinterpret_cast<float*>(take(kMaxL * 32));
  s.zc_all = reinterpret_cast<float*>(take(kMaxL * kK * 4));
  s.ms = reinterpret_cast<MergeSmem*>(take(sizeof(MergeSmem)));
  s.bar = reinterpret_cast<uint64_t*>(take(32));
  s.abort = reinterpret_cast<int*>(take(16));
  return s;
}

// Set m's rows for the pair scores, by warp m: set 0's candidates' B rows (into Q), set 1's
// predecessors' A rows (into P; every one the last verified token x0 when has_prev is false).
// mma: bf16 rows by bulk copies completing on bar[1 + m]; otherwise fp32 rows, A scaled by g.
__device__ __forceinline__ void gather_set_rows(const TailLaunch& a, const TailSmem& sm, int m, bool has_prev,
                                                int x0, bool mma) {
  const int* tok = m ? (has_prev ? sm.prev_id : nullptr) : sm.cand_id;
  if (mma)
    gather_rows_bulk(a, tok, x0, m ? a.A : a.Bt, reinterpret_cast<uint16_t*>(m ? sm.P : sm.Q),
                     smem_u32(sm.bar + 1 + m));
  else
    gather_rows_warp(a, tok, x0, m == 1, m ? sm.P : sm.Q, sm.g);
}

// The 16 x 16 scores once the rows are in place (after a block barrier); every thread first
// observes the bulk copies' completion on the tensor-core path.
__device__ __forceinline__ float pair_scores(const TailLaunch& a, const TailSmem& sm, bool mma, int& pair) {
  if (!mma) return pair_dot_block(a.r, sm.P, sm.Q, sm.cand_U, pair);
  mbar_wait_bounded(smem_u32(sm.bar + 1), 0, a.err, sm.abort);
  mbar_wait_bounded(smem_u32(sm.bar + 2), 0, a.err, sm.abort);
  return pair_dot_mma(a.r, reinterpret_cast<const uint16_t*>(sm.P), reinterpret_cast<const uint16_t*>(sm.Q),
                      sm.g, sm.cand_U, sm.S_all, pair);
}

// The greedy traversal: path mode 0, and mode 2 (the sampled traversal) at T = 0.
__device__ __forceinline__ bool greedy_path(const TailLaunch& a) {
  return a.path_mode == 0 || (a.path_mode == 2 && !(a.T > 0.f));
}

// Path and verification of request b, run by the block that completes it. The scores and
// candidates of every position are read back from global memory in one round trip.
__device__ void finish_request(const TailLaunch& a, const TailSmem& sm, int b) {
  const int P = a.L - 1;
  const bool greedy = greedy_path(a);
  // the greedy traversal needs only the position blocks' successor table (in place of S_all)
  const Seg seg[4] = {
      greedy ? Seg{reinterpret_cast<const uint4*>(a.succ + static_cast<size_t>(b) * P * kK),
                   reinterpret_cast<uint4*>(sm.S_all), P * kK / 2}
             : Seg{reinterpret_cast<const uint4*>(a.S + static_cast<size_t>(b) * P * kK * kK),
                   reinterpret_cast<uint4*>(sm.S_all), P * kK * kK / 4},
      {reinterpret_cast<const uint4*>(a.cand_ids + static_cast<size_t>(b) * P * kK),
       reinterpret_cast<uint4*>(sm.ids_all), P * kK / 4},
      {reinterpret_cast<const uint4*>(a.rstat + static_cast<size_t>(b) * a.L * 8),
       reinterpret_cast<uint4*>(sm.rstat), 2 * a.L},
      // at T > 0 the candidates' target logits, published by the position blocks
      {reinterpret_cast<const uint4*>(a.zc + static_cast<size_t>(b) * P * kK),
       reinterpret_cast<uint4*>(sm.zc_all), a.T > 0.f ? P * kK / 4 : 0}};
  staged_copy<5, 4>(seg);
  __syncthreads();
  // path mode 2 at T > 0: the sampled traversal, verified against its own proposal; at
  // T = 0 it is the greedy traversal. Mode 3 at T > 0: the joint path draw (the same
  // traversal with backward messages), verified against its own conditionals; at T = 0 it
  // is Viterbi, its T -> 0 limit.
  const bool sampled = (a.path_mode == 2 || a.path_mode == 3) && a.T > 0.f;
  if (greedy) {  // (mode 2 at T = 0 included): a walk of P table lookups from predecessor 0
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      if (lane == 0) {
        const int2* succ = reinterpret_cast<const int2*>(sm.S_all);
        float total = 0.f;
        int pa = 0;
        for (int p = 0; p < P; ++p) {
          const int2 e = succ[p * kK + pa];
          total += __int_as_float(e.y);
          sm.path_tok[p] = sm.ids_all[p * kK + e.x];
          sm.pidx[p] = e.x;
          pa = e.x;
        }
        if (a.path_score) a.path_score[b] = total;
      }
      __syncwarp();
      if (lane < P) a.path[static_cast<size_t>(b) * P + lane] = sm.path_tok[lane];
      if (!(a.T > 0.f)) {
        // greedy verification, by this warp alone: draft p is accepted while it is the argmax
        // of target row p (the position blocks published the rows' statistics)
        const int ry = lane < a.L ? __float_as_int(sm.rstat[lane * 8 + 1]) : 0;
        const unsigned fail = __ballot_sync(0xffffffffu, lane < P && sm.path_tok[lane] != ry);
        const int n = fail ? __ffs(fail) - 1 : P;  // accepted drafts
        int* out = a.out_tokens + static_cast<size_t>(b) * a.L;
        if (lane < a.L) out[lane] = lane < n ? sm.path_tok[lane] : (lane == n ? ry : -1);
        if (lane == 0) a.accept_len[b] = n + 1;
      }
    }
    if (!(a.T > 0.f)) return;  // the request is done
  } else if (sampled) {
    const float inv_T = 1.0f / a.T;
    if (a.path_mode == 3) backward_messages_block(sm.S_all, P, inv_T, sm.logb);
    const float score = path_sample_block(sm.S_all, sm.ids_all, P, inv_T, sm.rstat, sm.path_tok,
                                          sm.pidx, sm.qprop, sm.sdraw, sm.bp,
                                          a.path_mode == 3 ? sm.logb : nullptr);
    if (threadIdx.x < P) a.path[static_cast<size_t>(b) * P + threadIdx.x] = sm.path_tok[threadIdx.x];
    if (threadIdx.x == 0 && a.path_score) a.path_score[b] = score;
  } else {
    const float score = path_viterbi_block(sm.S_all, sm.ids_all, P, sm.path_tok, sm.bp, sm.delta, sm.pidx);
    if (threadIdx.x < P) a.path[static_cast<size_t>(b) * P + threadIdx.x] = sm.path_tok[threadIdx.x];
    if (threadIdx.x == 0 && a.path_score) a.path_score[b] = score;
  }
  __syncthreads();
  if (sampled)
    verify_block(a, b, sm.path_tok, *sm.vs, sm.qprop, sm.ids_all, sm.pidx, sm.rstat, sm.zc_all, sm.pidx);
  else
    verify_block(a, b, sm.path_tok, *sm.vs, nullptr, nullptr, nullptr, sm.rstat, sm.zc_all, sm.pidx);
}

// ------------------------------------------------------------------ kernels
// Fused tail: block (t-1, b). Merges the candidates of positions t (and t-1), scores the
// 16 x 16 pairs of position t, and the last block of request b runs path + verification.
__global__ void __launch_bounds__(kTailThreads, 2) k_tail_fused(const __grid_constant__ TailLaunch a) {
  extern __shared__ __align__(16) uint8_t tail_smem[];
  const int t = blockIdx.x + 1, b = blockIdx.y, L = a.L, P = L - 1;
  TailSmem sm = carve(tail_smem, a.G, a.r);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int k = 0; k < 3; ++k) mbar_init(smem_u32(sm.bar + k), 1);
    *sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const bool mma = a.dtype == 0 && a.r % 16 == 0;  // tensor-core products (bf16 rows)
  // the next step's LM-head kernel (a programmatic dependent) may set up on SMs this grid
  // leaves free; it waits for this grid's completion before touching memory
  grid_dependents_launch();
  grid_dependency_wait();  // the LM-head kernel's results (launched as its dependent)
  // the gate row and the partial top-16 lists of positions t and t-1: bulk copies
  const size_t lst = static_cast<size_t>(a.G) * kK;
  const size_t rc = static_cast<size_t>(b) * L + t;
  const int nm = t >= 2 ? 2 : 1;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(sm.bar);
    const uint32_t lb = static_cast<uint32_t>(lst * 4);
    mbar_arrive_expect_tx(bar, a.r * 4 + 2 * nm * lb);
    bulk_load(smem_u32(sm.g), a.gate + rc * a.r, a.r * 4, bar);
    bulk_load(smem_u32(sm.lv_cur), a.part_val + rc * lst, lb, bar);
    bulk_load(smem_u32(sm.li_cur), a.part_idx + rc * lst, lb, bar);
    if (nm == 2) {
      bulk_load(smem_u32(sm.lv_prev), a.part_val + (rc - 1) * lst, lb, bar);
      bulk_load(smem_u32(sm.li_prev), a.part_idx + (rc - 1) * lst, lb, bar);
    }
  }
  if (warp < 4) {
    // set 0 (warps 0 and 2): the candidates of position t, then warp 0 gathers their B rows;
    // set 1 (warps 1 and 3): the candidates of position t-1 (the predecessors), then warp 1
    // gathers their A rows scaled by the gate (at position 1 the predecessor is the last
    // verified token). The group heads are ranked from L2 while the bulk copies land.
    const int m = warp & 1;
    if (m < nm)
      merge_rank_groups(a.part_val + (rc - m) * lst, a.part_idx + (rc - m) * lst, m, warp >> 1, a.G, *sm.ms);
    // a wait that runs out leaves the error word set; the block runs on (every later index
    // is bounds-checked) and the host reads DFS_ERR_TIMEOUT
    mbar_wait_bounded(smem_u32(sm.bar), 0, a.err, sm.abort);
    if (warp < 2) {
      int c = 0;
      if (m < nm)
        c = merge_candidates_warp(m ? sm.lv_prev : sm.lv_cur, m ? sm.li_prev : sm.li_cur, m, a.G, *sm.ms,
                                  m ? sm.prev_U : sm.cand_U, m ? sm.prev_id : sm.cand_id);
      if ((threadIdx.x & 31) == 0) sm.ms->ncand[m] = c;
      if (c <= kCandMax) gather_set_rows(a, sm, m, t >= 2, a.x0[b], mma);
    }
    bar_sync_warps0to3();
    const bool over0 = sm.ms->ncand[0] > kCandMax, over1 = sm.ms->ncand[1] > kCandMax;
    if (over0 || over1) {  // too many candidates: the exact merge, then those rows
      merge_exact(sm.lv_cur, sm.li_cur, sm.lv_prev, sm.li_prev, nm, a.G, *sm.ms, sm.cand_U,
                  sm.cand_id, sm.prev_U, sm.prev_id, over0, over1);
      if (warp == 0 && over0) gather_set_rows(a, sm, 0, true, 0, mma);
      if (warp == 1 && over1) gather_set_rows(a, sm, 1, true, 0, mma);
    }
  } else {
    // meanwhile, warps 6 and 7: the statistics of target row t-1 (and of the bonus row L-1
    // for the last position), published for the request's last block
    if (warp == 6) row_stat_publish(a, b * L + t - 1, a.rstat + (static_cast<size_t>(b) * L + t - 1) * 8);
    if (warp == 7 && t == P) row_stat_publish(a, b * L + L - 1, a.rstat + (static_cast<size_t>(b) * L + L - 1) * 8);
  }
  __syncthreads();
  if (threadIdx.x < kK) {
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK + threadIdx.x;
    a.cand_ids[o] = sm.cand_id[threadIdx.x];
    a.cand_U[o] = sm.cand_U[threadIdx.x];
  }
  // at T > 0, the target logit of each candidate in row t-1 (the row that verifies position
  // t), for the last block's acceptance tests and residuals: loaded now, stored after the
  // pair scores so that the load's latency hides behind them
  const bool soft = a.T > 0.f;
  float zcand = -INFINITY;
  if (soft && warp == 5 && (threadIdx.x & 31) < kK) {
    const int c = sm.cand_id[threadIdx.x & 31];
    if (c >= 0 && c < a.V)
      zcand = load1(a.Z, a.zdtype == 0, (static_cast<size_t>(b) * L + t - 1) * a.V + c);
  }
  int pair;
  const float s = pair_scores(a, sm, mma, pair);
  a.S[(static_cast<size_t>(b) * P + (t - 1)) * kK * kK + pair] = s;
  if (soft && warp == 5 && (threadIdx.x & 31) < kK)
    a.zc[(static_cast<size_t>(b) * P + (t - 1)) * kK + (threadIdx.x & 31)] = zcand;
  if (greedy_path(a)) {
    // the greedy traversal's table for this position: each predecessor's best successor
    // (score desc, id asc; the same choice as path_greedy_warp's steps), for the last block's walk
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK;
    if (mma) {
      // pair = tid: half-warp a holds row a, lane c its pair (a, c); a shuffle argmax
      const int c = threadIdx.x & 15;
      unsigned long long bk = pack_key(s, sm.cand_id[c]);
      int bc = c;
      float bv = s;
#pragma unroll
      for (int d = 8; d > 0; d >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bk, d);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, d);
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
        if (ok > bk || (ok == bk && oc < bc)) {
          bk = ok;
          bc = oc;
          bv = ov;
        }
      }
      const float s0 = __shfl_sync(0xffffffffu, s, threadIdx.x & 16);  // the row's first pair
      if ((bk >> 32) == 0ull) {  // no candidate ranks above the empty key: the first one
        bc = 0;
        bv = s0;
      }
      if (c == 0) a.succ[o + (threadIdx.x >> 4)] = make_int2(bc, __float_as_int(bv));
    } else {
      sm.qprop[pair] = s;  // free in the position blocks
      __syncthreads();
      if (threadIdx.x < kK) {
        const float* row = sm.qprop + threadIdx.x * kK;
        unsigned long long bk = 0ull;
        int bc = 0;
#pragma unroll
        for (int c = 0; c < kK; ++c) {
          const unsigned long long k = pack_key(row[c], sm.cand_id[c]);
          if (k > bk) {
            bk = k;
            bc = c;
          }
        }
        if ((bk >> 32) == 0ull) bc = 0;
        a.succ[o + threadIdx.x] = make_int2(bc, __float_as_int(row[bc]));
      }
    }
  }
  // hand-off: the block's writes (candidates, pair scores, row statistics) are ordered before
  // thread 0's device-scope release by the barrier; the last block's acquire, then its
  // barrier, orders the other blocks' writes before its reads
  __syncthreads();
  if (threadIdx.x == 0) *sm.flag = (atomic_add_acq_rel_gpu(a.counters + b, 1) == P - 1);
  __syncthreads();
  if (!*sm.flag) return;
  finish_request(a, sm, b);
  if (threadIdx.x == 0) a.counters[b] = 0;
}

// Decode-loop hand-off: the last token request b emitted becomes the next cycle's last
// verified token (-1 for an accept length outside 1..L).
__global__ void k_next_tokens(int B, int L, const int32_t* __restrict__ out_tokens,
                              const int32_t* __restrict__ accept_len, int32_t* __restrict__ next) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = accept_len[b];
  next[b] = (n >= 1 && n <= L) ? out_tokens[static_cast<size_t>(b) * L + n - 1] : -1;
}

// dfs_lmhead_topk: block (t-1, b) merges the partial lists of draft row t.
__global__ void __launch_bounds__(kTailThreads) k_merge(const __grid_constant__ TailLaunch a) {
  extern __shared__ __align__(16) uint8_t tail_smem[];
  const int t = blockIdx.x + 1, b = blockIdx.y, P = a.L - 1;
  TailSmem sm = carve(tail_smem, a.G, a.r);
  const size_t lst = static_cast<size_t>(a.G) * kK;
  const size_t rc = static_cast<size_t>(b) * a.L + t;
  const Seg seg[2] = {
      {reinterpret_cast<const uint4*>(a.part_val + rc * lst), reinterpret_cast<uint4*>(sm.lv_cur), a.G * kK / 4},
      {reinterpret_cast<const uint4*>(a.part_idx + rc * lst), reinterpret_cast<uint4*>(sm.li_cur), a.G * kK / 4}};
  staged_copy<8, 2>(seg);
  __syncthreads();
  if (threadIdx.x < 128) {
    const int warp = threadIdx.x >> 5;
    if (warp == 0 || warp == 2)
      merge_rank_groups(a.part_val + rc * lst, a.part_idx + rc * lst, 0, warp >> 1, a.G, *sm.ms);
    if (warp == 0) {
      const int c = merge_candidates_warp(sm.lv_cur, sm.li_cur, 0, a.G, *sm.ms, sm.cand_U, sm.cand_id);
      if (threadIdx.x == 0) sm.ms->ncand[0] = c;
    }
    bar_sync_warps0to3();
    if (sm.ms->ncand[0] > kCandMax)
      merge_exact(sm.lv_cur, sm.li_cur, nullptr, nullptr, 1, a.G, *sm.ms, sm.cand_U, sm.cand_id,
                  nullptr, nullptr, true, false);
  }
  __syncthreads();
  if (threadIdx.x < kK) {
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK + threadIdx.x;
    a.cand_ids[o] = sm.cand_id[threadIdx.x];
    a.cand_U[o] = sm.cand_U[threadIdx.x];
  }
}

// dfs_pair_score: block (t-1, b) scores position t from the given candidate lists.
__global__ void __launch_bounds__(kTailThreads) k_pair(const __grid_constant__ TailLaunch a) {
  extern __shared__ __align__(16) uint8_t tail_smem[];
  const int t = blockIdx.x + 1, b = blockIdx.y, L = a.L, P = L - 1;
  TailSmem sm = carve(tail_smem, 1, a.r);
  const bool mma = a.dtype == 0 && a.r % 16 == 0;  // tensor-core products (bf16 rows)
  if (threadIdx.x == 0) {
    for (int k = 1; k < 3; ++k) mbar_init(smem_u32(sm.bar + k), 1);
    *sm.abort = 0;
    fence_barrier_init();
  }
  const Seg seg[1] = {{reinterpret_cast<const uint4*>(a.gate + (static_cast<size_t>(b) * L + t) * a.r),
                       reinterpret_cast<uint4*>(sm.g), a.r / 4}};
  staged_copy<1, 1>(seg);
  if (threadIdx.x < kK) {
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK + threadIdx.x;
    sm.cand_id[threadIdx.x] = a.cand_ids[o];
    sm.cand_U[threadIdx.x] = a.cand_U[o];
    sm.prev_id[threadIdx.x] = t >= 2 ? a.cand_ids[o - kK] : a.x0[b];
  }
  __syncthreads();
  if (threadIdx.x < 64) gather_set_rows(a, sm, threadIdx.x >> 5, true, 0, mma);
  __syncthreads();
  int pair;
  const float s = pair_scores(a, sm, mma, pair);
  a.S[(static_cast<size_t>(b) * P + (t - 1)) * kK * kK + pair] = s;
}

// dfs_path_select: one block per request; the block stages the scores, then one warp walks
// the greedy path, or the whole block runs Viterbi (the fused tail's code for both).
__global__ void __launch_bounds__(kTailThreads) k_path(const __grid_constant__ TailLaunch a) {
  __shared__ __align__(16) float S_all[kMaxL * kK * kK];
  __shared__ __align__(16) int ids_all[kMaxL * kK];
  __shared__ unsigned char bp[kMaxL * kK];
  __shared__ float delta[2 * kK];
  __shared__ int path_tok[kMaxL];
  const int b = blockIdx.x, P = a.L - 1;
  const Seg seg[2] = {
      {reinterpret_cast<const uint4*>(a.S + static_cast<size_t>(b) * P * kK * kK),
       reinterpret_cast<uint4*>(S_all), P * kK * kK / 4},
      {reinterpret_cast<const uint4*>(a.cand_ids + static_cast<size_t>(b) * P * kK),
       reinterpret_cast<uint4*>(ids_all), P * kK / 4}};
  staged_copy<4, 2>(seg);  // up to 15 * 68 chunks over 256 threads
  __syncthreads();
  float score;
  if (a.path_mode == 0) {
    if (threadIdx.x >= 32) return;
    score = path_greedy_warp(S_all, ids_all, P, path_tok);
  } else {
    score = path_viterbi_block(S_all, ids_all, P, path_tok, bp, delta, nullptr);
  }
  if (threadIdx.x < P) a.path[static_cast<size_t>(b) * P + threadIdx.x] = path_tok[threadIdx.x];
  if (threadIdx.x == 0 && a.path_score) a.path_score[b] = score;
}

// dfs_verify: one block per request, given its path.
__global__ void __launch_bounds__(kTailThreads) k_verify(const __grid_constant__ TailLaunch a) {
  __shared__ int path_tok[kMaxL];
  __shared__ VerifySmem vs;
  const int b = blockIdx.x, P = a.L - 1;
  if (threadIdx.x < P) path_tok[threadIdx.x] = a.path[static_cast<size_t>(b) * P + threadIdx.x];
  __syncthreads();
  verify_block(a, b, path_tok, vs);
}

// Launch as a programmatic dependent of the previous kernel on the stream: the launch is
// processed while that kernel drains; the kernel waits (griddepcontrol.wait) before it
// reads what its predecessor wrote.
template <typename K>
cudaError_t launch_dependent(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             const TailLaunch& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

// The status of a plain launch, counted when the runtime accepted it.
cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) note_launches(1);
  return e;
}

// A tail kernel may need up to tail_smem_bytes(kMaxLists, kMaxRank) of dynamic shared
// memory. The limit is raised once per kernel, on its first launch, so later launches
// (including ones recorded into a CUDA graph) make no other runtime call.
template <auto Kern>
cudaError_t allow_smem() {
  static const cudaError_t status = cudaFuncSetAttribute(
      Kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(tail_smem_bytes(kMaxLists, kMaxRank)));
  return status;
}

}  // namespace

cudaError_t launch_zreduce(const ZReduceLaunch& a, cudaStream_t s) {
  const bool strided = a.rows > 65535;
  dim3 grid(a.nchunk, strided ? 65535 : a.rows);
  auto kern = a.inv_T > 0.f ? (strided ? k_zreduce<true, true> : k_zreduce<true, false>)
                            : (strided ? k_zreduce<false, true> : k_zreduce<false, false>);
  kern<<<grid, 128, 0, s>>>(a.Z, a.zdtype == 0, a.rows, a.V, a.nchunk, a.inv_T, a.zmax, a.zarg,
                           a.zsum, a.zero_ptr, a.zero_count);
  return counted(cudaGetLastError());
}

cudaError_t launch_tail_fused(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(a.G, a.r);
  cudaError_t e = allow_smem<k_tail_fused>();
  if (e != cudaSuccess) return e;
  return launch_dependent(k_tail_fused, dim3(a.L - 1, a.B), dim3(kTailThreads), bytes, s, a);
}

cudaError_t launch_next_tokens(int B, int L, const int32_t* out_tokens, const int32_t* accept_len,
                               int32_t* next, cudaStream_t s) {
  k_next_tokens<<<(B + 255) / 256, 256, 0, s>>>(B, L, out_tokens, accept_len, next);
  return counted(cudaGetLastError());
}

cudaError_t launch_merge(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(a.G, a.r);
  cudaError_t e = allow_smem<k_merge>();
  if (e != cudaSuccess) return e;
  k_merge<<<dim3(a.L - 1, a.B), kTailThreads, bytes, s>>>(a);
  return counted(cudaGetLastError());
}

cudaError_t launch_pair(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(1, a.r);
  cudaError_t e = allow_smem<k_pair>();
  if (e != cudaSuccess) return e;
  k_pair<<<dim3(a.L - 1, a.B), kTailThreads, bytes, s>>>(a);
  return counted(cudaGetLastError());
}

cudaError_t launch_path(const TailLaunch& a, cudaStream_t s) {
  k_path<<<a.B, kTailThreads, 0, s>>>(a);
  return counted(cudaGetLastError());
}

cudaError_t launch_verify(const TailLaunch& a, cudaStream_t s) {
  k_verify<<<a.B, kTailThreads, 0, s>>>(a);
  return counted(cudaGetLastError());
}

}  // namespace dfs
