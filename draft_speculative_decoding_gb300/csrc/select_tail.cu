// select_tail.cu -- everything after the LM head: target-logit row statistics, the
// merge of partial top-16 lists, bilinear pair scores, greedy / Viterbi paths, greedy
// and rejection-sampling verification, and the Gumbel-max redraw.
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
// Memory-bound parts read with 16-byte coalesced loads; the dependent small steps
// (merge, pair scores, path) run in one block per (request, position), and the last
// block of a request to finish (an atomic counter, no spinning) selects the path and
// verifies it.
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

// ------------------------------------------------------------------ target rows
// One block of 128 threads reduces kZChunk (4096) elements of one row of Z: each thread
// holds 4 groups of 8 consecutive elements, the groups 1024 elements apart.
template <bool kSoft>
__global__ void __launch_bounds__(128) k_zreduce(const void* Z, int is_bf16, int V, int nchunk,
                                                 float inv_T, float* zmax, int* zarg, float* zsum,
                                                 int* zero_ptr, int zero_count) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && zero_ptr != nullptr)
    for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_ptr[i] = 0;
  const int row = blockIdx.y, chunk = blockIdx.x;
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
  __shared__ RowStat ws[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
}

// Merged statistics of one target row, computed by one warp.
__device__ RowStat row_stat_warp(const TailLaunch& a, int row) {
  RowStat st = rowstat_empty();
  const float inv_T = a.T > 0.f ? 1.0f / a.T : 0.f;
  for (int c = threadIdx.x & 31; c < a.nchunk; c += 32) {
    const size_t o = static_cast<size_t>(row) * a.nchunk + c;
    RowStat v{__ldcg(a.zmax + o), __ldcg(a.zarg + o), a.T > 0.f ? __ldcg(a.zsum + o) : 0.f};
    st = combine(st, v, inv_T);
  }
  return warp_combine(st, inv_T);
}

// ------------------------------------------------------------------ top-16 merge
// Copy the G partial lists (G x 16 values and ids, contiguous) of one row into shared memory.
__device__ __forceinline__ void stage_lists(const TailLaunch& a, int row, float* sv, int* si) {
  const size_t base = static_cast<size_t>(row) * a.G * kK;
  const int n4 = a.G * kK / 4;
  const float4* pv = reinterpret_cast<const float4*>(a.part_val + base);
  const int4* pi = reinterpret_cast<const int4*>(a.part_idx + base);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    reinterpret_cast<float4*>(sv)[i] = __ldcg(pv + i);
    reinterpret_cast<int4*>(si)[i] = __ldcg(pi + i);
  }
}

// One warp merges nl <= 256 sorted lists of 16 into the top 16 (value desc, id asc): a
// 16-round tournament, lane l watching the heads of lists l, l+32, ...
__device__ void merge_lists_warp(const float* sv, const int* si, int nl, float* outv, int* outi) {
  const int lane = threadIdx.x & 31;
  int head[8];
  float hv[8];
  int hi[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int l = lane + 32 * s;
    head[s] = 0;
    hv[s] = l < nl ? sv[l * kK] : -INFINITY;
    hi[s] = l < nl ? si[l * kK] : kIntMax;
  }
  for (int k = 0; k < kK; ++k) {
    float bv = -INFINITY;
    int bi = kIntMax, bs = -1;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (ranks_before(hv[s], hi[s], bv, bi)) {
        bv = hv[s];
        bi = hi[s];
        bs = s;
      }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, off);
      if (ranks_before(ov, oi, wv, wi)) {
        wv = ov;
        wi = oi;
      }
    }
    if (bs >= 0 && bi == wi && bv == wv) {
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s == bs) {
          const int l = lane + 32 * s;
          ++head[s];
          hv[s] = head[s] < kK ? sv[l * kK + head[s]] : -INFINITY;
          hi[s] = head[s] < kK ? si[l * kK + head[s]] : kIntMax;
        }
    }
    if (lane == 0) {
      outv[k] = wv;
      outi[k] = wi;
    }
  }
}

// ------------------------------------------------------------------ pair scores
struct PairSmem {
  float* P;     // [16][r+4]: A(a) (.) g_t
  float* Q;     // [16][r+4]: B(c)
  float* g;     // [r]
};

// S_t(a, c) = U_t(c) + sum_j A(a)_j g_j B(c)_j for the 16 x 16 pairs of one position.
// prev_tok[a] is the a-th predecessor token (all x0 for position 1); cur_tok/cur_U the
// position's candidates. Thread (a = tid/16, c = tid%16) returns its score.
__device__ float pair_scores_block(const TailLaunch& a, const PairSmem& sm, const int* prev_tok,
                                   const int* cur_tok, const float* cur_U, const float* gate_row) {
  const int r = a.r, rs = r + 4;
  for (int j = threadIdx.x; j < r; j += blockDim.x) sm.g[j] = __ldcg(gate_row + j);
  __syncthreads();
  const int per_row = r / 8;  // 8-element chunks per table row
  for (int idx = threadIdx.x; idx < 32 * per_row; idx += blockDim.x) {
    const int which = idx / per_row, ch = idx % per_row;
    const bool isP = which < 16;
    const int slot = isP ? which : which - 16;
    const int tok = isP ? prev_tok[slot] : cur_tok[slot];
    float x[8];
    if (tok >= 0 && tok < a.V) {
      load8(isP ? a.A : a.Bt, a.dtype == 0, static_cast<size_t>(tok) * r + ch * 8, x);
    } else {  // an id outside the vocabulary (bad input) scores as a zero embedding
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.f;
    }
    float* dst = (isP ? sm.P : sm.Q) + slot * rs + ch * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = isP ? x[j] * sm.g[ch * 8 + j] : x[j];
  }
  __syncthreads();
  const int ai = threadIdx.x >> 4, ci = threadIdx.x & 15;
  const float4* pr = reinterpret_cast<const float4*>(sm.P + ai * rs);
  const float4* qr = reinterpret_cast<const float4*>(sm.Q + ci * rs);
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  for (int j = 0; j < r / 4; ++j) {
    const float4 p = pr[j], q = qr[j];
    s0 = fmaf(p.x, q.x, s0);
    s1 = fmaf(p.y, q.y, s1);
    s2 = fmaf(p.z, q.z, s2);
    s3 = fmaf(p.w, q.w, s3);
  }
  return cur_U[ci] + ((s0 + s1) + (s2 + s3));
}

// ------------------------------------------------------------------ path
// One warp; S [P][16][16] and ids [P][16] in shared memory. Lanes 0..15 hold candidates.
// Writes path_tok[P] (shared) and returns the path score in lane 0.
__device__ float path_warp(const float* S, const int* ids, int P, int mode, int* path_tok,
                           unsigned char* bp) {
  const int lane = threadIdx.x & 31;
  const bool act = lane < kK;
  if (mode == 0) {
    // greedy: x_t = argmax_c S_t(x_{t-1}, c)
    int a = 0;
    float total = 0.f;
    for (int p = 0; p < P; ++p) {
      float v = act ? S[(p * kK + a) * kK + lane] : -INFINITY;
      int id = act ? ids[p * kK + lane] : kIntMax;
      int c = lane;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, id, off);
        const int oc = __shfl_xor_sync(0xffffffffu, c, off);
        if (ranks_before(ov, oi, v, id)) {
          v = ov;
          id = oi;
          c = oc;
        }
      }
      if (lane == 0) path_tok[p] = id;
      total += v;
      a = c;
    }
    return total;
  }
  // Viterbi: delta_1(c) = S_1(x0, c); delta_t(c) = max_a delta_{t-1}(a) + S_t(a, c)
  float delta = act ? S[lane] : -INFINITY;
  for (int p = 1; p < P; ++p) {
    float best = -INFINITY;
    int best_id = kIntMax, best_a = 0;
#pragma unroll
    for (int aa = 0; aa < kK; ++aa) {
      const float da = __shfl_sync(0xffffffffu, delta, aa);
      const float v = da + (act ? S[(p * kK + aa) * kK + lane] : 0.f);
      const int pid = ids[(p - 1) * kK + aa];
      if (ranks_before(v, pid, best, best_id)) {
        best = v;
        best_id = pid;
        best_a = aa;
      }
    }
    if (act) bp[p * kK + lane] = static_cast<unsigned char>(best_a);
    delta = act ? best : -INFINITY;
  }
  float v = delta;
  int id = act ? ids[(P - 1) * kK + lane] : kIntMax;
  int c = lane;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, id, off);
    const int oc = __shfl_xor_sync(0xffffffffu, c, off);
    if (ranks_before(ov, oi, v, id)) {
      v = ov;
      id = oi;
      c = oc;
    }
  }
  __syncwarp();
  if (lane == 0) {
    int cur = c;
    for (int p = P - 1; p >= 0; --p) {
      path_tok[p] = ids[p * kK + cur];
      if (p > 0) cur = bp[p * kK + cur];
    }
  }
  __syncwarp();
  return v;
}

// ------------------------------------------------------------------ verify
// Verification of request b given its path (shared memory). Uses every warp of the block
// for the row statistics, then thread 0 walks the positions.
__device__ void verify_block(const TailLaunch& a, int b, const int* path_tok, float* rm, float* rl,
                             int* ry) {
  const int L = a.L, P = L - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < L; i += blockDim.x >> 5) {
    const RowStat st = row_stat_warp(a, b * L + i);
    if (lane == 0) {
      rm[i] = st.m;
      ry[i] = st.i;
      rl[i] = a.T > 0.f ? logf(st.s) : 0.f;
    }
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  int* out = a.out_tokens + static_cast<size_t>(b) * L;
  if (!(a.T > 0.f)) {
    int n = 0;
    while (n < P && path_tok[n] == ry[n]) ++n;
    for (int i = 0; i < L; ++i) out[i] = i < n ? path_tok[i] : (i == n ? ry[n] : -1);
    a.accept_len[b] = n + 1;
    return;
  }
  const float inv_T = 1.0f / a.T;
  int* info = a.resample_info + static_cast<size_t>(b) * 4;
  for (int i = 0; i < L; ++i) out[i] = -1;
  for (int t = 1; t <= P; ++t) {
    const int x = path_tok[t - 1];
    const bool in_vocab = x >= 0 && x < a.V;  // an out-of-vocabulary proposal has p = 0
    const float z = in_vocab
        ? load1(a.Z, a.zdtype == 0, (static_cast<size_t>(b) * L + (t - 1)) * a.V + x) : -INFINITY;
    const float p = expf((z - rm[t - 1]) * inv_T - rl[t - 1]);
    const float u = uniform_accept(a.seed, b, t);
    if (u < p) {
      out[t - 1] = x;
      continue;
    }
    info[0] = t - 1;  // row redrawn from
    info[1] = x;      // token removed from it
    info[2] = t - 1;  // output slot
    info[3] = 1;
    a.accept_len[b] = t;
    return;
  }
  info[0] = P;
  info[1] = -1;
  info[2] = P;
  info[3] = 1;
  a.accept_len[b] = L;
}

// ------------------------------------------------------------------ shared memory plan
struct TailSmem {
  float* lv_cur; int* li_cur;    // staged partial lists of position t   [G*16]
  float* lv_prev; int* li_prev;  // staged partial lists of position t-1 [G*16]
  float* cand_U; int* cand_id;   // merged candidates of t   [16]
  float* prev_U; int* prev_id;   // merged candidates of t-1 [16]
  int* prev_tok;                 // predecessor tokens [16]
  PairSmem pair;
  float* S_all; int* ids_all;    // last block: [P][16][16], [P][16]
  unsigned char* bp;             // [16][16]
  int* path_tok;                 // [16]
  float* rm; float* rl; int* ry; // [16] row statistics
  int* flag;
};

__host__ __device__ inline size_t tail_smem_bytes(int G, int r, bool lists2) {
  size_t n = 0;
  n += static_cast<size_t>(G) * kK * 8 * (lists2 ? 2 : 1);
  n += 16 * 4 * 5;
  n += 2 * 16 * static_cast<size_t>(r + 4) * 4 + static_cast<size_t>(r) * 4;
  n += static_cast<size_t>(kMaxL) * kK * kK * 4 + kMaxL * kK * 4;
  n += kMaxL * kK + 16 * 4 * 4 + 64;
  return n + 256;
}

__device__ TailSmem carve(uint8_t* base, int G, int r, bool lists2) {
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
  if (lists2) {
    s.lv_prev = reinterpret_cast<float*>(take(lb));
    s.li_prev = reinterpret_cast<int*>(take(lb));
  } else {
    s.lv_prev = nullptr;
    s.li_prev = nullptr;
  }
  s.cand_U = reinterpret_cast<float*>(take(64));
  s.cand_id = reinterpret_cast<int*>(take(64));
  s.prev_U = reinterpret_cast<float*>(take(64));
  s.prev_id = reinterpret_cast<int*>(take(64));
  s.prev_tok = reinterpret_cast<int*>(take(64));
  s.pair.P = reinterpret_cast<float*>(take(16 * static_cast<size_t>(r + 4) * 4));
  s.pair.Q = reinterpret_cast<float*>(take(16 * static_cast<size_t>(r + 4) * 4));
  s.pair.g = reinterpret_cast<float*>(take(static_cast<size_t>(r) * 4));
  s.S_all = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxL) * kK * kK * 4));
  s.ids_all = reinterpret_cast<int*>(take(kMaxL * kK * 4));
  s.bp = take(kMaxL * kK);
  s.path_tok = reinterpret_cast<int*>(take(64));
  s.rm = reinterpret_cast<float*>(take(64));
  s.rl = reinterpret_cast<float*>(take(64));
  s.ry = reinterpret_cast<int*>(take(64));
  s.flag = reinterpret_cast<int*>(take(16));
  return s;
}

// Path and verification of request b, run by the block that completes it. S and the
// candidates of every position are read back from global memory.
__device__ void finish_request(const TailLaunch& a, const TailSmem& sm, int b) {
  const int P = a.L - 1;
  const float* Sg = a.S + static_cast<size_t>(b) * P * kK * kK;
  const int* Ig = a.cand_ids + static_cast<size_t>(b) * P * kK;
  for (int i = threadIdx.x; i < P * kK * kK; i += blockDim.x) sm.S_all[i] = __ldcg(Sg + i);
  for (int i = threadIdx.x; i < P * kK; i += blockDim.x) sm.ids_all[i] = __ldcg(Ig + i);
  __syncthreads();
  if (threadIdx.x < 32) {
    const float score = path_warp(sm.S_all, sm.ids_all, P, a.path_mode, sm.path_tok, sm.bp);
    if (threadIdx.x == 0 && a.path_score) a.path_score[b] = score;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < P; i += blockDim.x) a.path[static_cast<size_t>(b) * P + i] = sm.path_tok[i];
  verify_block(a, b, sm.path_tok, sm.rm, sm.rl, sm.ry);
}

// ------------------------------------------------------------------ kernels
// Fused tail: block (t-1, b). Merges the candidates of positions t (and t-1), scores the
// 16 x 16 pairs of position t, and the last block of request b runs path + verification.
__global__ void __launch_bounds__(kTailThreads) k_tail_fused(const __grid_constant__ TailLaunch a) {
  extern __shared__ __align__(16) uint8_t tail_smem[];
  grid_dependents_launch();  // a following redraw kernel may take free SMs and wait there
  grid_dependency_wait();    // the LM-head kernel's results (launched as its dependent)
  const int t = blockIdx.x + 1, b = blockIdx.y, L = a.L, P = L - 1;
  TailSmem sm = carve(tail_smem, a.G, a.r, true);
  const int warp = threadIdx.x >> 5;
  stage_lists(a, b * L + t, sm.lv_cur, sm.li_cur);
  if (t >= 2) stage_lists(a, b * L + t - 1, sm.lv_prev, sm.li_prev);
  __syncthreads();
  if (warp == 0) merge_lists_warp(sm.lv_cur, sm.li_cur, a.G, sm.cand_U, sm.cand_id);
  if (warp == 1 && t >= 2) merge_lists_warp(sm.lv_prev, sm.li_prev, a.G, sm.prev_U, sm.prev_id);
  __syncthreads();
  if (threadIdx.x < kK) {
    sm.prev_tok[threadIdx.x] = t >= 2 ? sm.prev_id[threadIdx.x] : a.x0[b];
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK + threadIdx.x;
    a.cand_ids[o] = sm.cand_id[threadIdx.x];
    a.cand_U[o] = sm.cand_U[threadIdx.x];
  }
  __syncthreads();
  const float s = pair_scores_block(a, sm.pair, sm.prev_tok, sm.cand_id, sm.cand_U,
                                    a.gate + static_cast<size_t>(b * L + t) * a.r);
  a.S[(static_cast<size_t>(b) * P + (t - 1)) * kK * kK + threadIdx.x] = s;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *sm.flag = (atomicAdd(a.counters + b, 1) == P - 1);
  __syncthreads();
  if (!*sm.flag) return;
  __threadfence();
  finish_request(a, sm, b);
  if (threadIdx.x == 0) a.counters[b] = 0;
}

// dfs_lmhead_topk: block (t-1, b) merges the partial lists of draft row t.
__global__ void __launch_bounds__(kTailThreads) k_merge(const __grid_constant__ TailLaunch a) {
  extern __shared__ __align__(16) uint8_t tail_smem[];
  const int t = blockIdx.x + 1, b = blockIdx.y, P = a.L - 1;
  TailSmem sm = carve(tail_smem, a.G, a.r, false);
  stage_lists(a, b * a.L + t, sm.lv_cur, sm.li_cur);
  __syncthreads();
  if (threadIdx.x < 32) merge_lists_warp(sm.lv_cur, sm.li_cur, a.G, sm.cand_U, sm.cand_id);
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
  TailSmem sm = carve(tail_smem, 1, a.r, false);
  if (threadIdx.x < kK) {
    const size_t o = (static_cast<size_t>(b) * P + (t - 1)) * kK + threadIdx.x;
    sm.cand_id[threadIdx.x] = a.cand_ids[o];
    sm.cand_U[threadIdx.x] = a.cand_U[o];
    sm.prev_tok[threadIdx.x] = t >= 2 ? a.cand_ids[o - kK] : a.x0[b];
  }
  __syncthreads();
  const float s = pair_scores_block(a, sm.pair, sm.prev_tok, sm.cand_id, sm.cand_U,
                                    a.gate + static_cast<size_t>(b * L + t) * a.r);
  a.S[(static_cast<size_t>(b) * P + (t - 1)) * kK * kK + threadIdx.x] = s;
}

// dfs_path_select: one warp per request.
__global__ void __launch_bounds__(32) k_path(const __grid_constant__ TailLaunch a) {
  __shared__ float S_all[kMaxL * kK * kK];
  __shared__ int ids_all[kMaxL * kK];
  __shared__ unsigned char bp[kMaxL * kK];
  __shared__ int path_tok[kMaxL];
  const int b = blockIdx.x, P = a.L - 1;
  const float* Sg = a.S + static_cast<size_t>(b) * P * kK * kK;
  const int* Ig = a.cand_ids + static_cast<size_t>(b) * P * kK;
  for (int i = threadIdx.x; i < P * kK * kK; i += 32) S_all[i] = Sg[i];
  for (int i = threadIdx.x; i < P * kK; i += 32) ids_all[i] = Ig[i];
  __syncwarp();
  const float score = path_warp(S_all, ids_all, P, a.path_mode, path_tok, bp);
  __syncwarp();
  for (int i = threadIdx.x; i < P; i += 32) a.path[static_cast<size_t>(b) * P + i] = path_tok[i];
  if (threadIdx.x == 0 && a.path_score) a.path_score[b] = score;
}

// dfs_verify: one block per request, given its path.
__global__ void __launch_bounds__(kTailThreads) k_verify(const __grid_constant__ TailLaunch a) {
  __shared__ int path_tok[kMaxL];
  __shared__ float rm[kMaxL], rl[kMaxL];
  __shared__ int ry[kMaxL];
  const int b = blockIdx.x, P = a.L - 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) path_tok[i] = a.path[static_cast<size_t>(b) * P + i];
  __syncthreads();
  verify_block(a, b, path_tok, rm, rl, ry);
}

// Gumbel-max redraw for T > 0: block (chunk, b) scans kRChunk tokens of the row named in
// resample_info[b]; the last block of the request merges the per-chunk winners.
__global__ void __launch_bounds__(256) k_resample(const __grid_constant__ TailLaunch a) {
  grid_dependency_wait();  // the verification kernel's redraw requests
  const int b = blockIdx.y, chunk = blockIdx.x, L = a.L;
  const int* info = a.resample_info + static_cast<size_t>(b) * 4;
  const int row = __ldcg(info), excl = __ldcg(info + 1), slot = __ldcg(info + 2);
  const float inv_T = 1.0f / a.T;
  const size_t rbase = (static_cast<size_t>(b) * L + row) * a.V;
  float bk = -INFINITY;
  int bi = kIntMax;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int v0 = chunk * kRChunk + g * 2048 + threadIdx.x * 8;
    if (v0 >= a.V) continue;
    float x[8];
    load8(a.Z, a.zdtype == 0, rbase + v0, x);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int vq = v0 + 4 * h;
      uint64_t c[4] = {static_cast<uint64_t>(vq >> 2), static_cast<uint64_t>(row + 1),
                       static_cast<uint64_t>(b), 1ull};
      philox4x64_10(c, a.seed, 0ull);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int v = vq + w;
        const float gmb = -logf(-logf(u01_from_word(c[w])));
        const float key = x[4 * h + w] * inv_T + gmb;
        if (v != excl && key > bk) {  // v increases within the thread
          bk = key;
          bi = v;
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (ranks_before(ok, oi, bk, bi)) {
      bk = ok;
      bi = oi;
    }
  }
  __shared__ float sk[8];
  __shared__ int si[8];
  __shared__ int last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sk[warp] = bk;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w)
      if (ranks_before(sk[w], si[w], bk, bi)) {
        bk = sk[w];
        bi = si[w];
      }
    a.gumbel_key[static_cast<size_t>(b) * a.nrchunk + chunk] = bk;
    a.gumbel_idx[static_cast<size_t>(b) * a.nrchunk + chunk] = bi;
    __threadfence();
    last = (atomicAdd(a.resample_counters + b, 1) == a.nrchunk - 1);
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  float fk = -INFINITY;
  int fi = kIntMax;
  for (int c = 0; c < a.nrchunk; ++c) {
    const float k = __ldcg(a.gumbel_key + static_cast<size_t>(b) * a.nrchunk + c);
    const int i = __ldcg(a.gumbel_idx + static_cast<size_t>(b) * a.nrchunk + c);
    if (ranks_before(k, i, fk, fi)) {
      fk = k;
      fi = i;
    }
  }
  a.out_tokens[static_cast<size_t>(b) * L + slot] = fi;
  a.resample_counters[b] = 0;
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

}  // namespace

cudaError_t launch_zreduce(const ZReduceLaunch& a, cudaStream_t s) {
  dim3 grid(a.nchunk, a.rows);
  if (a.inv_T > 0.f)
    k_zreduce<true><<<grid, 128, 0, s>>>(a.Z, a.zdtype == 0, a.V, a.nchunk, a.inv_T, a.zmax,
                                         a.zarg, a.zsum, a.zero_ptr, a.zero_count);
  else
    k_zreduce<false><<<grid, 128, 0, s>>>(a.Z, a.zdtype == 0, a.V, a.nchunk, 0.f, a.zmax,
                                          a.zarg, a.zsum, a.zero_ptr, a.zero_count);
  return cudaGetLastError();
}

cudaError_t launch_tail_fused(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(a.G, a.r, true);
  cudaError_t e = set_smem(k_tail_fused, bytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(k_tail_fused, dim3(a.L - 1, a.B), dim3(kTailThreads), bytes, s, a);
}

cudaError_t launch_merge(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(a.G, a.r, false);
  cudaError_t e = set_smem(k_merge, bytes);
  if (e != cudaSuccess) return e;
  k_merge<<<dim3(a.L - 1, a.B), kTailThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_pair(const TailLaunch& a, cudaStream_t s) {
  const size_t bytes = tail_smem_bytes(1, a.r, false);
  cudaError_t e = set_smem(k_pair, bytes);
  if (e != cudaSuccess) return e;
  k_pair<<<dim3(a.L - 1, a.B), kTailThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_path(const TailLaunch& a, cudaStream_t s) {
  k_path<<<a.B, 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_verify(const TailLaunch& a, cudaStream_t s) {
  k_verify<<<a.B, kTailThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_resample(const TailLaunch& a, cudaStream_t s) {
  return launch_dependent(k_resample, dim3(a.nrchunk, a.B), dim3(256), 0, s, a);
}

}  // namespace dfs
