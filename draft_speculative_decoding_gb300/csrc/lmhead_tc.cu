// lmhead_tc.cu -- the drafter's shared LM head with a fused keep-top-16 epilogue
// (and the context gate as extra tiles), on the sm_103a tensor cores.
//
// Sources: "DFlash 2: Keep Drafting Parallel", sections "The right tokens are
// already there" (keep the 16 best candidates per position) and "A lightweight
// path selector" (U_t(b) is the drafter's own logit; a context gate H(h_t) is
// computed from the position's hidden state).
//
// Shape of the work: logits[m, v] = sum_k h[m, k] W[k, v] for the m <= 256 block rows
// of one row group and every v of the vocabulary, then per row the 16 largest
// (logit, id) pairs. The logits never leave the SM.
//
// Design (both kernels persistent, one CTA per SM, warp-specialised):
//   * a TMA producer thread streams W_vocab (the MN-major B operand, vocabulary contiguous,
//     64x64 boxes, 128-byte swizzle, evict-first) and the hidden rows (the K-major A operand,
//     L2-resident, evict-last) through rings of shared memory guarded by mbarriers;
//   * one thread issues tcgen05.mma (bf16 in, fp32 accumulate, K = 16 per instruction) into
//     two TMEM accumulators, so the epilogue of one tile overlaps the MMAs of the next;
//   * four epilogue warps drain TMEM with tcgen05.ld, one row per thread, keeping the row's
//     running top-16 in registers (sorted, so the entry threshold is the last member); a
//     32-column chunk is first tested by its maximum, then only the lane's candidates are
//     inserted; at the end each thread writes its sorted list as one partial list of its row
//     (the tail kernel merges the partial lists of a row);
//   * gate tiles use W_g [r, d] (K-major) as the B operand; their epilogue applies the sigmoid
//     and stores g[m, j] in fp32;
//   * four more warps stream the target logits (16-byte loads, read once, a whole 4096-token
//     chunk per warp in flight) and write per-chunk row statistics (max, argmax, sum of exp)
//     for verification, so those bytes move while the tensor pipe works on W.
// k_lmhead_tc serves row groups of up to 128 rows (M = 128 x N = 256 per CTA, each CTA loading
// its own hidden-row and W boxes). k_lmhead_pair serves 129..256 rows with pair MMAs
// (cta_group::2, M = 256 x N = 256 across two SMs): each CTA stages only half of the W tile,
// which halves the shared-memory bytes per MMA -- at 256 rows the tensor pipe must run near
// full rate alongside the HBM stream, and shared-memory bandwidth, not HBM, was the limit.
// k_lmhead_vt is the pair kernel with vocabulary on M and only the drafted rows on N, for
// calls where that saves whole passes over W.
// Every mbarrier wait is bounded; on expiry the kernel sets the error word, stops all
// roles, and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_fp8.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "rowstat.cuh"

namespace dfs {

static_assert(kZChunk == 16 * 256, "zchunk_stat_warp covers a chunk as 16 loads x 32 lanes x 8");

struct LmheadParams {
  CUtensorMap tm_hq;  // E4M3 head: quantised rows [rows_total, d] bytes, box 128 x 128
  CUtensorMap tm_h;  // hidden [rows_total, d], box 64 (k) x 128 (rows)
  CUtensorMap tm_w;  // W_vocab [d, V], box 64 (vocab) x 64 (k)
  CUtensorMap tm_g;  // W_g [r, d], box 64 (k) x NT (rows of W_g)
  int row0, rows, L, V, d, r;
  int n_vocab_tiles, n_gate_tiles;
  int G;
  int write_partials;
  float* part_val;
  int* part_idx;
  float* gate_out;
  int* err;
  const void* Z;
  int zdtype, z_rows, z_nchunk;
  float z_inv_T;
  float* zmax;
  int* zarg;
  float* zsum;
  int* zero_ptr;
  int zero_count;
  unsigned long long wait_limit_ns;  // every bounded wait gives up after this long
  int stall_mma;                     // test hook: the MMA issuer stays idle
  const float* w_scale;              // E4M3 head: per-vocabulary scale [V]
  const float* h_scale;              // E4M3 head: per-row scale [rows_total]
  uint32_t h_box_bytes;              // bytes one hidden-row box delivers (k_lmhead_tc, MT = 1)
  // k_lmhead_vt: the drafted rows of requests b0 .. b0 + 2 nb - 1 (nb per CTA of a pair)
  CUtensorMap tm_h3;     // hidden as [B][L][d], box 64 (k) x (L - 1) (positions 1..) x nb
  int b0, nb, n_req;     // first request of the group, requests per CTA, requests in total
  uint32_t stage_bytes;  // one ring stage: 128 A rows + the group's drafted rows, 64 k each
};

template <int MT, int NT, int NBUF, int SW, int SH>
struct LmCfg {
  static constexpr int kWBytes = NT * 128;        // NT columns x 64 bf16 (or NT gate rows)
  static constexpr int kHBytes = MT * 128 * 128;  // MT tiles of 128 rows x 64 bf16
  static constexpr int kAccCols = MT * NT;        // fp32 TMEM columns per accumulator set
  static constexpr int kTmemCols = (kAccCols * NBUF <= 32)    ? 32
                                   : (kAccCols * NBUF <= 64)  ? 64
                                   : (kAccCols * NBUF <= 128) ? 128
                                   : (kAccCols * NBUF <= 256) ? 256
                                                              : 512;
  static constexpr int kEpiWarps = 4 * MT;
  static constexpr int kZWarps = 4;                // warp 3 and the last three
  static constexpr int kThreads = 32 * (4 + kEpiWarps + kZWarps - 1);
  static constexpr int kBarBytes = 8 * (2 * SW + 2 * SH + 2 * NBUF) + 16;
  static constexpr size_t kSmem =
      1024 + size_t(SW) * kWBytes + size_t(SH) * kHBytes + kBarBytes;
  static_assert(kAccCols * NBUF <= 512, "TMEM holds 512 fp32 columns");
  static_assert(NT % 64 == 0 && NT >= 64 && NT <= 256, "N tile");
  static_assert(kSmem <= 232448, "shared memory");
};

// A row's running top-16, kept sorted by (value desc, id asc); v[15] is the entry threshold.
// A thread offers the columns of its row in increasing id order (tiles in increasing order,
// columns increasing within a tile), so a newcomer ranks after every member of equal value:
// it enters only when it beats v[15] strictly, and goes after the members >= it.
struct Top16 {
  float v[kK];
  int i[kK];
};

__device__ __forceinline__ void top16_init(Top16& t) {
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    t.v[k] = -INFINITY;
    t.i[k] = 0x7fffffff;
  }
}

// Insert (x, id) (caller checked x > t.v[15]): the members >= x keep their slots, the rest
// shift down one. Every output slot depends only on two comparisons, so the 16 updates
// issue independently instead of as a chain.
__device__ __forceinline__ void top16_insert(Top16& t, float x, int id) {
  bool ge[kK];
#pragma unroll
  for (int k = 0; k < kK; ++k) ge[k] = t.v[k] >= x;
#pragma unroll
  for (int k = kK - 1; k >= 1; --k) {
    t.v[k] = ge[k] ? t.v[k] : (ge[k - 1] ? x : t.v[k - 1]);
    t.i[k] = ge[k] ? t.i[k] : (ge[k - 1] ? id : t.i[k - 1]);
  }
  t.v[0] = ge[0] ? t.v[0] : x;
  t.i[0] = ge[0] ? t.i[0] : id;
}

// r[j] for a run-time j in 0..31 by a five-level select tree (keeps r in registers).
__device__ __forceinline__ uint32_t pick32(const uint32_t (&r)[32], int j) {
  uint32_t a[16], b[8], c[4], d[2];
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = (j & 16) ? r[k + 16] : r[k];
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = (j & 8) ? a[k + 8] : a[k];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = (j & 4) ? b[k + 4] : b[k];
#pragma unroll
  for (int k = 0; k < 2; ++k) d[k] = (j & 2) ? c[k + 2] : c[k];
  return (j & 1) ? d[1] : d[0];
}

// Offer 32 consecutive logits (ids cbase..cbase+31, those at or past lim ignored): a
// tree maximum against the threshold first, then only the lane's candidates, lowest id
// first.
__device__ __forceinline__ void top16_offer32(Top16& t, const uint32_t (&r)[32], int cbase, int lim) {
  float m[16];
  if (lim >= 32) {
#pragma unroll
    for (int k = 0; k < 16; ++k) m[k] = fmaxf(__uint_as_float(r[k]), __uint_as_float(r[k + 16]));
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k)
      m[k] = fmaxf(k < lim ? __uint_as_float(r[k]) : -INFINITY,
                   k + 16 < lim ? __uint_as_float(r[k + 16]) : -INFINITY);
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int k = 0; k < w; ++k) m[k] = fmaxf(m[k], m[k + w]);
  const float thr = t.v[kK - 1];
  if (!(m[0] > thr)) return;
  uint32_t mask = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    mask |= (j < lim && __uint_as_float(r[j]) > thr) ? (1u << j) : 0u;
  while (mask) {
    const int j = __ffs(mask) - 1;
    mask &= mask - 1;
    const float x = __uint_as_float(pick32(r, j));
    if (x > t.v[kK - 1]) top16_insert(t, x, cbase + j);
  }
}

// sigmoid of 32 gate pre-activations (columns cbase.. of row `dst`), 16-byte stores; r is a
// multiple of 8, so each group of 4 is wholly inside or outside the r columns.
__device__ __forceinline__ void store_gate32(float* dst, const uint32_t (&r)[32], int cbase,
                                             int r_cols) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    if (cbase + j < r_cols) {
      float4 g;
      g.x = 1.0f / (1.0f + expf(-__uint_as_float(r[j])));
      g.y = 1.0f / (1.0f + expf(-__uint_as_float(r[j + 1])));
      g.z = 1.0f / (1.0f + expf(-__uint_as_float(r[j + 2])));
      g.w = 1.0f / (1.0f + expf(-__uint_as_float(r[j + 3])));
      *reinterpret_cast<float4*>(dst + cbase + j) = g;
    }
  }
}

template <int MT, int NT, int NBUF, int SW, int SH>
__global__ void __launch_bounds__(LmCfg<MT, NT, NBUF, SW, SH>::kThreads, 1)
    k_lmhead_tc(const __grid_constant__ LmheadParams p) {
  using Cfg = LmCfg<MT, NT, NBUF, SW, SH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* wring = smem;
  uint8_t* hring = smem + size_t(SW) * Cfg::kWBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(hring + size_t(SH) * Cfg::kHBytes);
  uint64_t* wfull = bars;
  uint64_t* wempty = bars + SW;
  uint64_t* hfull = bars + 2 * SW;
  uint64_t* hempty = bars + 2 * SW + SH;
  uint64_t* tfull = bars + 2 * SW + 2 * SH;
  uint64_t* tempty = tfull + NBUF;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + NBUF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(smem_u32(&wfull[s]), 1);
      mbar_init(smem_u32(&wempty[s]), 1);
    }
    for (int s = 0; s < SH; ++s) {
      mbar_init(smem_u32(&hfull[s]), 1);
      mbar_init(smem_u32(&hempty[s]), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), Cfg::kEpiWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&p.tm_h);
    prefetch_tensormap(&p.tm_w);
    prefetch_tensormap(&p.tm_g);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (MT == 1 && p.h_box_bytes < static_cast<uint32_t>(Cfg::kHBytes)) {
    // Fewer hidden rows than a tile: the boxes fill only the first rows of each stage, so the
    // rest is zeroed once (the MMA reads 128 rows; the epilogue skips the padding rows).
    uint4* hz = reinterpret_cast<uint4*>(hring);
    for (int i = threadIdx.x; i < SH * Cfg::kHBytes / 16; i += blockDim.x) hz[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // generic writes made visible to the tensor cores' reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Launched as a programmatic dependent: the set-up above overlaps the previous kernel on
  // the stream; nothing below touches global memory before that kernel has completed.
  grid_dependency_wait();
  // Every CTA of this persistent grid is resident now: let the dependent tail kernel launch
  // onto SMs as they free up (it waits for this grid's completion before reading).
  grid_dependents_launch();

  // Tiles: vocabulary tiles, then gate tiles; CTA c takes tiles c, c + grid, c + 2 grid, ...
  const int n_tiles = p.n_vocab_tiles + p.n_gate_tiles;
  const int KB = p.d / 64;
  const int first_z_extra = 4 + Cfg::kEpiWarps;  // warps first_z_extra.. are Z warps 1..3

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- TMA producer: W_vocab / W_g
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        const bool is_vocab = tile < p.n_vocab_tiles;
        const int n0 = (is_vocab ? tile : tile - p.n_vocab_tiles) * NT;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wempty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&wfull[stage]);
          mbar_arrive_expect_tx(fb, Cfg::kWBytes);
          const uint32_t sb = smem_u32(wring + size_t(stage) * Cfg::kWBytes);
          if (is_vocab) {
#pragma unroll
            for (int c = 0; c < NT / 64; ++c)
              tma_load_2d(sb + c * 8192, &p.tm_w, fb, n0 + c * 64, kb * 64, pol_stream);
          } else {
            tma_load_2d(sb, &p.tm_g, fb, kb * 64, n0, pol_keep);
          }
          if (++stage == SW) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------- TMA producer: hidden rows
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&hempty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&hfull[stage]);
          mbar_arrive_expect_tx(fb, MT == 1 ? p.h_box_bytes : static_cast<uint32_t>(Cfg::kHBytes));
          const uint32_t sa = smem_u32(hring + size_t(stage) * Cfg::kHBytes);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            tma_load_2d(sa + mt * 16384, &p.tm_h, fb, kb * 64, p.row0 + mt * 128, pol_keep);
          if (++stage == SH) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !p.stall_mma) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescVocab = idesc_bf16_f32(NT, true);
      constexpr uint32_t kIdescGate = idesc_bf16_f32(NT, false);
      int ws = 0, hs = 0;
      uint32_t wph = 0, hph = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        const bool is_vocab = tile < p.n_vocab_tiles;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wfull[ws]), wph, p.err, abort_flag, p.wait_limit_ns) ||
              !mbar_wait_bounded(smem_u32(&hfull[hs]), hph, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = smem_u32(wring + size_t(ws) * Cfg::kWBytes);
          const uint32_t sa = smem_u32(hring + size_t(hs) * Cfg::kHBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K = 16 per instruction: +32 B inside a K-major 128-byte row, or +16 rows
            // (2 x 1024-byte swizzle atoms) of an MN-major operand.
            const uint64_t bdesc = is_vocab ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                            : smem_desc_sw128(sb + kk * 32, 0, 1024);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint64_t adesc = smem_desc_sw128(sa + mt * 16384 + kk * 32, 0, 1024);
              tc_mma_bf16(d0 + mt * NT, adesc, bdesc, is_vocab ? kIdescVocab : kIdescGate,
                          (kb | kk) != 0);
            }
          }
          tc_commit(smem_u32(&wempty[ws]));
          tc_commit(smem_u32(&hempty[hs]));
          if (++ws == SW) {
            ws = 0;
            wph ^= 1;
          }
          if (++hs == SH) {
            hs = 0;
            hph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[acc]));
        if (++acc == NBUF) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else if (warp == 3 || warp >= first_z_extra) {
    // ------------------------------------------------ target-logit row statistics
    const int zw = warp == 3 ? 0 : warp - first_z_extra + 1;
    if (blockIdx.x == 0 && p.zero_ptr != nullptr)
      for (int i = zw * 32 + lane; i < p.zero_count; i += 32 * Cfg::kZWarps) p.zero_ptr[i] = 0;
    const int n_units = p.z_rows * p.z_nchunk;
    const int is_bf16 = p.zdtype == 0;
    for (int u = blockIdx.x * Cfg::kZWarps + zw; u < n_units; u += gridDim.x * Cfg::kZWarps) {
      const int row = u / p.z_nchunk, chunk = u - row * p.z_nchunk;
      const RowStat st = zchunk_stat_warp(p.Z, is_bf16, static_cast<size_t>(row) * p.V, chunk,
                                          p.V, p.z_inv_T, lane);
      if (lane == 0) {
        const size_t o = static_cast<size_t>(row) * p.z_nchunk + chunk;
        p.zmax[o] = st.m;
        p.zarg[o] = st.i;
        if (p.z_inv_T > 0.f) p.zsum[o] = st.s;
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int e = warp - 4;
    const int mt = e >> 2;
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = mt * 128 + q * 32 + lane;
    const int grow = p.row0 + row;
    const bool valid = row < p.rows && (grow % p.L) != 0;  // skip each block's verified slot
    Top16 top;
    top16_init(top);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      const bool is_vocab = tile < p.n_vocab_tiles;
      const int n0 = (is_vocab ? tile : tile - p.n_vocab_tiles) * NT;
      if (!mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, p.err, abort_flag, p.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::kAccCols + mt * NT);
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t rr[32];
        __syncwarp();  // tcgen05.ld is warp-collective; lanes diverged on row validity
        tmem_ld_32x32b_x32(tbase + c * 32, rr);
        tmem_ld_wait();
        if (!valid) continue;
        const int cbase = n0 + c * 32;
        if (is_vocab) {
          top16_offer32(top, rr, cbase, p.V - cbase);  // columns past V are not tokens
        } else {
          store_gate32(p.gate_out + static_cast<size_t>(grow) * p.r, rr, cbase, p.r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == NBUF) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (p.write_partials && valid) {
      const size_t off = (static_cast<size_t>(grow) * p.G + blockIdx.x) * kK;  // one list per CTA
      float4* pv = reinterpret_cast<float4*>(p.part_val + off);
      int4* pi = reinterpret_cast<int4*>(p.part_idx + off);
#pragma unroll
      for (int j = 0; j < kK / 4; ++j) {
        pv[j] = make_float4(top.v[4 * j], top.v[4 * j + 1], top.v[4 * j + 2], top.v[4 * j + 3]);
        pi[j] = make_int4(top.i[4 * j], top.i[4 * j + 1], top.i[4 * j + 2], top.i[4 * j + 3]);
      }
    }
  }

  // -------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}


// ------------------------------------------------------------------ CTA-pair kernel
// Row groups of 129..256 rows on CTA pairs with pair MMAs (cta_group::2): the pair takes one
// 256-column vocabulary tile at a time; each CTA stages its own 128 hidden rows and HALF of
// the W tile (128 columns), and the leader's M = 256 x N = 256 MMAs read the B halves of
// both CTAs, so each SM's shared memory takes and serves half the W bytes it would as a
// lone M = 128 x N = 256 CTA. A stage holds one k-block (64) of both operands; the leader's
// full barrier counts both CTAs' bytes; the MMA commits release both CTAs' stages and signal
// both CTAs' accumulators; both CTAs' epilogue warps release an accumulator on the leader.
// Tile t (0 .. n_tiles - 1) of the pair kernel, taken by pair t mod ncl. The gate tiles
// sit in the last slots of the first round: done early (their epilogue overlaps later
// MMAs), by the pairs that get one tile fewer when the tiles do not divide evenly. The
// vocabulary tiles fill the other slots in order. n0 = first column (or W_g row).
struct PairTile {
  bool vocab;
  int n0;
};
__device__ __forceinline__ PairTile pair_tile(int t, int ncl, int n_gate, int n_tiles) {
  const int first_round = ncl < n_tiles ? ncl : n_tiles;
  const int g0 = first_round > n_gate ? first_round - n_gate : 0;
  if (t >= g0 && t < g0 + n_gate) return {false, (t - g0) * 256};
  return {true, (t < g0 ? t : t - n_gate) * 256};
}

template <int S>
struct PairCfg {
  static constexpr int kHalfBytes = 128 * 128;  // 128 vocabulary columns (or W_g rows) x 64 k
  static constexpr int kHBytes = 128 * 128;     // 128 hidden rows x 64 k
  static constexpr int kStage = kHalfBytes + kHBytes;
  static constexpr int kNBuf = 2;
  static constexpr int kAccCols = 256;
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiWarps = 4;  // warps 4..7, one TMEM lane quarter each
  static constexpr int kZWarps = 4;    // warps 2, 3, 8, 9
  static constexpr int kThreads = 32 * 10;
  static constexpr int kBarBytes = 8 * (2 * S + 2 * kNBuf) + 16;
  static constexpr size_t kSmem = 1024 + size_t(S) * kStage + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(kAccCols * kNBuf <= kTmemCols, "TMEM");
};

// kE4M3: the operands are E4M3 (the quantised rows and the quantised head, tiled as
// dfs_pack_e4m3_head lays it out: each 128 vocabulary rows x 128 k bytes one contiguous
// 16 KB tile, both
// K-major 128-byte rows, 128 k per stage, kind::f8f6f4 with K = 32 per instruction), and
// the epilogue scales column v by w_scale[v] and the row by h_scale (no gate tiles).
template <int S, bool kE4M3>
__global__ void __launch_bounds__(PairCfg<S>::kThreads, 1)
    k_lmhead_pair(const __grid_constant__ LmheadParams p) {
  using Cfg = PairCfg<S>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + size_t(S) * Cfg::kStage);
  uint64_t* full = bars;            // leader: both CTAs' bytes of a stage have landed
  uint64_t* empty = bars + S;       // each CTA: the pair MMAs reading a stage are done
  uint64_t* tfull = bars + 2 * S;   // each CTA: an accumulator is complete
  uint64_t* tempty = tfull + Cfg::kNBuf;  // leader: both CTAs have drained an accumulator
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + Cfg::kNBuf);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < Cfg::kNBuf; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * Cfg::kEpiWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&p.tm_h);
    prefetch_tensormap(&p.tm_w);
    prefetch_tensormap(&p.tm_g);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // bf16: launched as a programmatic dependent of whatever precedes it on the stream; the
  // set-up above overlaps that kernel, nothing below touches global memory before it has
  // completed. E4M3: the dependent of the row quantisation; the roles that read its output
  // wait for it below, the target-row statistics do not.
  if (!kE4M3) grid_dependency_wait();
  grid_dependents_launch();

  const int n_tiles = p.n_vocab_tiles + p.n_gate_tiles;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;
  // k-blocks of a tile: 64 bf16 or 128 E4M3 elements (both 128 bytes per row)
  const int KB_bf16 = p.d / 64;
  const int KB_e4m3 = p.d / 128;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------- TMA producer: W half + hidden rows
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);  // the leader's barriers
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (kE4M3) grid_dependency_wait();  // the quantised rows (launched as a dependent)
      for (int tile = cid; ok && tile < n_tiles; tile += ncl) {
        const PairTile pt = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles);
        const bool is_vocab = pt.vocab;
        const bool q8 = kE4M3 && is_vocab;  // E4M3 operands (gate tiles stay bf16)
        const int n0 = pt.n0 + static_cast<int>(rank) * 128;
        const int KB = q8 ? KB_e4m3 : KB_bf16;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * Cfg::kStage);
          const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
          const uint32_t sw = smem_u32(ring + size_t(stage) * Cfg::kStage);
          if (q8) {  // 128 vocabulary rows x 128 k bytes (K-major), and the quantised rows
            // tile (n0 / 128, kb) of the packed head: 16 KB contiguous in memory
            tma_load_2d_pair(sw, &p.tm_w, fb, 0, ((n0 >> 7) * KB + kb) * 128, pol_stream);
            tma_load_2d_pair(sw + Cfg::kHalfBytes, &p.tm_hq, fb, kb * 128,
                             p.row0 + static_cast<int>(rank) * 128, pol_keep);
          } else {
            if (is_vocab) {
              tma_load_2d_pair(sw, &p.tm_w, fb, n0, kb * 64, pol_stream);
              tma_load_2d_pair(sw + 8192, &p.tm_w, fb, n0 + 64, kb * 64, pol_stream);
            } else {
              tma_load_2d_pair(sw, &p.tm_g, fb, kb * 64, n0, pol_keep);
            }
            tma_load_2d_pair(sw + Cfg::kHalfBytes, &p.tm_h, fb, kb * 64,
                             p.row0 + static_cast<int>(rank) * 128, pol_keep);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // The releases of the last stages arrive from the leader's commits; this CTA may exit
      // only after they have landed on its barriers.
      if (ok) {
        for (int i = 0; i < S; ++i) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader && !p.stall_mma) {
      // ------------------------------------------------------- pair MMA issuer (leader)
      constexpr uint32_t kIdescVocab = idesc_bf16_f32(256, true, 256);
      constexpr uint32_t kIdescGate = idesc_bf16_f32(256, false, 256);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < n_tiles; tile += ncl) {
        const bool is_vocab = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles).vocab;
        const bool q8 = kE4M3 && is_vocab;
        const int KB = q8 ? KB_e4m3 : KB_bf16;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = smem_u32(ring + size_t(stage) * Cfg::kStage);
          const uint32_t sh = sw + Cfg::kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // K = 16 (bf16) or 32 (E4M3): 32 bytes per step
            const uint64_t adesc = smem_desc_sw128(sh + kk * 32, 0, 1024);
            if (q8) {
              tc_mma_e4m3_pair(d0, adesc, smem_desc_sw128(sw + kk * 32, 0, 1024),
                               idesc_e4m3_f32(256, 256), (kb | kk) != 0);
            } else {
              const uint64_t bdesc = is_vocab ? smem_desc_sw128(sw + kk * 2048, 8192, 1024)
                                              : smem_desc_sw128(sw + kk * 32, 0, 1024);
              tc_mma_bf16_pair(d0, adesc, bdesc, is_vocab ? kIdescVocab : kIdescGate,
                               (kb | kk) != 0);
            }
          }
          tc_commit_pair_multicast(smem_u32(&empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(smem_u32(&tfull[acc]), 0x3);
        if (++acc == Cfg::kNBuf) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else if (warp == 2 || warp == 3 || warp >= 8) {
    // ------------------------------------------------ target-logit row statistics
    const int zw = warp < 4 ? warp - 2 : warp - 6;
    if (blockIdx.x == 0 && p.zero_ptr != nullptr)
      for (int i = zw * 32 + lane; i < p.zero_count; i += 32 * Cfg::kZWarps) p.zero_ptr[i] = 0;
    const int n_units = p.z_rows * p.z_nchunk;
    const int is_bf16 = p.zdtype == 0;
    for (int u = blockIdx.x * Cfg::kZWarps + zw; u < n_units; u += gridDim.x * Cfg::kZWarps) {
      const int row = u / p.z_nchunk, chunk = u - row * p.z_nchunk;
      const RowStat st = zchunk_stat_warp(p.Z, is_bf16, static_cast<size_t>(row) * p.V, chunk,
                                          p.V, p.z_inv_T, lane);
      if (lane == 0) {
        const size_t o = static_cast<size_t>(row) * p.z_nchunk + chunk;
        p.zmax[o] = st.m;
        p.zarg[o] = st.i;
        if (p.z_inv_T > 0.f) p.zsum[o] = st.s;
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = static_cast<int>(rank) * 128 + q * 32 + lane;
    const int grow = p.row0 + row;
    const bool valid = row < p.rows && (grow % p.L) != 0;  // skip each block's verified slot
    const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
    if (kE4M3) grid_dependency_wait();  // h_scale comes from the quantisation kernel
    const float hs = (kE4M3 && valid) ? p.h_scale[grow] : 1.f;
    Top16 top;
    top16_init(top);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cid; tile < n_tiles; tile += ncl) {
      const PairTile pt = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles);
      const bool is_vocab = pt.vocab;
      const int n0 = pt.n0;
      if (!mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, p.err, abort_flag, p.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::kAccCols);
      for (int c = 0; c < 8; ++c) {
        uint32_t rr[32];
        __syncwarp();  // tcgen05.ld is warp-collective; lanes diverged on row validity
        tmem_ld_32x32b_x32(tbase + c * 32, rr);
        tmem_ld_wait();
        if (!valid) continue;
        const int cbase = n0 + c * 32;
        if (kE4M3 && is_vocab) {  // u = acc * w_scale[v] * h_scale (past V: scale 0, not offered)
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (cbase + j < p.V) w4 = __ldg(reinterpret_cast<const float4*>(p.w_scale + cbase + j));
            rr[j] = __float_as_uint(__uint_as_float(rr[j]) * w4.x * hs);
            rr[j + 1] = __float_as_uint(__uint_as_float(rr[j + 1]) * w4.y * hs);
            rr[j + 2] = __float_as_uint(__uint_as_float(rr[j + 2]) * w4.z * hs);
            rr[j + 3] = __float_as_uint(__uint_as_float(rr[j + 3]) * w4.w * hs);
          }
        }
        if (is_vocab) {
          top16_offer32(top, rr, cbase, p.V - cbase);  // columns past V are not tokens
        } else {
          store_gate32(p.gate_out + static_cast<size_t>(grow) * p.r, rr, cbase, p.r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      if (++acc == Cfg::kNBuf) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (p.write_partials && valid) {
      const size_t off = (static_cast<size_t>(grow) * p.G + cid) * kK;  // one list per pair
      float4* pv = reinterpret_cast<float4*>(p.part_val + off);
      int4* pi = reinterpret_cast<int4*>(p.part_idx + off);
#pragma unroll
      for (int j = 0; j < kK / 4; ++j) {
        pv[j] = make_float4(top.v[4 * j], top.v[4 * j + 1], top.v[4 * j + 2], top.v[4 * j + 3]);
        pi[j] = make_int4(top.i[4 * j], top.i[4 * j + 1], top.i[4 * j + 2], top.i[4 * j + 3]);
      }
    }
  }

  // -------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every pair MMA and every TMEM read of both CTAs is complete
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
  cluster_sync();  // neither CTA leaves while its peer may still use the pair's resources
}

// ------------------------------------------------------------------ vocabulary-major tiles
// The same pair MMAs with the operands' roles exchanged: 256 vocabulary entries (or W_g
// rows) on M -- 128 in each CTA's TMEM lanes, W read MN-major exactly as the pair kernel
// stages it -- and the group's drafted rows on N. A block's verified slot (position 0) has
// no drafted token, so it needs no logits: each CTA fetches the rows of positions 1..L-1 of
// its nb requests as one 3-D box of h viewed as [B][L][d], and N = 2 nb (L - 1) (224 at 32
// blocks of 8) instead of the 256 rows the row-major tiles compute. The real gain is in
// passes over W: a group holds 2 nb requests whatever L is, so where B L rows exceed a
// multiple of 256 only because of the verified slots (32 blocks of 9: 288 rows, 256 drafted)
// one pass replaces two. At 32 blocks of 8 (one pass either way) the row-major kernel stays
// the faster: the turn-around below costs more than the 1/8 of tensor work it saves.
//
// Each CTA's accumulator holds 128 vocabulary entries (lanes) x N drafted rows (columns),
// but the keep-top-16 is per row over the vocabulary, i.e. across lanes. The epilogue
// therefore turns the rows around in shared memory, four 32-row chunks per round: all four
// epilogue warps load their lane quarter of the round's chunks with tcgen05.ld and store them
// as [row][vocabulary] (rows padded to 129 floats), then warp q reads back chunk q of the
// round, one row per thread and 128 consecutive vocabulary entries in increasing id order,
// and offers them to the row's sorted top-16 in registers (a thread owns rows 32 q + lane
// and 128 + 32 q + lane), so the four warps rank in parallel. Two named barriers per round
// order the stores, the reads and the next round's stores.
// At the end the odd CTA's lists (its 128 vocabulary entries per tile) are read by the
// leader through distributed shared memory and merged by (value desc, id asc) into one
// partial list per row and pair, the layout the tail reads.
template <int S>
struct VtCfg {
  static constexpr int kABytes = 128 * 128;  // 128 vocabulary entries (or W_g rows) x 64 k
  static constexpr int kHMaxBytes = 128 * 128;  // up to 128 drafted rows per CTA x 64 k
  static constexpr int kNBuf = 2;
  static constexpr int kAccCols = 256;  // N <= 256
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiWarps = 4;  // warps 4..7, one TMEM lane quarter each
  static constexpr int kZWarps = 4;    // warps 2, 3, 8, 9
  static constexpr int kThreads = 32 * 10;
  // a turned-around row: 128 floats + 1 of skew (the lanes' reads of one column hit 32 banks)
  static constexpr int kXStride = 129;
  static constexpr int kXBytes = 4 * 32 * kXStride * 4;  // one round: four 32-row chunks
  static constexpr int kAuxBytes = kXBytes;
  static constexpr int kBarBytes = 8 * (2 * S + 2 * kNBuf) + 16;
  static constexpr size_t smem(uint32_t stage_bytes) {
    return 1024 + size_t(S) * stage_bytes + size_t(kAuxBytes) + kBarBytes;
  }
  // five stages hold up to 120 drafted rows per CTA (a 31 KB stage); 128 rows take four
  static constexpr uint32_t kMaxStage = S >= 5 ? kABytes + 120 * 128 : kABytes + kHMaxBytes;
  static constexpr size_t kSmemMax = smem(kMaxStage);
  static_assert(kSmemMax <= 232448, "shared memory");
  static_assert(kXBytes >= 2 * 128 * 2 * kK * 4, "the peer's lists fit the round buffer");
  static_assert(kXBytes % 16 == 0, "the barriers follow 16-byte aligned");
};

// (x, id) enters t when it ranks before t's last member by (value desc, id asc); it goes
// after every member that ranks before it.
__device__ __forceinline__ void top16_insert_ranked(Top16& t, float x, int id) {
  if (!ranks_before(x, id, t.v[kK - 1], t.i[kK - 1])) return;
  bool ge[kK];
#pragma unroll
  for (int k = 0; k < kK; ++k) ge[k] = ranks_before(t.v[k], t.i[k], x, id);
#pragma unroll
  for (int k = kK - 1; k >= 1; --k) {
    t.v[k] = ge[k] ? t.v[k] : (ge[k - 1] ? x : t.v[k - 1]);
    t.i[k] = ge[k] ? t.i[k] : (ge[k - 1] ? id : t.i[k - 1]);
  }
  t.v[0] = ge[0] ? t.v[0] : x;
  t.i[0] = ge[0] ? t.i[0] : id;
}

// The tile's accumulator turned around through the round buffer, four 32-row chunks per
// round: all four epilogue warps store their lane quarter of the round's chunks as
// [row][vocabulary] rows, then warp q ranks chunk q, one row per thread, 128 consecutive
// entries in increasing id order. (Measured: a per-row threshold filter with queued
// candidates instead of this, after three such tiles, ran slower per tile on these warps.)
template <class Cfg>
__device__ __forceinline__ void vt_rank_turned(float* xbuf, uint32_t tbase, int nchunk, int q,
                                               int lane, int vbase, int V, Top16& top0,
                                               Top16& top1) {
#pragma unroll
  for (int rd = 0; rd < 2; ++rd) {
    if (4 * rd < nchunk) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {  // this warp's lane quarter of the round's chunks
        const int c = 4 * rd + k;
        if (c < nchunk) {
          uint32_t rr[32];
          tmem_ld_32x32b_x32(tbase + c * 32, rr);
          tmem_ld_wait();
          float* xb = xbuf + k * (32 * Cfg::kXStride) + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j) xb[j * Cfg::kXStride] = __uint_as_float(rr[j]);
        }
      }
      named_bar_sync(2, 128);
      if (4 * rd + q < nchunk) {  // row 32 (4 rd + q) + lane
        Top16& top = rd == 0 ? top0 : top1;
        const float* xrow = xbuf + (q * 32 + lane) * Cfg::kXStride;
#pragma unroll 1
        for (int sub = 0; sub < 4; ++sub) {
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(xrow[sub * 32 + u]);
          const int cbase = vbase + sub * 32;
          top16_offer32(top, v, cbase, V - cbase);  // entries past V are not tokens
        }
      }
      named_bar_sync(2, 128);  // the round's reads are done before the next stores
    }
  }
}

template <int S>
__global__ void __launch_bounds__(VtCfg<S>::kThreads, 1)
    k_lmhead_vt(const __grid_constant__ LmheadParams p) {
  using Cfg = VtCfg<S>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t stage_bytes = p.stage_bytes;
  uint8_t* ring = smem;
  float* xbuf = reinterpret_cast<float*>(ring + size_t(S) * stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xbuf) + Cfg::kAuxBytes);
  uint64_t* full = bars;            // leader: both CTAs' bytes of a stage have landed
  uint64_t* empty = bars + S;       // each CTA: the pair MMAs reading a stage are done
  uint64_t* tfull = bars + 2 * S;   // each CTA: an accumulator is complete
  uint64_t* tempty = tfull + Cfg::kNBuf;  // leader: both CTAs have drained an accumulator
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + Cfg::kNBuf);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int P = p.L - 1;
  const int hrows = p.nb * P;  // drafted rows per CTA; the pair MMAs' N is twice that
  const int N = 2 * hrows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < Cfg::kNBuf; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * Cfg::kEpiWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&p.tm_h3);
    prefetch_tensormap(&p.tm_w);
    prefetch_tensormap(&p.tm_g);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  grid_dependency_wait();  // programmatic dependent: the set-up above overlaps the previous kernel
  grid_dependents_launch();

  const int n_tiles = p.n_vocab_tiles + p.n_gate_tiles;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;
  const int KB = p.d / 64;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------- TMA producer: 128 A rows + this CTA's drafted rows
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);  // the leader's barriers
      const uint32_t tx = static_cast<uint32_t>(Cfg::kABytes + hrows * 128);
      const int hb = p.b0 + static_cast<int>(rank) * p.nb;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < n_tiles; tile += ncl) {
        const PairTile pt = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles);
        const int n0 = pt.n0 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * tx);
          const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
          const uint32_t sw = smem_u32(ring + size_t(stage) * stage_bytes);
          if (pt.vocab) {
            tma_load_2d_pair(sw, &p.tm_w, fb, n0, kb * 64, pol_stream);
            tma_load_2d_pair(sw + 8192, &p.tm_w, fb, n0 + 64, kb * 64, pol_stream);
          } else {
            tma_load_2d_pair(sw, &p.tm_g, fb, kb * 64, n0, pol_keep);
          }
          tma_load_3d_pair(sw + Cfg::kABytes, &p.tm_h3, fb, kb * 64, 1, hb, pol_keep);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (ok) {  // the releases of the last stages land before this CTA may exit
        for (int i = 0; i < S; ++i) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader && !p.stall_mma) {
      // ------------------------------------------------------- pair MMA issuer (leader)
      const uint32_t id_vocab = idesc_bf16_f32(N, false, 256, true);  // A = W, MN-major
      const uint32_t id_gate = idesc_bf16_f32(N, false, 256, false);  // A = W_g, K-major
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < n_tiles; tile += ncl) {
        const bool is_vocab = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles).vocab;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, p.err, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = smem_u32(ring + size_t(stage) * stage_bytes);
          const uint32_t sh = sw + Cfg::kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // K = 16 per instruction: 32 bytes of a K-major row
            const uint64_t bdesc = smem_desc_sw128(sh + kk * 32, 0, 1024);
            const uint64_t adesc = is_vocab ? smem_desc_sw128(sw + kk * 2048, 8192, 1024)
                                            : smem_desc_sw128(sw + kk * 32, 0, 1024);
            tc_mma_bf16_pair(d0, adesc, bdesc, is_vocab ? id_vocab : id_gate, (kb | kk) != 0);
          }
          tc_commit_pair_multicast(smem_u32(&empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(smem_u32(&tfull[acc]), 0x3);
        if (++acc == Cfg::kNBuf) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else if (warp == 2 || warp == 3 || warp >= 8) {
    // ------------------------------------------------ target-logit row statistics
    const int zw = warp < 4 ? warp - 2 : warp - 6;
    if (blockIdx.x == 0 && p.zero_ptr != nullptr)
      for (int i = zw * 32 + lane; i < p.zero_count; i += 32 * Cfg::kZWarps) p.zero_ptr[i] = 0;
    const int n_units = p.z_rows * p.z_nchunk;
    const int is_bf16 = p.zdtype == 0;
    for (int u = blockIdx.x * Cfg::kZWarps + zw; u < n_units; u += gridDim.x * Cfg::kZWarps) {
      const int row = u / p.z_nchunk, chunk = u - row * p.z_nchunk;
      const RowStat st = zchunk_stat_warp(p.Z, is_bf16, static_cast<size_t>(row) * p.V, chunk,
                                          p.V, p.z_inv_T, lane);
      if (lane == 0) {
        const size_t o = static_cast<size_t>(row) * p.z_nchunk + chunk;
        p.zmax[o] = st.m;
        p.zarg[o] = st.i;
        if (p.z_inv_T > 0.f) p.zsum[o] = st.s;
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const int nchunk = (N + 31) >> 5;
    Top16 top0, top1;  // rows 32 q + lane and 128 + 32 q + lane of the group's N
    top16_init(top0);
    top16_init(top1);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = cid; tile < n_tiles; tile += ncl) {
      const PairTile pt = pair_tile(tile, ncl, p.n_gate_tiles, n_tiles);
      const bool w_ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, p.err, abort_flag, p.wait_limit_ns);
      // all four warps go on, or none: the barriers below need every one of them
      if (!named_bar_and(2, 128, w_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::kAccCols);
      const int vbase = pt.n0 + static_cast<int>(rank) * 128;  // this CTA's first M entry
      if (pt.vocab) {
        vt_rank_turned<Cfg>(xbuf, tbase, nchunk, q, lane, vbase, p.V, top0, top1);
      } else {
        // gate tile: lane = unit j of g (a W_g row), column = drafted row; sigmoid, and the
        // 32 lanes of a store write 32 consecutive units of one row
        const int unit = vbase + q * 32 + lane;
        for (int c = 0; c < nchunk; ++c) {
          uint32_t rr[32];
          tmem_ld_32x32b_x32(tbase + c * 32, rr);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = c * 32 + j;
            const int half = col >= hrows, i = col - half * hrows;
            const int b = p.b0 + half * p.nb + i / P, t = 1 + i % P;
            if (col < N && b < p.n_req && unit < p.r)
              p.gate_out[(static_cast<size_t>(b) * p.L + t) * p.r + unit] =
                  1.0f / (1.0f + expf(-__uint_as_float(rr[j])));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      if (++acc == Cfg::kNBuf) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    // every warp's reads of the round buffer are done before it is reused for the lists
    named_bar_sync(2, 128);
    if (ok && !leader) {
      // the odd CTA leaves its lists in its own round buffer for the leader to read
      float* dst = xbuf + static_cast<size_t>(q * 32 + lane) * (2 * kK);
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        dst[k] = top0.v[k];
        dst[kK + k] = __int_as_float(top0.i[k]);
        dst[128 * 2 * kK + k] = top1.v[k];
        dst[128 * 2 * kK + kK + k] = __int_as_float(top1.i[k]);
      }
    }
    // -------------------------------------------------------------- teardown (epilogue)
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // every pair MMA and TMEM read of both CTAs is done; the lists are out
    if (ok && leader && p.write_partials) {
      const uint32_t peer = mapa_shared(smem_u32(xbuf), 1) +
                            static_cast<uint32_t>(q * 32 + lane) * (2 * kK * 4);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        Top16& top = s == 0 ? top0 : top1;
        const uint32_t src = peer + static_cast<uint32_t>(s) * (128 * 2 * kK * 4);
        float pv[kK];
        int pi[kK];
#pragma unroll
        for (int u = 0; u < kK / 4; ++u) {
          const float4 a = ld_dsmem_f4(src + u * 16);
          const float4 b = ld_dsmem_f4(src + kK * 4 + u * 16);
          pv[4 * u] = a.x; pv[4 * u + 1] = a.y; pv[4 * u + 2] = a.z; pv[4 * u + 3] = a.w;
          pi[4 * u] = __float_as_int(b.x); pi[4 * u + 1] = __float_as_int(b.y);
          pi[4 * u + 2] = __float_as_int(b.z); pi[4 * u + 3] = __float_as_int(b.w);
        }
#pragma unroll
        for (int k = 0; k < kK; ++k) top16_insert_ranked(top, pv[k], pi[k]);
        const int col = (4 * s + q) * 32 + lane;  // the drafted row this list belongs to
        const int half = col >= hrows, i = col - half * hrows;
        const int b = p.b0 + half * p.nb + i / P, t = 1 + i % P;
        if (col < N && b < p.n_req) {
          const size_t grow = static_cast<size_t>(b) * p.L + t;
          const size_t off = (grow * p.G + cid) * kK;  // one list per pair
          float4* ov = reinterpret_cast<float4*>(p.part_val + off);
          int4* oi = reinterpret_cast<int4*>(p.part_idx + off);
#pragma unroll
          for (int j = 0; j < kK / 4; ++j) {
            ov[j] = make_float4(top.v[4 * j], top.v[4 * j + 1], top.v[4 * j + 2], top.v[4 * j + 3]);
            oi[j] = make_int4(top.i[4 * j], top.i[4 * j + 1], top.i[4 * j + 2], top.i[4 * j + 3]);
          }
        }
      }
    }
    cluster_sync();  // the peer's lists stay in place until the leader has read them
    return;
  }

  // -------------------------------------------------------------- teardown (other warps)
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
  cluster_sync();
}

// ------------------------------------------------------------------ row quantisation
// One block per row of h [rows, d] bf16 (d a multiple of 8): the row's largest magnitude,
// its power-of-two scale (the smallest 2^e with amax <= 448 * 2^e, from the exponent and
// mantissa bits of amax; 1 when amax < 2^-100), then q = E4M3(h * 2^-e) rounded to nearest
// even (h * 2^-e is exact).
__global__ void __launch_bounds__(256) k_quantize_rows_e4m3(const uint16_t* __restrict__ h, int d,
                                                          uint8_t* __restrict__ q,
                                                          float* __restrict__ scale) {
  __shared__ float wmax[8];
  grid_dependents_launch();  // the LM-head kernel may set up while the rows are quantised
  const size_t base = static_cast<size_t>(blockIdx.x) * d;
  const int nch = d / 8;
  float amax = 0.f;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(h + base) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[j] & 0xFFFFu)),
                               fabsf(bf16_bits_to_float(w[j] >> 16))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
  for (int i = 1; i < (blockDim.x >> 5); ++i) amax = fmaxf(amax, wmax[i]);
  // amax = 1.M 2^(Eb - 127) = f 2^E with f = 1.M / 2, E = Eb - 126; 448 = 0.875 2^9:
  // e = E - 9 + (f > 0.875) = Eb - 135 + (M > 0x600000)
  const uint32_t bits = __float_as_uint(amax);
  const int Eb = static_cast<int>(bits >> 23) & 0xFF;
  int e = 0;
  if (Eb >= 27) e = Eb - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);  // amax >= 2^-100
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
  if (threadIdx.x == 0) scale[blockIdx.x] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(h + base) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const float2 a = make_float2(bf16_bits_to_float(w[j] & 0xFFFFu) * inv,
                                   bf16_bits_to_float(w[j] >> 16) * inv);
      const float2 b = make_float2(bf16_bits_to_float(w[j + 1] & 0xFFFFu) * inv,
                                   bf16_bits_to_float(w[j + 1] >> 16) * inv);
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
      out[j >> 1] = lo | (hi << 16);
    }
    reinterpret_cast<uint2*>(q + base)[c] = make_uint2(out[0], out[1]);
  }
}

// ------------------------------------------------------------------ head packing
// One block per 128 x 128-byte tile (vb, kb) of the E4M3 head: rows 128 vb .. of Wq [V, d]
// (row-major bytes), k bytes 128 kb .., written as one contiguous 16 KB tile, row after row;
// rows past V are zeros.
__global__ void __launch_bounds__(256) k_pack_e4m3_head(const uint8_t* __restrict__ Wq, int V,
                                                         int d, uint8_t* __restrict__ out) {
  const int KB = d / 128;
  const int vb = blockIdx.x / KB, kb = blockIdx.x - vb * KB;
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(blockIdx.x) * 16384);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = threadIdx.x + 256 * i;  // 16-byte piece: row e / 8, bytes 16 (e % 8) ..
    const int row = vb * 128 + (e >> 3);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (row < V)
      x = __ldg(reinterpret_cast<const uint4*>(Wq + static_cast<size_t>(row) * d + kb * 128) +
                (e & 7));
    dst[e] = x;
  }
}

// ------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major bf16 matrix [outer, inner] (inner contiguous), box inner_box x outer_box,
// 128-byte swizzle, zero fill outside the matrix.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                    uint32_t inner_box, uint32_t outer_box) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {inner_box, outer_box};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major byte matrix [outer, inner] (E4M3), box inner_box x outer_box, 128-byte swizzle.
bool encode_u8_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                  uint32_t inner_box, uint32_t outer_box) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {inner_box, outer_box};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// h [B][L][d] bf16 seen as a 3-D tensor (d innermost), box 64 (k) x (L - 1) positions x nb
// requests, 128-byte swizzle: one box is the drafted rows of nb requests, 128 B each, in
// (request, position) order; requests past B are zero-filled.
bool encode_bf16_drafted_rows(CUtensorMap* m, const void* base, int d, int L, int B, int nb) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(L) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(L - 1), static_cast<cuuint32_t>(nb)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int S>
cudaError_t launch_vt(const LmheadParams& prm, int grid, cudaStream_t s) {
  using Cfg = VtCfg<S>;
  auto kern = k_lmhead_vt<S>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmemMax));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::smem(prm.stage_bytes);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int MT, int NT, int NBUF, int SW, int SH>
cudaError_t launch_cfg(const LmheadParams& prm, int grid, cudaStream_t s) {
  using Cfg = LmCfg<MT, NT, NBUF, SW, SH>;
  auto kern = k_lmhead_tc<MT, NT, NBUF, SW, SH>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int S, bool kE4M3 = false>
cudaError_t launch_pair(const LmheadParams& prm, int grid, cudaStream_t s, bool dependent = false) {
  using Cfg = PairCfg<S>;
  auto kern = k_lmhead_pair<S, kE4M3>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

// Requests per CTA of a vocabulary-major group: a multiple of 8 (so N = 2 nb (L - 1) is a
// multiple of 16) with nb (L - 1) <= 128; 0 when a block has more than 16 drafted positions.
int vt_requests_per_cta(int L) { return (L >= 2 && L - 1 <= 16) ? 8 * (16 / (L - 1)) : 0; }

// The vocabulary launches of a call with more than 128 rows on k_lmhead_vt: groups of up to
// 2 nb_max requests, the last one with nb shrunk to what it holds (rounded up to 8).
cudaError_t launch_vt_groups(const LmheadLaunch& a, LmheadParams& prm, int nb_max, cudaStream_t s) {
  const int B = a.rows_total / a.L;
  prm.n_vocab_tiles = (a.V + 255) / 256;
  prm.n_gate_tiles = a.gate ? (a.r + 255) / 256 : 0;
  prm.write_partials = 1;
  if (!encode_bf16_2d(&prm.tm_g, a.gate ? a.Wg : a.hidden, a.d, a.gate ? a.r : a.rows_total, 64,
                      128))
    return cudaErrorInvalidValue;
  for (int b0 = 0; b0 < B; b0 += 2 * nb_max) {
    const int bg = B - b0 < 2 * nb_max ? B - b0 : 2 * nb_max;
    const int half = (((bg + 1) / 2) + 7) / 8 * 8;
    const int nb = half < nb_max ? half : nb_max;
    if (!encode_bf16_drafted_rows(&prm.tm_h3, a.hidden, a.d, a.L, B, nb)) return cudaErrorInvalidValue;
    prm.b0 = b0;
    prm.nb = nb;
    prm.n_req = B;
    prm.stage_bytes = static_cast<uint32_t>(VtCfg<5>::kABytes + nb * (a.L - 1) * 128);
    const bool first = b0 == 0;  // the statistics and the counter reset ride on the first
    prm.Z = a.Z;
    prm.zdtype = a.zdtype;
    prm.z_rows = first ? a.z_rows : 0;
    prm.z_nchunk = a.z_nchunk;
    prm.z_inv_T = a.z_inv_T;
    prm.zmax = a.zmax;
    prm.zarg = a.zarg;
    prm.zsum = a.zsum;
    prm.zero_ptr = first ? a.zero_ptr : nullptr;
    prm.zero_count = first ? a.zero_count : 0;
    // five ring stages when they fit next to the turn-around buffers, else four
    const cudaError_t e = prm.stage_bytes <= VtCfg<5>::kMaxStage ? launch_vt<5>(prm, a.G, s)
                                                                   : launch_vt<4>(prm, a.G, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool lmhead_row_split(int rows_total, int G) { return rows_total > 128 && G % 2 == 0; }

cudaError_t launch_lmhead_tc(const LmheadLaunch& a, cudaStream_t s) {
  LmheadParams prm;
  memset(&prm, 0, sizeof(prm));
  // A row group smaller than a tile is fetched as one box of its rows rounded up to 8 (the
  // single-CTA kernel zeroes the rest once); larger groups take 128-row boxes.
  const int h_rows = a.rows_total <= 128 ? ((a.rows_total + 7) / 8) * 8 : 128;
  prm.h_box_bytes = static_cast<uint32_t>(h_rows) * 128u;
  if (!encode_bf16_2d(&prm.tm_h, a.hidden, a.d, a.rows_total, 64, h_rows))
    return cudaErrorInvalidValue;
  // Dummy-but-valid maps when a tile kind is not used, so every map is well formed.
  if (!encode_bf16_2d(&prm.tm_w, a.vocab ? a.W : a.hidden, a.vocab ? a.V : a.d,
                      a.vocab ? a.d : a.rows_total, 64, 64))
    return cudaErrorInvalidValue;
  prm.L = a.L;
  prm.V = a.V;
  prm.d = a.d;
  prm.r = a.r;
  // More than 128 rows: CTA pairs split each row group (gate-only launches included)
  const bool rs = lmhead_row_split(a.rows_total, a.vocab ? a.G : 2);
  prm.G = rs ? a.G / 2 : a.G;  // partial lists per row: one per CTA, or per pair when split
  prm.part_val = a.part_val;
  prm.part_idx = a.part_idx;
  prm.gate_out = a.gate_out;
  prm.err = a.err;
  prm.wait_limit_ns = a.wait_limit_ns > 0 ? a.wait_limit_ns : kWaitLimitNs;
  prm.stall_mma = a.stall_mma;
  // More than 128 rows with the vocabulary: the vocabulary-major pair kernel computes the
  // drafted rows only, so it needs fewer passes over W when the verified slots tip the rows
  // over a multiple of 256 (e.g. 32 blocks of 9); per pass it is a little slower than the
  // row-major pair kernel (its epilogue turns the rows around in shared memory). Chosen when
  // it saves a pass (variant 0), or always (6); 5 forces the row-major pair kernel.
  int vt_nb = (rs && a.vocab) ? vt_requests_per_cta(a.L) : 0;
  if (vt_nb > 0 && a.lmhead_variant != 6) {
    const int B = a.rows_total / a.L;
    const int vt_passes = (B + 2 * vt_nb - 1) / (2 * vt_nb);
    const int pair_passes = (a.rows_total + 255) / 256;
    if (a.lmhead_variant != 0 || vt_passes >= pair_passes) vt_nb = 0;
  }
  if (vt_nb > 0) return launch_vt_groups(a, prm, vt_nb, s);
  for (int row0 = 0; row0 < a.rows_total; row0 += 256) {
    prm.row0 = row0;
    // the target-logit statistics and the counter reset ride on the first launch only
    const bool first = row0 == 0;
    prm.Z = a.Z;
    prm.zdtype = a.zdtype;
    prm.z_rows = first ? a.z_rows : 0;
    prm.z_nchunk = a.z_nchunk;
    prm.z_inv_T = a.z_inv_T;
    prm.zmax = a.zmax;
    prm.zarg = a.zarg;
    prm.zsum = a.zsum;
    prm.zero_ptr = first ? a.zero_ptr : nullptr;
    prm.zero_count = first ? a.zero_count : 0;
    prm.rows = a.rows_total - row0 < 256 ? a.rows_total - row0 : 256;
    // Row groups of up to 128 rows: one M tile x 256 vocabulary columns per CTA,
    // double-buffered TMEM. 129..256 rows: CTA pairs on one 256-column tile, 128 rows each,
    // pair MMAs with each CTA staging half of the W tile.
    const int NT = 256;
    prm.n_vocab_tiles = a.vocab ? (a.V + NT - 1) / NT : 0;
    prm.n_gate_tiles = a.gate ? (a.r + NT - 1) / NT : 0;
    prm.write_partials = a.vocab ? 1 : 0;
    if (!encode_bf16_2d(&prm.tm_g, a.gate ? a.Wg : a.hidden, a.d, a.gate ? a.r : a.rows_total,
                        64, static_cast<uint32_t>(a.gate ? (rs ? NT / 2 : NT) : 128)))
      return cudaErrorInvalidValue;
    const int grid = a.vocab ? a.G : (prm.n_gate_tiles > 0 ? prm.n_gate_tiles : 1) * (rs ? 2 : 1);
    const cudaError_t e = rs ? launch_pair<7, false>(prm, grid, s, true)
                             : launch_cfg<1, 256, 2, 5, 4>(prm, grid, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t e4m3_head_bytes(int V, int d) {
  return static_cast<size_t>((V + 127) / 128) * 128 * static_cast<size_t>(d);
}

cudaError_t launch_pack_e4m3_head(const void* Wq, int V, int d, void* out, cudaStream_t s) {
  const int tiles = ((V + 127) / 128) * (d / 128);
  k_pack_e4m3_head<<<tiles, 256, 0, s>>>(static_cast<const uint8_t*>(Wq), V, d,
                                          static_cast<uint8_t*>(out));
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launches(1);
  return e;
}

cudaError_t launch_quantize_rows_e4m3(const void* h, int rows, int d, void* q, float* scale,
                                      cudaStream_t s) {
  k_quantize_rows_e4m3<<<rows, 256, 0, s>>>(static_cast<const uint16_t*>(h), d,
                                             static_cast<uint8_t*>(q), scale);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launches(1);
  return e;
}

cudaError_t launch_lmhead_e4m3(const LmheadLaunch& a, cudaStream_t s) {
  LmheadParams prm;
  memset(&prm, 0, sizeof(prm));
  if (!encode_u8_2d(&prm.tm_hq, a.hq, a.d, a.rows_total, 128, 128)) return cudaErrorInvalidValue;
  // the packed head as rows of 128 bytes: tile (vb, kb) is rows (vb * d / 128 + kb) * 128 ..
  if (!encode_u8_2d(&prm.tm_w, a.Wq, 128, static_cast<uint64_t>(e4m3_head_bytes(a.V, a.d) / 128),
                    128, 128))
    return cudaErrorInvalidValue;
  // gate tiles stay bf16: the bf16 rows and W_g (128 W_g rows per CTA of a pair)
  if (!encode_bf16_2d(&prm.tm_h, a.hidden, a.d, a.rows_total, 64, 128)) return cudaErrorInvalidValue;
  prm.h_box_bytes = 128u * 128u;
  if (!encode_bf16_2d(&prm.tm_g, a.gate ? a.Wg : a.hidden, a.d, a.gate ? a.r : a.rows_total, 64,
                      128))
    return cudaErrorInvalidValue;
  prm.L = a.L;
  prm.V = a.V;
  prm.d = a.d;
  prm.r = a.r;
  prm.G = a.G / 2;  // one partial list per CTA pair
  prm.part_val = a.part_val;
  prm.part_idx = a.part_idx;
  prm.gate_out = a.gate_out;
  prm.err = a.err;
  prm.wait_limit_ns = a.wait_limit_ns > 0 ? a.wait_limit_ns : kWaitLimitNs;
  prm.stall_mma = a.stall_mma;
  prm.w_scale = a.w_scale;
  prm.h_scale = a.h_scale;
  prm.n_vocab_tiles = (a.V + 255) / 256;
  prm.n_gate_tiles = a.gate ? (a.r + 255) / 256 : 0;
  prm.write_partials = 1;
  for (int row0 = 0; row0 < a.rows_total; row0 += 256) {
    const bool first = row0 == 0;
    prm.row0 = row0;
    prm.rows = a.rows_total - row0 < 256 ? a.rows_total - row0 : 256;
    prm.Z = a.Z;
    prm.zdtype = a.zdtype;
    prm.z_rows = first ? a.z_rows : 0;
    prm.z_nchunk = a.z_nchunk;
    prm.z_inv_T = a.z_inv_T;
    prm.zmax = a.zmax;
    prm.zarg = a.zarg;
    prm.zsum = a.zsum;
    prm.zero_ptr = first ? a.zero_ptr : nullptr;
    prm.zero_count = first ? a.zero_count : 0;
    // the first group is a programmatic dependent of the row quantisation
    const cudaError_t e = launch_pair<7, true>(prm, a.G, s, first);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool encode_bf16_2d_tile(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t inner_box, uint32_t outer_box) {
  return encode_bf16_2d(m, base, inner, outer, inner_box, outer_box);
}

}  // namespace dfs
