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
// Design:
//   * persistent grid, one CTA per SM; CTA i takes vocabulary tiles i, i+G, ...;
//   * two TMA producers fill two rings of shared memory guarded by mbarriers, 128-byte
//     swizzle: warp 0 streams W_vocab (the MN-major B operand, vocabulary contiguous,
//     64x64 boxes) through a deep ring, because HBM latency times the per-SM share of
//     bandwidth needs ~100 KB of W in flight per SM; warp 2 feeds the hidden rows (the
//     K-major A operand, L2-resident, 64x128 boxes) through a shallow ring;
//   * warp 1 issues tcgen05.mma (M = 128 rows, N = NT vocabulary columns, K = 16 per
//     instruction) into TMEM accumulators, NBUF of them so the epilogue of one tile
//     overlaps the MMAs of the next;
//   * warps 4.. (4 per 128-row tile) drain TMEM with tcgen05.ld: each thread owns one
//     row and keeps its running top-16 in registers (unsorted, weakest member tracked); per
//     32-column load it tests the maximum against the weakest, then visits only the
//     lane's own candidates, so a warp does not run insertion code for its other lanes;
//     at the end it sorts the 16 and writes them as one partial list of the row (the tail
//     kernel merges the G lists of a row).
//   * gate tiles use W_g [r, d] (K-major) as the B operand; their epilogue applies the
//     sigmoid and stores g[m, j] in fp32;
//   * four more warps (3 and the last three) stream the target logits (16-byte loads,
//     read once, 8 per lane in flight) and write per-chunk row statistics (max, argmax,
//     sum of exp) for verification, so those bytes move while the tensor pipe works on W
//     instead of in a kernel of their own.
// Every mbarrier wait is bounded; on expiry the kernel sets the error word, stops all
// roles, and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "rowstat.cuh"

namespace dfs {

struct LmheadParams {
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
};

template <int MT, int NT, int NBUF, int SW, int SH, int CL, int RS>
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
  static_assert(CL == 1 || CL == 2 || CL == 4, "cluster size");
  static_assert(!RS || (CL == 2 && MT == 1), "a row-split pair is a cluster of two 128-row CTAs");
  static constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << CL) - 1u);
};

// A row's running top-16, unsorted, with its weakest member tracked (lowest value; among
// equal values the highest id, which ranks last). Ids arrive in increasing order, so a new
// value enters only when it beats the weakest strictly.
struct Top16 {
  float v[kK];
  int i[kK];
  float wv;  // weakest value (the entry threshold)
  int wi;    // its id
  int wp;    // its slot
};

__device__ __forceinline__ void top16_init(Top16& t) {
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    t.v[k] = -INFINITY;
    t.i[k] = 0x7fffffff;
  }
  t.wv = -INFINITY;
  t.wi = 0x7fffffff;
  t.wp = 0;
}

// Replace the weakest member by (x, id) (caller checked x > t.wv), then find the new weakest.
__device__ __forceinline__ void top16_replace(Top16& t, float x, int id) {
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    const bool here = k == t.wp;
    t.v[k] = here ? x : t.v[k];
    t.i[k] = here ? id : t.i[k];
  }
  float wv = t.v[0];
  int wi = t.i[0], wp = 0;
#pragma unroll
  for (int k = 1; k < kK; ++k) {
    const bool weaker = t.v[k] < wv || (t.v[k] == wv && t.i[k] > wi);
    wv = weaker ? t.v[k] : wv;
    wi = weaker ? t.i[k] : wi;
    wp = weaker ? k : wp;
  }
  t.wv = wv;
  t.wi = wi;
  t.wp = wp;
}

// Sort into (value desc, id asc): odd-even transposition, static indices only.
__device__ __forceinline__ void top16_sort(Top16& t) {
#pragma unroll
  for (int pass = 0; pass < kK; ++pass) {
#pragma unroll
    for (int k = pass & 1; k + 1 < kK; k += 2) {
      const bool swap = t.v[k + 1] > t.v[k] || (t.v[k + 1] == t.v[k] && t.i[k + 1] < t.i[k]);
      const float a = t.v[k], b = t.v[k + 1];
      const int ia = t.i[k], ib = t.i[k + 1];
      t.v[k] = swap ? b : a;
      t.v[k + 1] = swap ? a : b;
      t.i[k] = swap ? ib : ia;
      t.i[k + 1] = swap ? ia : ib;
    }
  }
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

// Offer 32 consecutive logits (ids cbase..cbase+31, those at or past lim ignored): a cheap
// maximum test first, then only the lanes' actual candidates, lowest id first.
__device__ __forceinline__ void top16_offer32(Top16& t, const uint32_t (&r)[32], int cbase, int lim) {
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) mx = fmaxf(mx, j < lim ? __uint_as_float(r[j]) : -INFINITY);
  if (!(mx > t.wv)) return;
  uint32_t mask = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    mask |= (j < lim && __uint_as_float(r[j]) > t.wv) ? (1u << j) : 0u;
  while (mask) {
    const int j = __ffs(mask) - 1;
    mask &= mask - 1;
    const float x = __uint_as_float(pick32(r, j));
    if (x > t.wv) top16_replace(t, x, cbase + j);
  }
}

template <int MT, int NT, int NBUF, int SW, int SH, int CL, int RS>
__global__ void __launch_bounds__(LmCfg<MT, NT, NBUF, SW, SH, CL, RS>::kThreads, 1)
    k_lmhead_tc(const __grid_constant__ LmheadParams p) {
  using Cfg = LmCfg<MT, NT, NBUF, SW, SH, CL, RS>;
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
      mbar_init(smem_u32(&wempty[s]), RS ? 2 : 1);  // a shared W stage: both CTAs release it
    }
    for (int s = 0; s < SH; ++s) {
      mbar_init(smem_u32(&hfull[s]), 1);
      mbar_init(smem_u32(&hempty[s]), RS ? 1 : CL);  // shared hidden rows: every CTA releases
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
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();  // peers' barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Every CTA of this persistent grid is resident now: let the dependent tail kernel launch
  // onto SMs as they free up (it waits for this grid's completion before reading).
  grid_dependents_launch();

  // Tiles: vocabulary tiles, then gate tiles. Clusters either share the hidden rows (each
  // CTA its own tile; tiles padded so the CL CTAs of a cluster process the same number: a
  // CTA takes tile s*CL + rank for super-tiles s = cluster, cluster + clusters, ..., and a
  // padding tile streams zeros and produces nothing) or, as a row-split pair (RS), share
  // the W tile: both CTAs take the same tile t = cluster, cluster + clusters, ..., CTA
  // rank r computing rows 128r..128r+127 of it.
  const int n_tiles = p.n_vocab_tiles + p.n_gate_tiles;
  const int n_loop = RS ? n_tiles : (n_tiles + CL - 1) / CL;
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cid = blockIdx.x / CL;
  const int ncl = gridDim.x / CL;
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
      for (int sup = cid; ok && sup < n_loop; sup += ncl) {
        const int tile = RS ? sup : sup * CL + rank;
        const bool is_pad = tile >= n_tiles;
        const bool is_vocab = tile < p.n_vocab_tiles || is_pad;
        // padding tiles load boxes wholly past the vocabulary: zeros
        const int n0 = is_pad ? ((p.V + 63) / 64) * 64 : (is_vocab ? tile : tile - p.n_vocab_tiles) * NT;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wempty[stage]), phase ^ 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&wfull[stage]);
          mbar_arrive_expect_tx(fb, Cfg::kWBytes);
          const uint32_t sb = smem_u32(wring + size_t(stage) * Cfg::kWBytes);
          if (RS) {  // this CTA's half of the boxes, delivered to both CTAs of the pair
            if (is_vocab) {
#pragma unroll
              for (int c = 0; c < NT / 64; ++c)
                if ((c & 1) == rank)
                  tma_load_2d_multicast(sb + c * 8192, &p.tm_w, fb, n0 + c * 64, kb * 64,
                                        Cfg::kClusterMask, pol_stream);
            } else {
              tma_load_2d_multicast(sb + rank * (NT / 2) * 128, &p.tm_g, fb, kb * 64,
                                    n0 + rank * (NT / 2), Cfg::kClusterMask, pol_keep);
            }
          } else if (is_vocab) {
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
      // A shared stage is released by both CTAs; this CTA may exit only after the peer's
      // last releases have arrived on its barriers.
      if (RS && ok) {
        for (int i = 0; i < SW; ++i) {
          if (!mbar_wait_bounded(smem_u32(&wempty[stage]), phase ^ 1, p.err, abort_flag)) break;
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
      for (int sup = cid; ok && sup < n_loop; sup += ncl) {
        const int tile = RS ? sup : sup * CL + rank;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&hempty[stage]), phase ^ 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&hfull[stage]);
          mbar_arrive_expect_tx(fb, Cfg::kHBytes);
          const uint32_t sa = smem_u32(hring + size_t(stage) * Cfg::kHBytes);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (RS)
              tma_load_2d(sa, &p.tm_h, fb, kb * 64, p.row0 + rank * 128, pol_keep);
            else if (CL == 1)
              tma_load_2d(sa + mt * 16384, &p.tm_h, fb, kb * 64, p.row0 + mt * 128, pol_keep);
            else if (mt % CL == rank)  // this CTA's share, delivered to every CTA of the cluster
              tma_load_2d_multicast(sa + mt * 16384, &p.tm_h, fb, kb * 64, p.row0 + mt * 128,
                                    Cfg::kClusterMask, pol_keep);
          }
          if (++stage == SH) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Before this CTA may exit, every stage must have been released by every CTA of the
      // cluster (their releases arrive on this CTA's barriers).
      if (CL > 1 && !RS && ok) {
        for (int i = 0; i < SH; ++i) {
          if (!mbar_wait_bounded(smem_u32(&hempty[stage]), phase ^ 1, p.err, abort_flag)) break;
          if (++stage == SH) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescVocab = idesc_bf16_f32(NT, true);
      constexpr uint32_t kIdescGate = idesc_bf16_f32(NT, false);
      int ws = 0, hs = 0;
      uint32_t wph = 0, hph = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int sup = cid; ok && sup < n_loop; sup += ncl) {
        const int tile = RS ? sup : sup * CL + rank;
        const bool is_vocab = tile < p.n_vocab_tiles || tile >= n_tiles;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wfull[ws]), wph, p.err, abort_flag) ||
              !mbar_wait_bounded(smem_u32(&hfull[hs]), hph, p.err, abort_flag)) {
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
          if (RS)
            tc_commit_multicast(smem_u32(&wempty[ws]), Cfg::kClusterMask);
          else
            tc_commit(smem_u32(&wempty[ws]));
          if (CL == 1 || RS)
            tc_commit(smem_u32(&hempty[hs]));
          else
            tc_commit_multicast(smem_u32(&hempty[hs]), Cfg::kClusterMask);
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
      const size_t rbase = static_cast<size_t>(row) * p.V;
      RowStat st = rowstat_empty();
#pragma unroll 1
      for (int bt = 0; bt < 2; ++bt) {
        float x[8][8];
        int v0[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          v0[g] = chunk * kZChunk + (bt * 8 + g) * 256 + lane * 8;
          if (v0[g] < p.V) load8_stream(p.Z, is_bf16, rbase + v0[g], x[g]);
        }
        if (p.z_inv_T > 0.f)
          rowstat_fold<8, true>(st, x, v0, p.V, p.z_inv_T);
        else
          rowstat_fold<8, false>(st, x, v0, p.V, 0.f);
      }
      st = warp_combine(st, p.z_inv_T);
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
    const int row = (RS ? rank : mt) * 128 + q * 32 + lane;
    const int grow = p.row0 + row;
    const bool valid = row < p.rows && (grow % p.L) != 0;  // skip each block's verified slot
    Top16 top;
    top16_init(top);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int sup = cid; sup < n_loop; sup += ncl) {
      const int tile = RS ? sup : sup * CL + rank;
      const bool is_pad = tile >= n_tiles;
      const bool is_vocab = tile < p.n_vocab_tiles;
      const int n0 = (is_vocab ? tile : tile - p.n_vocab_tiles) * NT;
      if (!mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, p.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::kAccCols + mt * NT);
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t rr[32];
        __syncwarp();  // tcgen05.ld is warp-collective; lanes diverged on row validity
        tmem_ld_32x32b_x32(tbase + c * 32, rr);
        tmem_ld_wait();
        if (!valid || is_pad) continue;
        const int cbase = n0 + c * 32;
        if (is_vocab) {
          top16_offer32(top, rr, cbase, p.V - cbase);  // columns past V are not tokens
        } else {
          float* dst = p.gate_out + static_cast<size_t>(grow) * p.r;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (cbase + j < p.r) dst[cbase + j] = 1.0f / (1.0f + expf(-__uint_as_float(rr[j])));
          }
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
      top16_sort(top);
      // one list per CTA computing the row: per cluster for a row-split pair
      const size_t off = (static_cast<size_t>(grow) * p.G + (RS ? cid : blockIdx.x)) * kK;
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
  if (CL > 1) cluster_sync();  // no CTA leaves while a peer may still signal its barriers
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

template <int MT, int NT, int NBUF, int SW, int SH, int CL, int RS = 0>
cudaError_t launch_cfg(const LmheadParams& prm, int grid, cudaStream_t s) {
  using Cfg = LmCfg<MT, NT, NBUF, SW, SH, CL, RS>;
  auto kern = k_lmhead_tc<MT, NT, NBUF, SW, SH, CL, RS>;
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
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int MT, int NT, int NBUF, int SW, int SH>
cudaError_t launch_cluster(const LmheadParams& prm, int grid, int cl, cudaStream_t s) {
  if (cl == 4 && grid % 4 == 0) return launch_cfg<MT, NT, NBUF, SW, SH, 4>(prm, grid, s);
  if (cl >= 2 && grid % 2 == 0) return launch_cfg<MT, NT, NBUF, SW, SH, 2>(prm, grid, s);
  return launch_cfg<MT, NT, NBUF, SW, SH, 1>(prm, grid, s);
}

}  // namespace

bool lmhead_row_split(int rows_total, int variant, int G) {
  return rows_total > 128 && variant == 4 && G % 2 == 0;
}

cudaError_t launch_lmhead_tc(const LmheadLaunch& a, cudaStream_t s) {
  LmheadParams prm;
  memset(&prm, 0, sizeof(prm));
  if (!encode_bf16_2d(&prm.tm_h, a.hidden, a.d, a.rows_total, 64, 128))
    return cudaErrorInvalidValue;
  // Dummy-but-valid maps when a tile kind is not used, so every map is well formed.
  if (!encode_bf16_2d(&prm.tm_w, a.vocab ? a.W : a.hidden, a.vocab ? a.V : a.d,
                      a.vocab ? a.d : a.rows_total, 64, 64))
    return cudaErrorInvalidValue;
  prm.L = a.L;
  prm.V = a.V;
  prm.d = a.d;
  prm.r = a.r;
  const bool rs = a.vocab && lmhead_row_split(a.rows_total, a.lmhead_variant, a.G);
  prm.G = rs ? a.G / 2 : a.G;  // partial lists per row: one per CTA, or per pair when split
  prm.part_val = a.part_val;
  prm.part_idx = a.part_idx;
  prm.gate_out = a.gate_out;
  prm.err = a.err;
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
    // Row groups of up to 128 rows: one M tile x 256 vocabulary columns, double-buffered
    // TMEM. Up to 256 rows: two M tiles x 128 columns with double-buffered TMEM (variants
    // 1 and 3 differ in how the 224 KB of rings split between W and the hidden rows), or
    // x 256 columns with one TMEM buffer (variant 2), or a row-split pair (variant 4: two
    // CTAs of 128 rows x 256 columns sharing each W tile by multicast).
    const bool two = prm.rows > 128;
    const int variant = rs ? 4 : two ? (a.lmhead_variant >= 1 && a.lmhead_variant <= 3 ? a.lmhead_variant : 1) : 0;
    const int NT = (variant == 1 || variant == 3) ? 128 : 256;
    prm.n_vocab_tiles = a.vocab ? (a.V + NT - 1) / NT : 0;
    prm.n_gate_tiles = a.gate ? (a.r + NT - 1) / NT : 0;
    prm.write_partials = a.vocab ? 1 : 0;
    if (!encode_bf16_2d(&prm.tm_g, a.gate ? a.Wg : a.hidden, a.d, a.gate ? a.r : a.rows_total,
                        64, static_cast<uint32_t>(a.gate ? (variant == 4 ? NT / 2 : NT) : 128)))
      return cudaErrorInvalidValue;
    const int grid = a.vocab ? a.G : (prm.n_gate_tiles > 0 ? prm.n_gate_tiles : 1);
    cudaError_t e;
    // Clusters share the hidden rows by multicast; the gate-only launch (a tile or two)
    // runs without.
    const int cl = a.vocab ? a.cluster : 1;
    if (variant == 4)
      e = launch_cfg<1, 256, 2, 5, 4, 2, 1>(prm, grid, s);
    else if (variant == 0)
      e = launch_cluster<1, 256, 2, 5, 4>(prm, grid, cl, s);
    else if (variant == 1)
      e = launch_cluster<2, 128, 2, 8, 3>(prm, grid, cl, s);
    else if (variant == 2)
      e = launch_cluster<2, 256, 1, 4, 3>(prm, grid, cl, s);
    else
      e = launch_cluster<2, 128, 2, 6, 4>(prm, grid, cl, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dfs
