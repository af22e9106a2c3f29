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
//   * warp 0 issues TMA loads (hidden rows as the K-major A operand, a 64x64 box per
//     row tile; W_vocab as the MN-major B operand, vocabulary contiguous, 64x64 boxes),
//     128-byte swizzle, into a STAGES-deep ring guarded by mbarriers;
//   * warp 1 issues tcgen05.mma (M = 128 rows, N = NT vocabulary columns, K = 16 per
//     instruction) into TMEM accumulators, NBUF of them so the epilogue of one tile
//     overlaps the MMAs of the next;
//   * warps 4.. (4 per 128-row tile) drain TMEM with tcgen05.ld: each thread owns one
//     row and keeps its running top-16 in registers, inserting a logit only when it
//     beats the row's current 16th value; at the end it writes its list as one partial
//     list of the row (the tail kernel merges the G lists of a row).
//   * gate tiles use W_g [r, d] (K-major) as the B operand; their epilogue applies the
//     sigmoid and stores g[m, j] in fp32;
//   * warps 2-3 stream the target logits (16-byte loads, read once) and write per-chunk
//     row statistics (max, argmax, sum of exp) for verification, so those bytes move
//     while the tensor pipe works on W instead of in a kernel of their own.
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

template <int MT, int NT, int NBUF, int STAGES>
struct LmCfg {
  static constexpr int kABytes = MT * 128 * 128;  // MT tiles of 128 rows x 64 bf16
  static constexpr int kBBytes = NT * 128;        // NT columns x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = MT * NT;        // fp32 TMEM columns per accumulator set
  static constexpr int kTmemCols = (kAccCols * NBUF <= 32)    ? 32
                                   : (kAccCols * NBUF <= 64)  ? 64
                                   : (kAccCols * NBUF <= 128) ? 128
                                   : (kAccCols * NBUF <= 256) ? 256
                                                              : 512;
  static constexpr int kEpiWarps = 4 * MT;
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 2 * NBUF) + 16;
  static constexpr size_t kSmem = 1024 + size_t(STAGES) * kStageBytes + kBarBytes;
  static_assert(kAccCols * NBUF <= 512, "TMEM holds 512 fp32 columns");
  static_assert(NT % 64 == 0 && NT >= 64 && NT <= 256, "N tile");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void top16_insert(float (&tv)[kK], int (&ti)[kK], float x, int id) {
  // Insert (x, id) into a list sorted by value desc; x > tv[15] and id larger than every
  // id already present with an equal value (ids arrive in increasing order).
#pragma unroll
  for (int j = kK - 1; j > 0; --j) {
    const bool shift = x > tv[j - 1];
    const bool here = !shift && (x > tv[j]);
    const float nv = shift ? tv[j - 1] : (here ? x : tv[j]);
    const int ni = shift ? ti[j - 1] : (here ? id : ti[j]);
    tv[j] = nv;
    ti[j] = ni;
  }
  if (x > tv[0]) {
    tv[0] = x;
    ti[0] = id;
  }
}

template <int MT, int NT, int NBUF, int STAGES>
__global__ void __launch_bounds__(LmCfg<MT, NT, NBUF, STAGES>::kThreads, 1)
    k_lmhead_tc(const __grid_constant__ LmheadParams p) {
  using Cfg = LmCfg<MT, NT, NBUF, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(STAGES) * Cfg::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + NBUF;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NBUF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
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
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Every CTA of this persistent grid is resident now: let the dependent tail kernel launch
  // onto SMs as they free up (it waits for this grid's completion before reading).
  grid_dependents_launch();

  const int n_tiles = p.n_vocab_tiles + p.n_gate_tiles;
  const int KB = p.d / 64;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const bool is_vocab = tile < p.n_vocab_tiles;
        const int n0 = (is_vocab ? tile : tile - p.n_vocab_tiles) * NT;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          const uint32_t sa = smem_u32(smem + size_t(stage) * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            tma_load_2d(sa + mt * 16384, &p.tm_h, fb, kb * 64, p.row0 + mt * 128, pol_keep);
          if (is_vocab) {
#pragma unroll
            for (int c = 0; c < NT / 64; ++c)
              tma_load_2d(sb + c * 8192, &p.tm_w, fb, n0 + c * 64, kb * 64, pol_stream);
          } else {
            tma_load_2d(sb, &p.tm_g, fb, kb * 64, n0, pol_keep);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescVocab = idesc_bf16_f32(NT, true);
      constexpr uint32_t kIdescGate = idesc_bf16_f32(NT, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const bool is_vocab = tile < p.n_vocab_tiles;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + size_t(stage) * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
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
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
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
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------ target-logit row statistics
    if (blockIdx.x == 0 && p.zero_ptr != nullptr)
      for (int i = threadIdx.x - 64; i < p.zero_count; i += 64) p.zero_ptr[i] = 0;
    const int n_units = p.z_rows * p.z_nchunk;
    const int is_bf16 = p.zdtype == 0;
    for (int u = blockIdx.x * 2 + (warp - 2); u < n_units; u += gridDim.x * 2) {
      const int row = u / p.z_nchunk, chunk = u - row * p.z_nchunk;
      const size_t rbase = static_cast<size_t>(row) * p.V;
      RowStat st = rowstat_empty();
#pragma unroll 1
      for (int bt = 0; bt < 4; ++bt) {
        float x[4][8];
        int v0[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          v0[g] = chunk * kZChunk + (bt * 4 + g) * 256 + lane * 8;
          if (v0[g] < p.V) load8_stream(p.Z, is_bf16, rbase + v0[g], x[g]);
        }
        if (p.z_inv_T > 0.f)
          rowstat_fold<4, true>(st, x, v0, p.V, p.z_inv_T);
        else
          rowstat_fold<4, false>(st, x, v0, p.V, 0.f);
      }
      st = warp_combine(st, p.z_inv_T);
      if (lane == 0) {
        const size_t o = static_cast<size_t>(row) * p.z_nchunk + chunk;
        p.zmax[o] = st.m;
        p.zarg[o] = st.i;
        if (p.z_inv_T > 0.f) p.zsum[o] = st.s;
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- epilogue
    const int e = warp - 4;
    const int mt = e >> 2;
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = mt * 128 + q * 32 + lane;
    const int grow = p.row0 + row;
    const bool valid = row < p.rows && (grow % p.L) != 0;  // skip each block's verified slot
    float tv[kK];
    int ti[kK];
#pragma unroll
    for (int j = 0; j < kK; ++j) {
      tv[j] = -INFINITY;
      ti[j] = 0x7fffffff;
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
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
        if (!valid) continue;
        const int cbase = n0 + c * 32;
        if (is_vocab) {
          const int lim = p.V - cbase;  // columns at or past lim are outside the vocabulary
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) mx = fmaxf(mx, j < lim ? __uint_as_float(rr[j]) : -INFINITY);
          if (mx > tv[kK - 1]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float x = j < lim ? __uint_as_float(rr[j]) : -INFINITY;
              if (x > tv[kK - 1]) top16_insert(tv, ti, x, cbase + j);
            }
          }
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
      const size_t off = (static_cast<size_t>(grow) * p.G + blockIdx.x) * kK;
      float4* pv = reinterpret_cast<float4*>(p.part_val + off);
      int4* pi = reinterpret_cast<int4*>(p.part_idx + off);
#pragma unroll
      for (int j = 0; j < kK / 4; ++j) {
        pv[j] = make_float4(tv[4 * j], tv[4 * j + 1], tv[4 * j + 2], tv[4 * j + 3]);
        pi[j] = make_int4(ti[4 * j], ti[4 * j + 1], ti[4 * j + 2], ti[4 * j + 3]);
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

template <int MT, int NT, int NBUF, int STAGES>
cudaError_t launch_cfg(const LmheadParams& prm, int grid, cudaStream_t s) {
  using Cfg = LmCfg<MT, NT, NBUF, STAGES>;
  auto kern = k_lmhead_tc<MT, NT, NBUF, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

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
  prm.G = a.G;
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
    const bool two = prm.rows > 128;
    const int variant = two ? (a.lmhead_variant == 2 ? 2 : 1) : 0;
    const int NT = (variant == 1) ? 128 : 256;
    prm.n_vocab_tiles = a.vocab ? (a.V + NT - 1) / NT : 0;
    prm.n_gate_tiles = a.gate ? (a.r + NT - 1) / NT : 0;
    prm.write_partials = a.vocab ? 1 : 0;
    if (!encode_bf16_2d(&prm.tm_g, a.gate ? a.Wg : a.hidden, a.d, a.gate ? a.r : a.rows_total,
                        64, static_cast<uint32_t>(a.gate ? NT : 128)))
      return cudaErrorInvalidValue;
    const int grid = a.vocab ? a.G : (prm.n_gate_tiles > 0 ? prm.n_gate_tiles : 1);
    cudaError_t e;
    if (variant == 0)
      e = launch_cfg<1, 256, 2, 4>(prm, grid, s);
    else if (variant == 1)
      e = launch_cfg<2, 128, 2, 4>(prm, grid, s);
    else
      e = launch_cfg<2, 256, 1, 3>(prm, grid, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dfs
