// conv2tap.cu -- two-tap dynamic depthwise convolution over draft blocks ("DFlash 2: Keep
// Drafting Parallel", §"A lightweight local convolution": its equation and Fig. 4):
//   out[b][t][c] = k0[b][t][c] x[b][t][c] + k1[b][t][c] x[b][t-1][c]     (x[b][-1] = 0)
//   kj[b][t][c]  = base[j][c] + corr[b][t][j G + c / 16],  corr[b][t] = Wc x[b][t],  G = d/16
// Two kernels:
//   k_conv_corr  -- the correction GEMM corr = X Wc^T (M = rows, N = 2G, K = d) on the tensor
//                   cores: 128 x 80 output tiles with K split over the grid (at most 8 ways)
//                   so that about one CTA per SM streams its share through an 8-stage TMA
//                   ring; one thread issues tcgen05.mma (bf16 in, fp32 in tensor memory), the
//                   four warps drain the accumulator into per-split partial sums (fp32, L2).
//   k_conv_apply -- a programmatic dependent, one block per row and 1024 channels: sums the
//                   partials in split order, forms both taps' kernels and writes the bf16
//                   output, 8 channels per thread.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace dfs {
namespace {

constexpr int kCM = 128;                      // rows per tile
constexpr int kCN = 80;                       // correction outputs per tile
constexpr int kCStages = 8;
constexpr int kCXBytes = kCM * 128;           // 128 rows x 64 k, bf16
constexpr int kCWBytes = kCN * 128;           // 80 rows x 64 k
constexpr int kCStage = kCXBytes + kCWBytes;  // 26 KB, a multiple of 1024
constexpr int kCThreads = 128;
constexpr uint32_t kCTmemCols = 128;
constexpr int kMaxSplit = 8;
constexpr size_t kCSmem = 1024 + size_t(kCStages) * kCStage + 8 * (2 * kCStages + 1) + 16;
constexpr int kApplyThreads = 128;                // one block: 128 chunks of 8 channels of a row
constexpr int kStilePitch = kCN + 1;               // fp32 staging rows: conflict-free scalar writes
static_assert(kCStage % 1024 == 0, "stages keep the 1024-byte alignment of 128-byte swizzle");
static_assert(size_t(kCM) * (kCN + 1) * 4 <= size_t(kCStages) * kCStage, "the staging tile fits in the ring");

struct ConvParams {
  CUtensorMap tm_x;  // x as [rows, d] bf16, box 64 x 128
  CUtensorMap tm_w;  // Wc as [2G, d] bf16, box 64 x 80
  float* partial;    // [n_split][rows][2G]
  int rows, n_out, n_kb, kb_per_split;
  int* err;
  unsigned long long wait_limit_ns;
};

__global__ void __launch_bounds__(kCThreads, 1) k_conv_corr(const __grid_constant__ ConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + size_t(kCStages) * kCStage);
  uint64_t* empty = full + kCStages;
  uint64_t* tfull = empty + kCStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kCN, m0 = blockIdx.y * kCM, split = blockIdx.z;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.n_kb, kb0 + p.kb_per_split);  // the host gives every split >= 1 block

  if (threadIdx.x == 0) {
    for (int st = 0; st < kCStages; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      mbar_init(smem_u32(&empty[st]), 1);
    }
    mbar_init(smem_u32(tfull), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&p.tm_x);
    prefetch_tensormap(&p.tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kCTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dependents_launch();  // k_conv_apply may start launching; it waits for this grid

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol = policy_evict_last();  // x is re-read by every output-tile column
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
      const uint32_t fb = smem_u32(&full[stage]);
      mbar_arrive_expect_tx(fb, kCStage);
      const uint32_t sx = smem_u32(ring + size_t(stage) * kCStage);
      tma_load_2d(sx, &p.tm_x, fb, kb * 64, m0, pol);
      tma_load_2d(sx + kCXBytes, &p.tm_w, fb, kb * 64, n0, pol);
      if (++stage == kCStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    // the MMAs' releases of the last stages land on this CTA's barriers before it exits
    for (int i = 0; i < kCStages; ++i) {
      if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, p.err, abort_flag, p.wait_limit_ns)) break;
      if (++stage == kCStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32(kCN, false, kCM);  // both operands K-major
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, p.err, abort_flag, p.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t sx = smem_u32(ring + size_t(stage) * kCStage);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // K = 16 per instruction: 32 bytes along the row
        tc_mma_bf16(tmem, smem_desc_sw128(sx + kk * 32, 0, 1024),
                    smem_desc_sw128(sx + kCXBytes + kk * 32, 0, 1024), kIdesc, (kb > kb0 || kk > 0));
      tc_commit(smem_u32(&empty[stage]));
      if (++stage == kCStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    tc_commit(smem_u32(tfull));
  }
  __syncwarp();
  // ---------------------------------------------------------------- epilogue (all warps)
  // tensor-memory loads are warp-collective: a warp reads only if all its lanes' waits held
  const bool ok = __all_sync(0xffffffffu,
                             mbar_wait_bounded(smem_u32(tfull), 0, p.err, abort_flag, p.wait_limit_ns));
  tc_fence_after();
  // accumulator -> shared staging tile (the ring is free: every stage has been consumed) ->
  // coalesced rows of the per-split partials
  float* stile = reinterpret_cast<float*>(ring);  // [128][kStilePitch]
  __syncthreads();
  if (ok) {
    uint32_t r[3][32];
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    tmem_ld_32x32b_x32(taddr, r[0]);
    tmem_ld_32x32b_x32(taddr + 32, r[1]);
    tmem_ld_32x32b_x32(taddr + 64, r[2]);  // columns 80..95 are read and dropped
    tmem_ld_wait();
    float* srow = stile + (warp * 32 + lane) * kStilePitch;
#pragma unroll
    for (int j = 0; j < kCN; ++j) srow[j] = __uint_as_float(r[j >> 5][j & 31]);
  }
  __syncthreads();
  if (ok) {
    const int nv4 = min(kCN, p.n_out - n0) / 4;  // float4s per row (n_out - n0 is a multiple of 8)
    for (int i = threadIdx.x; i < kCM * (kCN / 4); i += kCThreads) {
      const int rr = i / (kCN / 4), q4 = i - rr * (kCN / 4);
      const int row = m0 + rr;
      if (row >= p.rows || q4 >= nv4) continue;
      const float* sv = stile + rr * kStilePitch + 4 * q4;
      *reinterpret_cast<float4*>(p.partial + (static_cast<size_t>(split) * p.rows + row) * p.n_out + n0 +
                                 4 * q4) = make_float4(sv[0], sv[1], sv[2], sv[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kCTmemCols);
}

__global__ void __launch_bounds__(kApplyThreads) k_conv_apply(const uint16_t* __restrict__ x,
                                                              const float* __restrict__ base,
                                                              const float* __restrict__ partial,
                                                              uint16_t* __restrict__ out, int rows,
                                                              int L, int d, int n_out, int n_split) {
  // block (row, chunk block): 8 channels per thread
  const int row = blockIdx.x;
  const int c = (blockIdx.y * kApplyThreads + threadIdx.x) * 8;
  const bool live = c < d;
  const int t = row % L, g = c >> 4, G = d >> 4;
  // the inputs (not written by k_conv_corr) first, then wait for the partial sums
  uint4 xv = make_uint4(0u, 0u, 0u, 0u), pv = make_uint4(0u, 0u, 0u, 0u);
  float4 b[4];
  if (live) {
    xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * d + c));
    if (t > 0) pv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(row - 1) * d + c));
    b[0] = __ldg(reinterpret_cast<const float4*>(base + c));
    b[1] = __ldg(reinterpret_cast<const float4*>(base + c + 4));
    b[2] = __ldg(reinterpret_cast<const float4*>(base + d + c));
    b[3] = __ldg(reinterpret_cast<const float4*>(base + d + c + 4));
  }
  grid_dependency_wait();
  if (!live) return;
  float pc0[kMaxSplit], pc1[kMaxSplit];
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s)  // every split's partial, loads issued together
    if (s < n_split) {
      const float* pr = partial + (static_cast<size_t>(s) * rows + row) * n_out;
      pc0[s] = __ldcg(pr + g);
      pc1[s] = __ldcg(pr + G + g);
    }
  float c0 = 0.f, c1 = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s)  // summed in split order: the same sums on every run
    if (s < n_split) {
      c0 += pc0[s];
      c1 += pc1[s];
    }
  const float k0[8] = {b[0].x, b[0].y, b[0].z, b[0].w, b[1].x, b[1].y, b[1].z, b[1].w};
  const float k1[8] = {b[2].x, b[2].y, b[2].z, b[2].w, b[3].x, b[3].y, b[3].z, b[3].w};
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, pw[4] = {pv.x, pv.y, pv.z, pv.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float xa = bf16_bits_to_float(xw[j] & 0xFFFFu), xb = bf16_bits_to_float(xw[j] >> 16);
    const float pa = bf16_bits_to_float(pw[j] & 0xFFFFu), pb = bf16_bits_to_float(pw[j] >> 16);
    const float ya = (k0[2 * j] + c0) * xa + (k1[2 * j] + c1) * pa;
    const float yb = (k0[2 * j + 1] + c0) * xb + (k1[2 * j + 1] + c1) * pb;
    const __nv_bfloat162 v = __floats2bfloat162_rn(ya, yb);
    o[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

ConvSplit conv2tap_split(int d) {
  ConvSplit s;
  s.n_kb = d / 64;
  const int per = (s.n_kb + kMaxSplit - 1) / kMaxSplit;  // at most 8 splits, none empty
  s.kb_per_split = per;
  s.n_split = (s.n_kb + per - 1) / per;
  return s;
}

size_t conv2tap_partial_bytes(int B, int L, int d) {
  return 4 * static_cast<size_t>(conv2tap_split(d).n_split) * B * L * (d / 8);
}

cudaError_t launch_conv2tap(const ConvLaunch& a, cudaStream_t s) {
  const ConvSplit sp = conv2tap_split(a.d);
  ConvParams p{};
  const int rows = a.B * a.L;
  if (!encode_bf16_2d_tile(&p.tm_x, a.x, a.d, rows, 64, kCM)) return cudaErrorInvalidValue;
  if (!encode_bf16_2d_tile(&p.tm_w, a.Wc, a.d, a.d / 8, 64, kCN)) return cudaErrorInvalidValue;
  p.partial = a.partial;
  p.rows = rows;
  p.n_out = a.d / 8;
  p.n_kb = sp.n_kb;
  p.kb_per_split = sp.kb_per_split;
  p.err = a.err;
  p.wait_limit_ns = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs;
  static bool attr_set = false;  // raised once, so that a recorded launch makes no other call
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(k_conv_corr, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kCSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid((p.n_out + kCN - 1) / kCN, (rows + kCM - 1) / kCM, sp.n_split);
  k_conv_corr<<<grid, kCThreads, kCSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launches(1);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows), (a.d / 8 + kApplyThreads - 1) / kApplyThreads);
  cfg.blockDim = dim3(kApplyThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_conv_apply, static_cast<const uint16_t*>(a.x), a.base,
                         static_cast<const float*>(a.partial), static_cast<uint16_t*>(a.out), rows,
                         a.L, a.d, p.n_out, sp.n_split);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace dfs
