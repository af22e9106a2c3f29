// lmhead_simt.cu -- the LM head, keep-top-16 and context gate for fp32 inputs, on
// CUDA cores with exact fp32 products (tensor cores have no fp32-exact mode). Used for
// small checkable cases; it materialises the logits in the workspace.
//
// Sources: "DFlash 2: Keep Drafting Parallel", sections "The right tokens are already
// there" (keep top-16) and "A lightweight path selector" (drafter logits; context gate).
#include "common.cuh"
#include "kernels.h"

namespace dfs {

namespace {

constexpr int kRowsPerBlock = 8;
constexpr int kKTile = 256;

// logits[r, v] = sum_k h[r, k] W[k, v]; one thread per vocabulary column, 8 rows per block.
__global__ void k_logits_simt(const float* __restrict__ h, const float* __restrict__ W, int rows,
                              int V, int d, float* __restrict__ logits) {
  __shared__ float hs[kRowsPerBlock][kKTile];
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  const int r0 = blockIdx.y * kRowsPerBlock;
  float acc[kRowsPerBlock];
#pragma unroll
  for (int i = 0; i < kRowsPerBlock; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < d; k0 += kKTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kRowsPerBlock * kKTile; idx += blockDim.x) {
      const int i = idx / kKTile, k = idx % kKTile;
      hs[i][k] = (r0 + i < rows && k0 + k < d) ? h[static_cast<size_t>(r0 + i) * d + k0 + k] : 0.f;
    }
    __syncthreads();
    if (v < V) {
      const int kend = min(kKTile, d - k0);
      for (int k = 0; k < kend; ++k) {
        const float w = W[static_cast<size_t>(k0 + k) * V + v];
#pragma unroll
        for (int i = 0; i < kRowsPerBlock; ++i) acc[i] = fmaf(hs[i][k], w, acc[i]);
      }
    }
  }
  if (v < V) {
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i)
      if (r0 + i < rows) logits[static_cast<size_t>(r0 + i) * V + v] = acc[i];
  }
}

// Top-16 of one logits row (skipping each block's verified slot): every thread keeps a
// register list over a strided slice, then one warp merges the 256 lists.
__global__ void k_row_top16(const float* __restrict__ logits, int V, int L, float* part_val,
                            int* part_idx) {
  const int row = blockIdx.x;
  if (row % L == 0) return;
  __shared__ float sv[256][kK + 1];
  __shared__ int si[256][kK + 1];
  float tv[kK];
  int ti[kK];
#pragma unroll
  for (int j = 0; j < kK; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0x7fffffff;
  }
  const float* x = logits + static_cast<size_t>(row) * V;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float z = x[v];
    if (z > tv[kK - 1]) {
#pragma unroll
      for (int j = kK - 1; j > 0; --j) {
        const bool shift = z > tv[j - 1];
        const bool here = !shift && (z > tv[j]);
        const float nv = shift ? tv[j - 1] : (here ? z : tv[j]);
        const int ni = shift ? ti[j - 1] : (here ? v : ti[j]);
        tv[j] = nv;
        ti[j] = ni;
      }
      if (z > tv[0]) {
        tv[0] = z;
        ti[0] = v;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kK; ++j) {
    sv[threadIdx.x][j] = tv[j];
    si[threadIdx.x][j] = ti[j];
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  // tournament over the 256 sorted lists: lane owns lists lane + 32*s
  int head[8];
  float hv[8];
  int hi[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    head[s] = 0;
    hv[s] = sv[lane + 32 * s][0];
    hi[s] = si[lane + 32 * s][0];
  }
  float* ov = part_val + static_cast<size_t>(row) * kK;
  int* oi = part_idx + static_cast<size_t>(row) * kK;
  for (int k = 0; k < kK; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, bs = -1;
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
      const float ovv = __shfl_xor_sync(0xffffffffu, wv, off);
      const int oii = __shfl_xor_sync(0xffffffffu, wi, off);
      if (ranks_before(ovv, oii, wv, wi)) {
        wv = ovv;
        wi = oii;
      }
    }
    if (bs >= 0 && bi == wi && bv == wv) {
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s == bs) {
          ++head[s];
          hv[s] = head[s] < kK ? sv[lane + 32 * s][head[s]] : -INFINITY;
          hi[s] = head[s] < kK ? si[lane + 32 * s][head[s]] : 0x7fffffff;
        }
    }
    if (lane == 0) {
      ov[k] = wv;
      oi[k] = wi;
    }
  }
}

// g[row, j] = sigmoid(sum_k Wg[j, k] h[row, k]); one warp per (row, j).
__global__ void k_gate_simt(const float* __restrict__ h, const float* __restrict__ Wg, int rows,
                            int L, int d, int r, float* __restrict__ gate) {
  const int row = blockIdx.x;
  if (row % L == 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* hr = h + static_cast<size_t>(row) * d;
  for (int j = warp; j < r; j += blockDim.x >> 5) {
    const float* w = Wg + static_cast<size_t>(j) * d;
    float acc = 0.f;
    for (int k = lane; k < d; k += 32) acc = fmaf(w[k], hr[k], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) gate[static_cast<size_t>(row) * r + j] = 1.0f / (1.0f + expf(-acc));
  }
}

}  // namespace

cudaError_t launch_lmhead_simt(const LmheadSimtLaunch& a, cudaStream_t s) {
  if (a.vocab) {
    dim3 grid((a.V + 255) / 256, (a.rows_total + kRowsPerBlock - 1) / kRowsPerBlock);
    k_logits_simt<<<grid, 256, 0, s>>>(a.hidden, a.W, a.rows_total, a.V, a.d, a.logits_ws);
    k_row_top16<<<a.rows_total, 256, 0, s>>>(a.logits_ws, a.V, a.L, a.part_val, a.part_idx);
  }
  if (a.gate) k_gate_simt<<<a.rows_total, 256, 0, s>>>(a.hidden, a.Wg, a.rows_total, a.L, a.d, a.r, a.gate_out);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launches((a.vocab ? 2 : 0) + (a.gate ? 1 : 0));
  return e;
}

}  // namespace dfs
