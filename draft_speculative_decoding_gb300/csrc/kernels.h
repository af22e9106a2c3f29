// kernels.h -- internal launchers of libdfs.so (host side). The C ABI in
// include/dfs.h validates arguments and lays out the workspace, then calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dfs.h"

namespace dfs {

constexpr int kK = 16;          // candidates kept per draft position
constexpr int kMaxL = 16;       // longest block handled
constexpr int kMaxRank = 512;   // widest selector rank handled
constexpr int kMaxLists = 256;  // partial top-16 lists merged per row
constexpr int kZChunk = 4096;   // target-logit elements per row-statistics unit and redraw chunk
constexpr int kMaxZChunks = 1024;  // chunks per target row handled (V <= 4194304)

// ---- a1 (+a2): LM head with fused top-16 (and gate) on the tensor cores ----
struct LmheadLaunch {
  const void* hidden;  // [rows_total, d] bf16 (rows_total = B*L)
  const void* W;       // [d, V] bf16
  const void* Wg;      // [r, d] bf16 (gate tiles), may be null when !gate
  int rows_total, L, V, d, r;
  bool vocab;          // compute the vocabulary tiles (top-16 partial lists)
  bool gate;           // compute the gate tiles
  float* part_val;     // [rows_total][G][16]
  int* part_idx;
  int G;               // grid of the vocabulary launch = lists per row
  float* gate_out;     // [rows_total][r]
  int* err;
  int lmhead_variant;  // more than 128 rows: 0 = 6 where it needs fewer passes over W,
                       // else 5; 6 = CTA pairs with pair MMAs over 256 vocabulary entries x
                       // the drafted rows of up to 2 nb requests; 5 = pair MMAs over 256-row
                       // groups (each CTA stages half of the W tile)
  // Test hooks: the limit of every bounded wait (0: the default), and a switch that keeps the
  // MMA issuer idle so that the other roles' waits run out and report DFS_ERR_TIMEOUT.
  unsigned long long wait_limit_ns;
  int stall_mma;
  // E4M3 LM head (launch_lmhead_e4m3): rows quantised by launch_quantize_rows_e4m3 and the
  // head given as E4M3 bytes [V, d] with one fp32 scale per vocabulary entry
  const void* hq;        // [rows_total, d] E4M3
  const float* h_scale;  // [rows_total]
  const void* Wq;        // E4M3 head, packed: [ceil(V/128)][d/128][128][128] bytes
  const float* w_scale;  // [V]
  // Target-logit row statistics computed by the kernel's spare warps (z_rows = 0: none).
  const void* Z;       // [z_rows, V]
  int zdtype, z_rows, z_nchunk;
  float z_inv_T;       // 0: max/argmax only
  float* zmax;         // [z_rows][z_nchunk]
  int* zarg;
  float* zsum;
  int* zero_ptr;       // counters cleared for the later kernels of the call
  int zero_count;
};
// ---- two-tap dynamic depthwise convolution (drafter side) ----
struct ConvLaunch {
  const void* x;       // [B*L, d] bf16
  const float* base;   // [2][d]
  const void* Wc;      // [d/8, d] bf16
  void* out;           // [B*L, d] bf16
  float* partial;      // [n_split][B*L][d/8] fp32 (conv2tap_partial_bytes)
  int* err;
  int B, L, d;
  unsigned long long wait_limit_ns;  // 0: the default
};
// How the correction GEMM splits K = d: n_kb blocks of 64, kb_per_split per CTA, n_split
// splits (at most 8, none empty).
struct ConvSplit {
  int n_kb, kb_per_split, n_split;
};
ConvSplit conv2tap_split(int d);
size_t conv2tap_partial_bytes(int B, int L, int d);
cudaError_t launch_conv2tap(const ConvLaunch& a, cudaStream_t s);
// Row-major bf16 matrix [outer, inner] as a TMA tensor map with an inner_box x outer_box box,
// 128-byte swizzle, zero fill outside the matrix (the LM-head kernels' encoding).
bool encode_bf16_2d_tile(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t inner_box, uint32_t outer_box);

// The shape checks every verification entry point makes (dfs_verify, dfs_verify_noalloc and,
// inside check_dims, every other call): B, L, K, V and zdtype. DFS_OK or the status to return.
int check_verify_dims(const dfs_dims* d);

// Adds n to the process-wide count of kernels this library has launched. Every launch site
// calls it once the runtime has accepted the launch; dfs_launch_count reads the total.
void note_launches(int n);

cudaError_t launch_lmhead_tc(const LmheadLaunch& a, cudaStream_t s);
// The E4M3 LM head on CTA pairs: vocabulary tiles with kind::f8f6f4 pair MMAs on the
// quantised rows, gate tiles (when gate) in bf16 from hidden and Wg, the target-row
// statistics; launched as a programmatic dependent of launch_quantize_rows_e4m3. Partial
// lists: one per CTA pair (G / 2 per row).
cudaError_t launch_lmhead_e4m3(const LmheadLaunch& a, cudaStream_t s);
// Bytes of the packed E4M3 head, and the packing of a row-major Wq [V, d] into it (each 128
// vocabulary rows x 128 k bytes one contiguous tile; tiles ordered by vocabulary block, then
// k block; rows past V zero).
size_t e4m3_head_bytes(int V, int d);
cudaError_t launch_pack_e4m3_head(const void* Wq, int V, int d, void* out, cudaStream_t s);
// Rows of h [rows, d] bf16 quantised to E4M3 with per-row power-of-two scales.
cudaError_t launch_quantize_rows_e4m3(const void* h, int rows, int d, void* q, float* scale,
                                      cudaStream_t s);
// Whether a call with these rows runs on CTA pairs that split the rows (then each row gets
// G / 2 partial lists, one per pair, instead of G).
bool lmhead_row_split(int rows_total, int G);

// ---- a1 (+a2) for fp32 inputs, on CUDA cores ----
struct LmheadSimtLaunch {
  const float* hidden;  // [rows_total, d]
  const float* W;       // [d, V]
  const float* Wg;      // [r, d]
  int rows_total, L, V, d, r;
  bool vocab, gate;
  float* logits_ws;     // [rows_total, V] scratch
  float* part_val;      // [rows_total][1][16]
  int* part_idx;
  float* gate_out;      // [rows_total][r]
};
cudaError_t launch_lmhead_simt(const LmheadSimtLaunch& a, cudaStream_t s);

// ---- target-logit row statistics (a5/a6 preparation) ----
struct ZReduceLaunch {
  const void* Z;   // [rows, V]
  int zdtype;      // 0 bf16, 1 fp32
  int rows, V, nchunk;
  float inv_T;     // 0 for greedy (max/argmax only)
  float* zmax;     // [rows][nchunk]
  int* zarg;
  float* zsum;     // [rows][nchunk] sum of exp((z - chunk max) * inv_T)
  int* zero_ptr;   // counters cleared for the later kernels of this call
  int zero_count;
};
cudaError_t launch_zreduce(const ZReduceLaunch& a, cudaStream_t s);

// ---- everything after the LM head: merge, pair scores, path, verify ----
struct TailLaunch {
  int B, L, V, r, G;
  int dtype;                 // of A/Bt
  int zdtype;
  const float* part_val;     // [B*L][G][16]
  const int* part_idx;
  const float* gate;         // [B*L][r]
  const void* A;             // [V, r]
  const void* Bt;
  const int* x0;             // [B]
  const void* Z;             // [B, L, V]
  const float* zmax;         // [B*L][nchunk]
  const int* zarg;
  const float* zsum;
  int nchunk;                // row-statistics chunks per target row
  float T;                   // 0 = greedy verification
  uint64_t seed;
  int path_mode;
  int* cand_ids;             // [B][L-1][16]
  float* cand_U;
  float* S;                  // [B][L-1][16][16]
  int* path;                 // [B][L-1]
  float* path_score;         // [B] or null
  int* out_tokens;           // [B][L]
  int* accept_len;           // [B]
  int* counters;             // [B]
  int* err;
  float* rstat;              // fused tail: [B*L][8] target-row statistics (max, argmax bits,
                             // log-sum-exp) and, at T > 0, the row's acceptance, redraw and
                             // (drawn paths) path uniforms, published by the position blocks
  float* zc;                 // fused tail at T > 0: [B][L-1][16] each candidate's target logit
                             // in its verifying row (-inf outside the vocabulary)
  int2* succ;                // fused tail, greedy path: [B][L-1][16] each predecessor's best
                             // successor (candidate index, score bits), from the position blocks
};
// Fused tail for dfs_select_verify: (L-1) x B blocks; the last block of each request
// selects its path and verifies it.
cudaError_t launch_tail_fused(const TailLaunch& a, cudaStream_t s);
cudaError_t launch_next_tokens(int B, int L, const int32_t* out_tokens, const int32_t* accept_len,
                               int32_t* next, cudaStream_t s);
// Stage launchers for the separate entry points (same device code).
cudaError_t launch_merge(const TailLaunch& a, cudaStream_t s);    // partial lists -> cand
cudaError_t launch_pair(const TailLaunch& a, cudaStream_t s);     // cand + gate -> S
cudaError_t launch_path(const TailLaunch& a, cudaStream_t s);     // S -> path
cudaError_t launch_verify(const TailLaunch& a, cudaStream_t s);   // path + Z stats -> out

}  // namespace dfs
