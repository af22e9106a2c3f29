// dfs_api.cu -- the C ABI of libdfs.so (declared in include/dfs.h): argument checks,
// workspace layout and the order of kernel launches for each entry point. Nothing here
// allocates, frees or synchronises except dfs_get_device_error.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/dfs.h"
#include "kernels.h"

namespace {

using dfs::kK;

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Tile-shape choice for calls of more than 128 rows: 0 (default) = the vocabulary-major pair
// kernel where it needs fewer passes over W, else the row-major pair kernel; 6 = always the
// vocabulary-major pair kernel (pair MMAs over 256 vocabulary entries x the drafted rows);
// 5 = always the row-major pair kernel (256 rows x 256 vocabulary columns, each CTA staging
// half of the W tile). Read from DFS_LMHEAD_VARIANT on each call, for tuning.
int lmhead_variant_override() {
  const char* s = std::getenv("DFS_LMHEAD_VARIANT");
  const int v = s != nullptr ? std::atoi(s) : 0;
  return (v == 5 || v == 6) ? v : 0;
}

struct Layout {
  size_t err, counters;
  size_t part_val, part_idx, gate;
  size_t zmax, zarg, zsum;
  size_t cand_ids, cand_U, S, path;
  size_t logits;
  size_t hq, h_scale;  // E4M3 LM head: quantised rows and their scales
  size_t rstat;        // fused tail: target-row statistics and uniforms [B*L][8]
  size_t zc;           // fused tail at T > 0: the candidates' target logits [B][L-1][16]
  size_t succ;         // fused tail, greedy path: best successors [B][L-1][16] (int2)
  size_t total;
  int G, nchunk;
};

// Everything after the verification's own checks: the LM head's width, rank and dtype.
int check_dims(const dfs_dims* d) {
  if (d == nullptr) return DFS_ERR_INVALID;
  if (d->d < 1 || d->r < 1) return DFS_ERR_INVALID;
  const int rc = dfs::check_verify_dims(d);
  if (rc != DFS_OK) return rc;
  if (d->dtype != DFS_BF16 && d->dtype != DFS_FP32) return DFS_ERR_UNSUPPORTED;
  if (d->r % 8 != 0 || d->r > dfs::kMaxRank) return DFS_ERR_UNSUPPORTED;
  if (d->dtype == DFS_BF16 && d->d % 64 != 0) return DFS_ERR_UNSUPPORTED;
  return DFS_OK;
}

// Test hook, read on each call (the workspace layout follows it): DFS_DEBUG_LMHEAD_CTAS = an
// even number from 2 to the SM count runs the persistent LM-head kernels on that many CTAs,
// so that rows get fewer partial lists for the tail to merge; unset or out of range, one CTA
// per SM.
int lmhead_ctas(int sms) {
  const char* s = std::getenv("DFS_DEBUG_LMHEAD_CTAS");
  const int v = s ? std::atoi(s) : 0;
  return (v >= 2 && v <= sms && v % 2 == 0) ? v : sms;
}

bool make_layout(const dfs_dims& d, Layout* L) {
  const int sms = lmhead_ctas(device_sm_count());
  if (sms <= 0) return false;
  // one list per CTA of the persistent LM-head grid: even, so CTA pairs tile it
  L->G = d.dtype == DFS_BF16 ? ((sms < dfs::kMaxLists ? sms : dfs::kMaxLists) / 2) * 2 : 1;
  if (L->G < 1) L->G = 1;
  L->nchunk = (d.V + dfs::kZChunk - 1) / dfs::kZChunk;
  const size_t rows = static_cast<size_t>(d.B) * d.L;
  const size_t P = static_cast<size_t>(d.L - 1);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L->err = take(16);
  L->counters = take(4 * static_cast<size_t>(d.B));
  L->part_val = take(4 * rows * L->G * kK);
  L->part_idx = take(4 * rows * L->G * kK);
  L->gate = take(4 * rows * d.r);
  L->zmax = take(4 * rows * L->nchunk);
  L->zarg = take(4 * rows * L->nchunk);
  L->zsum = take(4 * rows * L->nchunk);
  L->cand_ids = take(4 * d.B * P * kK);
  L->cand_U = take(4 * d.B * P * kK);
  L->S = take(4 * d.B * P * kK * kK);
  L->path = take(4 * d.B * P);
  L->logits = take(d.dtype == DFS_FP32 ? 4 * rows * d.V : 0);
  L->hq = take(d.dtype == DFS_BF16 ? rows * static_cast<size_t>(d.d) : 0);
  L->h_scale = take(4 * rows);
  L->rstat = take(32 * rows);
  L->zc = take(4 * d.B * P * kK);
  L->succ = take(8 * d.B * P * kK);
  L->total = off;
  return true;
}

// Partial top-16 lists per row that the LM-head kernel leaves for the tail.
int lists_per_row(const dfs_dims& d, const Layout& L) {
  return (d.dtype == DFS_BF16 &&
          dfs::lmhead_row_split(d.B * d.L, L.G)) ? L.G / 2 : L.G;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_ptrs(std::initializer_list<const void*> req, std::initializer_list<const void*> opt) {
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return DFS_ERR_INVALID;
  for (const void* p : opt)
    if (p != nullptr && !aligned16(p)) return DFS_ERR_INVALID;
  return DFS_OK;
}

int prepare(const dfs_dims* dims, void* ws, size_t ws_bytes, Layout* L) {
  int rc = check_dims(dims);
  if (rc != DFS_OK) return rc;
  if (ws == nullptr || !aligned16(ws)) return DFS_ERR_INVALID;
  if (!make_layout(*dims, L)) return DFS_ERR_CUDA;
  if (ws_bytes < L->total) return DFS_ERR_WORKSPACE;
  return DFS_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? DFS_OK : DFS_ERR_CUDA; }

thread_local cudaEvent_t g_trace_start = nullptr;
thread_local cudaEvent_t g_trace_stop = nullptr;
cudaEvent_t vocab_trace_start() { return g_trace_start; }
cudaEvent_t vocab_trace_stop() { return g_trace_stop; }

dfs::TailLaunch tail_args(const dfs_dims& d, const Layout& L, void* ws) {
  dfs::TailLaunch t{};
  t.B = d.B;
  t.L = d.L;
  t.V = d.V;
  t.r = d.r;
  t.G = L.G;
  t.dtype = d.dtype;
  t.zdtype = d.zdtype;
  t.part_val = at<float>(ws, L.part_val);
  t.part_idx = at<int>(ws, L.part_idx);
  t.gate = at<float>(ws, L.gate);
  t.zmax = at<float>(ws, L.zmax);
  t.zarg = at<int>(ws, L.zarg);
  t.zsum = at<float>(ws, L.zsum);
  t.nchunk = L.nchunk;
  t.cand_ids = at<int>(ws, L.cand_ids);
  t.cand_U = at<float>(ws, L.cand_U);
  t.S = at<float>(ws, L.S);
  t.path = at<int>(ws, L.path);
  t.counters = at<int>(ws, L.counters);
  t.err = at<int>(ws, L.err);
  t.rstat = at<float>(ws, L.rstat);
  t.zc = at<float>(ws, L.zc);
  t.succ = at<int2>(ws, L.succ);
  return t;
}

cudaError_t run_lmhead_kernels(const dfs_dims& d, const Layout& L, void* ws, const void* hidden,
                               const void* W, const void* Wg, bool vocab, bool gate, cudaStream_t s,
                               int rows, const void* Z, float T);
cudaError_t run_zreduce(const dfs_dims& d, const Layout& L, void* ws, const void* Z, float T,
                        cudaStream_t s);

// Where the target-logit row statistics are computed: 1 = by the LM-head kernel's spare
// warps (default), 0 = by the standalone reduction kernel before it. Read from DFS_Z_FUSED
// on each call, for tuning; both do the same work.
// Test hooks for the failure path, read on each call: DFS_DEBUG_WAIT_LIMIT_NS sets the limit
// of the LM-head kernels' bounded waits (unset: 1 s); DFS_DEBUG_STALL_MMA=1 keeps their MMA
// issuer idle, so that the producers' and the epilogue's waits run out.
unsigned long long debug_wait_limit_ns() {
  const char* s = std::getenv("DFS_DEBUG_WAIT_LIMIT_NS");
  const long long v = s ? std::atoll(s) : 0;
  return v > 0 ? static_cast<unsigned long long>(v) : 0ull;
}
int debug_stall_mma() {
  const char* s = std::getenv("DFS_DEBUG_STALL_MMA");
  return (s != nullptr && std::atoi(s) != 0) ? 1 : 0;
}

bool z_fused() {
  const char* s = std::getenv("DFS_Z_FUSED");
  return s == nullptr || std::atoi(s) != 0;
}

// Step a1 (+ a2 when gate): LM head, partial top-16 lists, gate rows.
// With Z != nullptr the target-logit row statistics (and the per-call counter reset) are
// produced alongside: by the tensor-core kernel's spare warps, or by the standalone
// reduction kernel on the fp32 path.
cudaError_t run_lmhead(const dfs_dims& d, const Layout& L, void* ws, const void* hidden,
                       const void* W, const void* Wg, bool vocab, bool gate, cudaStream_t s,
                       const void* Z = nullptr, float T = 0.f) {
  const int rows = d.B * d.L;
  if (Z != nullptr && (d.dtype != DFS_BF16 || !z_fused())) {
    cudaError_t ez = run_zreduce(d, L, ws, Z, T, s);
    if (ez != cudaSuccess) return ez;
  }
  if (vocab && g_trace_start != nullptr && cudaEventRecord(g_trace_start, s) != cudaSuccess)
    return cudaErrorInvalidResourceHandle;
  cudaError_t e = run_lmhead_kernels(d, L, ws, hidden, W, Wg, vocab, gate, s, rows,
                                     (d.dtype == DFS_BF16 && z_fused()) ? Z : nullptr, T);
  if (e == cudaSuccess && vocab && g_trace_stop != nullptr) e = cudaEventRecord(g_trace_stop, s);
  return e;
}

cudaError_t run_lmhead_kernels(const dfs_dims& d, const Layout& L, void* ws, const void* hidden,
                               const void* W, const void* Wg, bool vocab, bool gate, cudaStream_t s,
                               int rows, const void* Z, float T) {
  if (d.dtype == DFS_BF16) {
    dfs::LmheadLaunch a{};
    a.hidden = hidden;
    a.W = W;
    a.Wg = Wg;
    a.rows_total = rows;
    a.L = d.L;
    a.V = d.V;
    a.d = d.d;
    a.r = d.r;
    a.vocab = vocab;
    a.gate = gate;
    a.part_val = at<float>(ws, L.part_val);
    a.part_idx = at<int>(ws, L.part_idx);
    a.G = L.G;
    a.gate_out = at<float>(ws, L.gate);
    a.err = at<int>(ws, L.err);
    a.lmhead_variant = lmhead_variant_override();
    a.wait_limit_ns = debug_wait_limit_ns();
    a.stall_mma = debug_stall_mma();
    if (Z != nullptr) {
      a.Z = Z;
      a.zdtype = d.zdtype;
      a.z_rows = rows;
      a.z_nchunk = L.nchunk;
      a.z_inv_T = T > 0.f ? 1.0f / T : 0.f;
      a.zmax = at<float>(ws, L.zmax);
      a.zarg = at<int>(ws, L.zarg);
      a.zsum = at<float>(ws, L.zsum);
      a.zero_ptr = at<int>(ws, L.counters);
      a.zero_count = static_cast<int>((L.part_val - L.counters) / 4);
    }
    return dfs::launch_lmhead_tc(a, s);
  }
  dfs::LmheadSimtLaunch a{};
  a.hidden = static_cast<const float*>(hidden);
  a.W = static_cast<const float*>(W);
  a.Wg = static_cast<const float*>(Wg);
  a.rows_total = rows;
  a.L = d.L;
  a.V = d.V;
  a.d = d.d;
  a.r = d.r;
  a.vocab = vocab;
  a.gate = gate;
  a.logits_ws = at<float>(ws, L.logits);
  a.part_val = at<float>(ws, L.part_val);
  a.part_idx = at<int>(ws, L.part_idx);
  a.gate_out = at<float>(ws, L.gate);
  return dfs::launch_lmhead_simt(a, s);
}

cudaError_t run_zreduce(const dfs_dims& d, const Layout& L, void* ws, const void* Z, float T,
                        cudaStream_t s) {
  dfs::ZReduceLaunch z{};
  z.Z = Z;
  z.zdtype = d.zdtype;
  z.rows = d.B * d.L;
  z.V = d.V;
  z.nchunk = L.nchunk;
  z.inv_T = T > 0.f ? 1.0f / T : 0.f;
  z.zmax = at<float>(ws, L.zmax);
  z.zarg = at<int>(ws, L.zarg);
  z.zsum = at<float>(ws, L.zsum);
  // the per-request counters, cleared at the start of each call
  z.zero_ptr = at<int>(ws, L.counters);
  z.zero_count = static_cast<int>((L.part_val - L.counters) / 4);
  return dfs::launch_zreduce(z, s);
}

std::atomic<unsigned long long> g_launches{0};

}  // namespace

namespace dfs {
void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

int check_verify_dims(const dfs_dims* d) {
  if (d == nullptr) return DFS_ERR_INVALID;
  if (d->B < 1 || d->L < 2 || d->K < 1 || d->V < 1) return DFS_ERR_INVALID;
  if (d->zdtype != DFS_BF16 && d->zdtype != DFS_FP32) return DFS_ERR_UNSUPPORTED;
  if (d->K != kK || d->L > kMaxL || d->V < kK || d->V % 8 != 0) return DFS_ERR_UNSUPPORTED;
  if (d->V > kMaxZChunks * kZChunk) return DFS_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->B) * d->L > (1LL << 30)) return DFS_ERR_UNSUPPORTED;
  if (d->B > 65535) return DFS_ERR_UNSUPPORTED;  // requests index the tail's second grid dimension
  return DFS_OK;
}
}  // namespace dfs

extern "C" {

int dfs_version(void) { return 1; }

uint64_t dfs_launch_count(void) { return g_launches.load(); }

int dfs_set_trace_events(void* start, void* stop) {
  g_trace_start = static_cast<cudaEvent_t>(start);
  g_trace_stop = static_cast<cudaEvent_t>(stop);
  return DFS_OK;
}

const char* dfs_status_string(int status) {
  switch (status) {
    case DFS_OK: return "ok";
    case DFS_ERR_INVALID: return "invalid argument";
    case DFS_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case DFS_ERR_WORKSPACE: return "workspace too small";
    case DFS_ERR_CUDA: return "CUDA error";
    case DFS_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

size_t dfs_workspace_size(const dfs_dims* dims) {
  if (check_dims(dims) != DFS_OK) return 0;
  Layout L;
  if (!make_layout(*dims, &L)) return 0;
  return L.total;
}

int dfs_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || !aligned16(ws) || ws_bytes < 16) return DFS_ERR_INVALID;
  return cuda_rc(cudaMemsetAsync(ws, 0, ws_bytes < 4096 ? ws_bytes : 4096,
                                 static_cast<cudaStream_t>(stream)));
}

int dfs_get_device_error(void* ws, size_t ws_bytes, int* err, void* stream) {
  if (ws == nullptr || err == nullptr || ws_bytes < 16) return DFS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DFS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DFS_ERR_CUDA;
  *err = word ? DFS_ERR_TIMEOUT : DFS_OK;
  if (word) {
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return DFS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DFS_ERR_CUDA;
  }
  return DFS_OK;
}

int dfs_lmhead_topk(const dfs_dims* dims, const void* hidden, const void* W_vocab,
                    int32_t* cand_ids, float* cand_U, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if ((rc = check_ptrs({hidden, W_vocab, cand_ids, cand_U}, {})) != DFS_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = run_lmhead(*dims, L, ws, hidden, W_vocab, nullptr, true, false, s);
  if (e != cudaSuccess) return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.G = lists_per_row(*dims, L);
  t.cand_ids = cand_ids;
  t.cand_U = cand_U;
  return cuda_rc(dfs::launch_merge(t, s));
}

int dfs_pair_score(const dfs_dims* dims, const void* hidden, const void* W_g, const void* A,
                   const void* Btab, const int32_t* last_verified, const int32_t* cand_ids,
                   const float* cand_U, float* S, float* gate_opt, void* ws, size_t ws_bytes,
                   void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if ((rc = check_ptrs({hidden, W_g, A, Btab, last_verified, cand_ids, cand_U, S}, {gate_opt})) != DFS_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = run_lmhead(*dims, L, ws, hidden, nullptr, W_g, false, true, s);
  if (e != cudaSuccess) return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.A = A;
  t.Bt = Btab;
  t.x0 = last_verified;
  t.cand_ids = const_cast<int*>(cand_ids);
  t.cand_U = const_cast<float*>(cand_U);
  t.S = S;
  if ((e = dfs::launch_pair(t, s)) != cudaSuccess) return DFS_ERR_CUDA;
  if (gate_opt != nullptr) {
    const size_t row = static_cast<size_t>(dims->r) * sizeof(float);
    e = cudaMemcpy2DAsync(gate_opt, (dims->L - 1) * row, at<char>(ws, L.gate) + row, dims->L * row,
                          (dims->L - 1) * row, dims->B, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return DFS_ERR_CUDA;
  }
  return DFS_OK;
}

int dfs_path_select(const dfs_dims* dims, const float* S, const int32_t* cand_ids, int path_mode,
                    int32_t* path, float* path_score, void* stream) {
  int rc = check_dims(dims);
  if (rc != DFS_OK) return rc;
  if (path_mode != DFS_PATH_GREEDY && path_mode != DFS_PATH_VITERBI) return DFS_ERR_INVALID;
  if ((rc = check_ptrs({S, cand_ids, path}, {path_score})) != DFS_OK) return rc;
  dfs::TailLaunch t{};
  t.B = dims->B;
  t.L = dims->L;
  t.path_mode = path_mode;
  t.S = const_cast<float*>(S);
  t.cand_ids = const_cast<int*>(cand_ids);
  t.path = path;
  t.path_score = path_score;
  return cuda_rc(dfs::launch_path(t, static_cast<cudaStream_t>(stream)));
}

int dfs_verify(const dfs_dims* dims, const int32_t* path, const void* target_logits,
               float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accept_len,
               void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if (!(temperature >= 0.f) || temperature != temperature) return DFS_ERR_INVALID;
  if ((rc = check_ptrs({path, target_logits, out_tokens, accept_len}, {})) != DFS_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (run_zreduce(*dims, L, ws, target_logits, temperature, s) != cudaSuccess) return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.Z = target_logits;
  t.T = temperature;
  t.seed = seed;
  t.path = const_cast<int*>(path);
  t.out_tokens = out_tokens;
  t.accept_len = accept_len;
  if (dfs::launch_verify(t, s) != cudaSuccess) return DFS_ERR_CUDA;
  return DFS_OK;
}

int dfs_select_verify(const dfs_dims* dims, const void* hidden, const void* W_vocab,
                      const void* W_g, const void* A, const void* Btab,
                      const int32_t* last_verified, const void* target_logits, int path_mode,
                      float temperature, uint64_t seed, int32_t* path, int32_t* out_tokens,
                      int32_t* accept_len, int32_t* cand_ids_opt, float* cand_U_opt,
                      float* S_opt, float* path_score_opt, void* ws, size_t ws_bytes,
                      void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if (path_mode != DFS_PATH_GREEDY && path_mode != DFS_PATH_VITERBI &&
      path_mode != DFS_PATH_SAMPLE && path_mode != DFS_PATH_SAMPLE_JOINT)
    return DFS_ERR_INVALID;
  if (!(temperature >= 0.f) || temperature != temperature) return DFS_ERR_INVALID;
  if ((rc = check_ptrs({hidden, W_vocab, W_g, A, Btab, last_verified, target_logits, path,
                        out_tokens, accept_len},
                       {cand_ids_opt, cand_U_opt, S_opt, path_score_opt})) != DFS_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (run_lmhead(*dims, L, ws, hidden, W_vocab, W_g, true, true, s, target_logits, temperature) !=
      cudaSuccess)
    return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.G = lists_per_row(*dims, L);
  t.A = A;
  t.Bt = Btab;
  t.x0 = last_verified;
  t.Z = target_logits;
  t.T = temperature;
  t.seed = seed;
  t.path_mode = path_mode;
  if (cand_ids_opt) t.cand_ids = cand_ids_opt;
  if (cand_U_opt) t.cand_U = cand_U_opt;
  if (S_opt) t.S = S_opt;
  t.path = path;
  t.path_score = path_score_opt;
  t.out_tokens = out_tokens;
  t.accept_len = accept_len;
  if (dfs::launch_tail_fused(t, s) != cudaSuccess) return DFS_ERR_CUDA;
  return DFS_OK;
}

int dfs_quantize_rows_e4m3(const dfs_dims* dims, const void* hidden, void* q, float* scale,
                           void* stream) {
  if (dims == nullptr || dims->B < 1 || dims->L < 1 || dims->d < 8) return DFS_ERR_INVALID;
  if (dims->dtype != DFS_BF16 || dims->d % 8 != 0 ||
      static_cast<long long>(dims->B) * dims->L > (1LL << 30))
    return DFS_ERR_UNSUPPORTED;
  int rc = check_ptrs({hidden, q, scale}, {});
  if (rc != DFS_OK) return rc;
  return cuda_rc(dfs::launch_quantize_rows_e4m3(hidden, dims->B * dims->L, dims->d, q, scale,
                                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Shape and pointer checks of the E4M3 LM head: bf16 hidden states (quantised per row by
// the call), d a multiple of 128 (one stage is 128 bytes of k), Wq the packed E4M3 head
// (dfs_pack_e4m3_head) and w_scale [V] fp32, 16-byte aligned.
int check_e4m3(const dfs_dims* dims, const void* Wq, const float* w_scale) {
  if (dims->dtype != DFS_BF16 || dims->d % 128 != 0) return DFS_ERR_UNSUPPORTED;
  return check_ptrs({Wq, w_scale}, {});
}

// Quantise the rows, then the E4M3 vocabulary tiles with the bf16 gate tiles when W_g is
// given (and the target-row statistics when Z is given), one kernel launched as a
// programmatic dependent of the quantisation.
cudaError_t run_lmhead_e4m3(const dfs_dims& d, const Layout& L, void* ws, const void* hidden,
                            const void* Wq, const float* w_scale, const void* Wg, cudaStream_t s,
                            const void* Z = nullptr, float T = 0.f) {
  const int rows = d.B * d.L;
  cudaError_t e = dfs::launch_quantize_rows_e4m3(hidden, rows, d.d, at<uint8_t>(ws, L.hq),
                                                 at<float>(ws, L.h_scale), s);
  if (e != cudaSuccess) return e;
  dfs::LmheadLaunch a{};
  a.hidden = hidden;
  a.Wg = Wg;
  a.gate = Wg != nullptr;  // gate tiles (bf16) in the same kernel
  a.rows_total = rows;
  a.L = d.L;
  a.V = d.V;
  a.d = d.d;
  a.r = d.r;
  a.G = L.G;
  a.part_val = at<float>(ws, L.part_val);
  a.part_idx = at<int>(ws, L.part_idx);
  a.gate_out = at<float>(ws, L.gate);
  a.err = at<int>(ws, L.err);
  a.wait_limit_ns = debug_wait_limit_ns();
  a.stall_mma = debug_stall_mma();
  a.hq = at<uint8_t>(ws, L.hq);
  a.h_scale = at<float>(ws, L.h_scale);
  a.Wq = Wq;
  a.w_scale = w_scale;
  a.zero_ptr = at<int>(ws, L.counters);
  a.zero_count = static_cast<int>((L.part_val - L.counters) / 4);
  if (Z != nullptr) {
    a.Z = Z;
    a.zdtype = d.zdtype;
    a.z_rows = rows;
    a.z_nchunk = L.nchunk;
    a.z_inv_T = T > 0.f ? 1.0f / T : 0.f;
    a.zmax = at<float>(ws, L.zmax);
    a.zarg = at<int>(ws, L.zarg);
    a.zsum = at<float>(ws, L.zsum);
  }
  if (vocab_trace_start() != nullptr && cudaEventRecord(vocab_trace_start(), s) != cudaSuccess)
    return cudaErrorInvalidResourceHandle;
  e = dfs::launch_lmhead_e4m3(a, s);
  if (e == cudaSuccess && vocab_trace_stop() != nullptr) e = cudaEventRecord(vocab_trace_stop(), s);
  return e;
}

}  // namespace

extern "C" {

size_t dfs_e4m3_head_bytes(int V, int d) {
  if (V < 1 || d < 128 || d % 128 != 0) return 0;
  return dfs::e4m3_head_bytes(V, d);
}

int dfs_pack_e4m3_head(int V, int d, const void* Wq, void* Wq_packed, void* stream) {
  if (V < 1 || d < 128) return DFS_ERR_INVALID;
  if (d % 128 != 0 || V > dfs::kMaxZChunks * dfs::kZChunk) return DFS_ERR_UNSUPPORTED;
  const int rc = check_ptrs({Wq, Wq_packed}, {});
  if (rc != DFS_OK) return rc;
  if (overlaps(Wq, static_cast<size_t>(V) * d, Wq_packed, dfs::e4m3_head_bytes(V, d)))
    return DFS_ERR_INVALID;
  return cuda_rc(dfs::launch_pack_e4m3_head(Wq, V, d, Wq_packed, static_cast<cudaStream_t>(stream)));
}

int dfs_lmhead_topk_e4m3(const dfs_dims* dims, const void* hidden, const void* Wq,
                         const float* w_scale, int32_t* cand_ids, float* cand_U, void* ws,
                         size_t ws_bytes, void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if ((rc = check_e4m3(dims, Wq, w_scale)) != DFS_OK) return rc;
  if ((rc = check_ptrs({hidden, cand_ids, cand_U}, {})) != DFS_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (run_lmhead_e4m3(*dims, L, ws, hidden, Wq, w_scale, nullptr, s) != cudaSuccess)
    return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.G = L.G / 2;
  t.cand_ids = cand_ids;
  t.cand_U = cand_U;
  return cuda_rc(dfs::launch_merge(t, s));
}

int dfs_select_verify_e4m3(const dfs_dims* dims, const void* hidden, const void* Wq,
                           const float* w_scale, const void* W_g, const void* A,
                           const void* Btab, const int32_t* last_verified,
                           const void* target_logits, int path_mode, float temperature,
                           uint64_t seed, int32_t* path, int32_t* out_tokens,
                           int32_t* accept_len, int32_t* cand_ids_opt, float* cand_U_opt,
                           float* S_opt, float* path_score_opt, void* ws, size_t ws_bytes,
                           void* stream) {
  Layout L;
  int rc = prepare(dims, ws, ws_bytes, &L);
  if (rc != DFS_OK) return rc;
  if ((rc = check_e4m3(dims, Wq, w_scale)) != DFS_OK) return rc;
  if (path_mode != DFS_PATH_GREEDY && path_mode != DFS_PATH_VITERBI &&
      path_mode != DFS_PATH_SAMPLE && path_mode != DFS_PATH_SAMPLE_JOINT)
    return DFS_ERR_INVALID;
  if (!(temperature >= 0.f) || temperature != temperature) return DFS_ERR_INVALID;
  if ((rc = check_ptrs({hidden, W_g, A, Btab, last_verified, target_logits, path, out_tokens,
                        accept_len},
                       {cand_ids_opt, cand_U_opt, S_opt, path_score_opt})) != DFS_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (run_lmhead_e4m3(*dims, L, ws, hidden, Wq, w_scale, W_g, s, target_logits, temperature) !=
      cudaSuccess)
    return DFS_ERR_CUDA;
  dfs::TailLaunch t = tail_args(*dims, L, ws);
  t.G = L.G / 2;
  t.A = A;
  t.Bt = Btab;
  t.x0 = last_verified;
  t.Z = target_logits;
  t.T = temperature;
  t.seed = seed;
  t.path_mode = path_mode;
  if (cand_ids_opt) t.cand_ids = cand_ids_opt;
  if (cand_U_opt) t.cand_U = cand_U_opt;
  if (S_opt) t.S = S_opt;
  t.path = path;
  t.path_score = path_score_opt;
  t.out_tokens = out_tokens;
  t.accept_len = accept_len;
  if (dfs::launch_tail_fused(t, s) != cudaSuccess) return DFS_ERR_CUDA;
  return DFS_OK;
}

}  // extern "C"

// ---- two-tap dynamic depthwise convolution ----
namespace {

int check_conv(int B, int L, int d) {
  if (B < 1 || L < 1 || d < 64) return DFS_ERR_INVALID;
  // rows index the GEMM's second grid dimension in 128-row tiles (at most 65535 of them)
  if (d % 64 != 0 || d > 16384 || static_cast<long long>(B) * L > (1LL << 22)) return DFS_ERR_UNSUPPORTED;
  return DFS_OK;
}

// The error word, then the correction GEMM's per-split partial sums.
size_t conv_ws_bytes(int B, int L, int d) { return kAlign + align_up(dfs::conv2tap_partial_bytes(B, L, d)); }


}  // namespace

extern "C" {

int dfs_next_tokens(int B, int L, const int32_t* out_tokens, const int32_t* accept_len,
                    int32_t* next_last_verified, void* stream) {
  if (B < 1 || L < 1 || L > dfs::kMaxL) return DFS_ERR_INVALID;
  const int rc = check_ptrs({out_tokens, accept_len, next_last_verified}, {});
  if (rc != DFS_OK) return rc;
  return cuda_rc(dfs::launch_next_tokens(B, L, out_tokens, accept_len, next_last_verified,
                                         static_cast<cudaStream_t>(stream)));
}

size_t dfs_conv2tap_workspace_size(int B, int L, int d) {
  return check_conv(B, L, d) == DFS_OK ? conv_ws_bytes(B, L, d) : 0;
}

int dfs_conv2tap(int B, int L, int d, const void* x, const float* base, const void* Wc, void* out,
                 void* ws, size_t ws_bytes, void* stream) {
  int rc = check_conv(B, L, d);
  if (rc != DFS_OK) return rc;
  if ((rc = check_ptrs({x, base, Wc, out, ws}, {})) != DFS_OK) return rc;
  const size_t xbytes = 2 * static_cast<size_t>(B) * L * d;
  if (overlaps(x, xbytes, out, xbytes)) return DFS_ERR_INVALID;
  if (ws_bytes < conv_ws_bytes(B, L, d)) return DFS_ERR_WORKSPACE;
  dfs::ConvLaunch a{};
  a.x = x;
  a.base = base;
  a.Wc = Wc;
  a.out = out;
  a.err = at<int>(ws, 0);
  a.partial = at<float>(ws, kAlign);
  a.B = B;
  a.L = L;
  a.d = d;
  a.wait_limit_ns = debug_wait_limit_ns();
  return cuda_rc(dfs::launch_conv2tap(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
