// verify_noalloc.cu -- dfs_verify_noalloc: the verification step (target-row statistics,
// then greedy or rejection-sampling acceptance with the redraw) with its scratch memory
// built into the library instead of passed in by the caller.
//
// It exists for callers that cannot allocate device memory at the point where they verify:
// code running inside a serving loop whose memory pool is owned by another component,
// plugins handed only the input and output tensors of one step, or a host thread that must
// not enter the CUDA allocator (which can synchronise the device). Such a caller passes its
// inputs and outputs and nothing else.
//
// The scratch is one file-scope device array of kScratchBytes. Every GPU that loads the
// library holds it until the process exits. All calls share it and it keeps the last
// call's contents; the counters that must start at zero are cleared by the first kernel of
// each call. Calls whose work overlaps on the GPU (different streams, or different host
// threads) race on the array: issue them in order on one stream.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dfs.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr size_t kAlign = 256;

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

inline size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// The device address of g_verify_scratch on the current device. In host code the array's
// name only stands in for the symbol; the address a kernel can use comes from the runtime,
// asked on every call with the caller's device current (a lookup that allocates nothing), so
// it is never stale, even after the device's context has been reset and created again.
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess) return nullptr;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int dfs_verify_noalloc(const dfs_dims* d, const int32_t* path,
                                  const void* target_logits, float temperature, uint64_t seed,
                                  int32_t* out_tokens, int32_t* accept_len, void* stream) {
  // the same shape checks as dfs_verify, then the same argument checks
  const int rc = dfs::check_verify_dims(d);
  if (rc != DFS_OK) return rc;
  if (!(temperature >= 0.f)) return DFS_ERR_INVALID;
  if (path == nullptr || target_logits == nullptr || out_tokens == nullptr || accept_len == nullptr)
    return DFS_ERR_INVALID;
  if (!aligned16(path) || !aligned16(target_logits) || !aligned16(out_tokens) ||
      !aligned16(accept_len))
    return DFS_ERR_INVALID;

  const size_t B = static_cast<size_t>(d->B);
  const size_t rows = B * static_cast<size_t>(d->L);
  const int nchunk = (d->V + dfs::kZChunk - 1) / dfs::kZChunk;
  // Layout inside the array: the counters first (cleared by the first kernel of each call).
  size_t off = 0;
  const size_t o_cnt = off;
  off = up(off + 4 * B);
  const size_t zero_end = off;
  const size_t o_zmax = off;
  off = up(off + 4 * rows * nchunk);
  const size_t o_zarg = off;
  off = up(off + 4 * rows * nchunk);
  const size_t o_zsum = off;
  off = up(off + 4 * rows * nchunk);
  const size_t o_err = off;
  off = up(off + 16);
  if (off > kScratchBytes) return DFS_ERR_WORKSPACE;  // the built-in scratch is too small

  char* base = static_cast<char*>(scratch_on_current_device());
  if (base == nullptr) return DFS_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  dfs::ZReduceLaunch z{};
  z.Z = target_logits;
  z.zdtype = d->zdtype;
  z.rows = static_cast<int>(rows);
  z.V = d->V;
  z.nchunk = nchunk;
  z.inv_T = temperature > 0.f ? 1.0f / temperature : 0.f;
  z.zmax = reinterpret_cast<float*>(base + o_zmax);
  z.zarg = reinterpret_cast<int*>(base + o_zarg);
  z.zsum = reinterpret_cast<float*>(base + o_zsum);
  z.zero_ptr = reinterpret_cast<int*>(base + o_cnt);
  z.zero_count = static_cast<int>(zero_end / 4);
  if (dfs::launch_zreduce(z, s) != cudaSuccess) return DFS_ERR_CUDA;

  dfs::TailLaunch t{};
  t.B = d->B;
  t.L = d->L;
  t.V = d->V;
  t.zdtype = d->zdtype;
  t.Z = target_logits;
  t.zmax = z.zmax;
  t.zarg = z.zarg;
  t.zsum = z.zsum;
  t.nchunk = nchunk;
  t.T = temperature;
  t.seed = seed;
  t.path = const_cast<int*>(path);
  t.out_tokens = out_tokens;
  t.accept_len = accept_len;
  t.counters = reinterpret_cast<int*>(base + o_cnt);
  t.err = reinterpret_cast<int*>(base + o_err);
  if (dfs::launch_verify(t, s) != cudaSuccess) return DFS_ERR_CUDA;
  return DFS_OK;
}
