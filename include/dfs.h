/*
 * dfs.h -- C ABI of libdfs.so, the GB300 (sm_103a) draft-block select-and-verify
 * library for DFlash 2 block drafting.
 *
 * One call of dfs_select_verify runs, for each request b of a batch and each
 * draft position t of its block:
 *   (a1) the drafter's shared LM head u_t = h_t . W_vocab, keeping the 16 best
 *        (logit, token) pairs of each position;
 *   (a2) the context gate H(h_t) = sigmoid(W_g . h_t);
 *   (a3) the bilinear pair scores S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>
 *        over every adjacent candidate pair;
 *   (a4) the path: greedy best-successor traversal or Viterbi max-sum;
 *   (a5/a6) verification against the target's logits, greedy (T = 0) or by
 *        rejection sampling (T > 0).
 * Sources, by page title and section:
 *   "DFlash 2: Keep Drafting Parallel" (blog translation), sections "The right
 *     tokens are already there" (keep top-16) and "A lightweight path selector"
 *     (pair-score equation, gate, greedy traversal, rejection sampling);
 *   "DFlash 2 讓 Qwen3.8-27B 快了兩倍" section 2 (Viterbi) and section "The output is
 *     exactly the same" (greedy output equals autoregressive decoding; sampling
 *     keeps the target distribution).
 *
 * Conventions for every entry point:
 *   * Pointers named in the signatures are DEVICE pointers owned by the caller,
 *     row-major and contiguous, 16-byte aligned. The library never allocates,
 *     frees or synchronises inside these calls (dfs_get_device_error excepted);
 *     scratch space is the caller's workspace of dfs_workspace_size() bytes,
 *     16-byte aligned, initialised once with dfs_workspace_init().
 *   * `stream` is a cudaStream_t passed as void*. Work is enqueued on it and the
 *     call returns without waiting. One workspace serves one stream at a time:
 *     calls that share a workspace and may run concurrently on the GPU race.
 *   * Token ids are int32 in [0, V). Ties: among equal values the lower token id
 *     wins, in every argmax (top-K order, path steps, target argmax, draws).
 *   * K must be 16. 2 <= L <= 16, 1 <= B <= 65535 (DFS_ERR_UNSUPPORTED beyond).
 *     Block row 0 of each request holds the verified
 *     slot (the last verified token x0); rows 1..L-1 are the draft positions, so a
 *     request proposes L-1 tokens.
 *   * Return value: DFS_OK, or a negative dfs_status. Argument errors are found
 *     on the host before anything is enqueued. A device-side bounded wait that
 *     expires sets a sticky error word in the workspace, read (and cleared) by
 *     dfs_get_device_error.
 */
#ifndef DFS_H_
#define DFS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFS_OK = 0,
  DFS_ERR_INVALID = -1,     /* null pointer, bad size, misaligned pointer      */
  DFS_ERR_UNSUPPORTED = -2, /* shape or dtype outside what the kernels handle  */
  DFS_ERR_WORKSPACE = -3,   /* workspace smaller than dfs_workspace_size()     */
  DFS_ERR_CUDA = -4,        /* a CUDA launch or driver call failed             */
  DFS_ERR_TIMEOUT = -5      /* a device-side bounded wait expired (sticky)     */
} dfs_status;

/* Element type of hidden states, W_vocab, W_g and the A/B tables (dtype), and of
 * the target logits (zdtype). A dense FP16/BF16/FP32 LM head is required, as the
 * pages' selector requires a dense lm_head; BF16 runs on the tensor cores, FP32 on
 * CUDA cores (exact fp32 products, for small checkable cases). */
typedef enum { DFS_BF16 = 0, DFS_FP32 = 1 } dfs_dtype;

/* DFS_PATH_SAMPLE and DFS_PATH_SAMPLE_JOINT ("A lightweight path selector": sampling
 * draws from the same scores) are the fused call's sampled traversal and joint path draw;
 * see dfs_select_verify. */
typedef enum {
  DFS_PATH_GREEDY = 0,
  DFS_PATH_VITERBI = 1,
  DFS_PATH_SAMPLE = 2,
  DFS_PATH_SAMPLE_JOINT = 3
} dfs_path_mode;

typedef struct {
  int B;      /* requests in the batch, >= 1                                 */
  int L;      /* block length incl. the verified slot, 2..16                 */
  int K;      /* candidates kept per position; must be 16                    */
  int V;      /* vocabulary size, >= K, <= 4194304; multiple of 8            */
  int d;      /* drafter hidden width; multiple of 64 for BF16               */
  int r;      /* selector rank (A/B table width, gate width); multiple of 8, <= 512 */
  int dtype;  /* dfs_dtype of hidden, W_vocab, W_g, A, Btab                  */
  int zdtype; /* dfs_dtype of target_logits                                  */
} dfs_dims;

/* Library ABI version (currently 1). */
int dfs_version(void);

/* Static string for a dfs_status value. */
const char* dfs_status_string(int status);

/* Workspace bytes needed by any entry point for `dims` on the current device
 * (depends on the device's SM count). Returns 0 for invalid dims. */
size_t dfs_workspace_size(const dfs_dims* dims);

/* Clears the workspace's control words (error word, counters). Call once after
 * allocating a workspace, before its first use. Enqueued on `stream`. */
int dfs_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Reads the workspace's sticky device error word into *err (DFS_OK or
 * DFS_ERR_TIMEOUT), then clears it. Synchronises `stream`. */
int dfs_get_device_error(void* ws, size_t ws_bytes, int* err, void* stream);

/* Optional tracing, for timing the dominant kernel inside a running pipeline: while
 * set, every later dfs_select_verify or dfs_lmhead_topk call made from this host
 * thread records `start` (a cudaEvent_t, as void*) on its stream just before the
 * LM-head kernel and `stop` just after it. NULL, NULL disables. Host-side only. */
int dfs_set_trace_events(void* start, void* stop);

/* The number of kernels this library has launched in this process, over all calls,
 * threads and devices (launches the CUDA runtime accepted). Host-side only; never
 * fails. Differences between two reads count the kernels of the calls in between. */
uint64_t dfs_launch_count(void);

/* Step a1 -- LM head and keep top-16 ("The right tokens are already there";
 * "A lightweight path selector": U_t(b) is the drafter's own logit).
 *   hidden   [B, L, d]   dtype
 *   W_vocab  [d, V]      dtype (the shared LM head, vocabulary contiguous)
 *   cand_ids [B, L-1, 16] int32  out: for draft row t = 1..L-1 the 16 tokens with
 *            the largest logits u_t[v] = sum_k hidden[b,t,k] W_vocab[k,v], ordered by
 *            (logit desc, id asc)
 *   cand_U   [B, L-1, 16] fp32   out: their logits (fp32 accumulation)
 * The full [B*(L-1), V] logits are never written to memory. */
int dfs_lmhead_topk(const dfs_dims* dims, const void* hidden, const void* W_vocab,
                    int32_t* cand_ids, float* cand_U, void* ws, size_t ws_bytes, void* stream);

/* Steps a2 and a3 -- context gate and pair scores ("A lightweight path selector",
 * S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>).
 *   hidden        [B, L, d]  dtype; row t feeds the gate of position t
 *   W_g           [r, d]     dtype; gate g_t = sigmoid(W_g . hidden[b,t]) in fp32
 *   A, Btab       [V, r]     dtype; per-token predecessor / successor embeddings
 *   last_verified [B]        int32: x0, the predecessor of position 1
 *   cand_ids, cand_U [B, L-1, 16]  as written by dfs_lmhead_topk
 *   S       [B, L-1, 16, 16] fp32 out: S[b, t-1, a, c] = S_t(a, cand c of t), with a
 *           the a-th candidate of position t-1 for t >= 2; for t = 1 every a-row holds
 *           S_1(x0, .)
 *   gate_opt [B, L-1, r] fp32 out, or NULL: the gate values g_t */
int dfs_pair_score(const dfs_dims* dims, const void* hidden, const void* W_g, const void* A,
                   const void* Btab, const int32_t* last_verified, const int32_t* cand_ids,
                   const float* cand_U, float* S, float* gate_opt, void* ws, size_t ws_bytes,
                   void* stream);

/* Step a4 -- path over the (L-1) x 16 lattice.
 *   DFS_PATH_GREEDY ("A lightweight path selector"): x_1 = argmax_c S_1(x0, c),
 *     x_t = argmax_c S_t(x_{t-1}, c).
 *   DFS_PATH_VITERBI ("DFlash 2 讓 ..." section 2): max-sum dynamic programming,
 *     delta_t(c) = max_a [delta_{t-1}(a) + S_t(a, c)], backtracked from the best end.
 *   path       [B, L-1] int32 out: x_1..x_{L-1} (token ids)
 *   path_score [B] fp32 out, or NULL: the summed pair scores of the path */
int dfs_path_select(const dfs_dims* dims, const float* S, const int32_t* cand_ids, int path_mode,
                    int32_t* path, float* path_score, void* stream);

/* Steps a5/a6 -- verification against the target ("The output is exactly the same";
 * "A lightweight path selector": rejection sampling recovers the target distribution).
 *   target_logits [B, L, V] zdtype: row i is the target's prediction after x_i
 *                 (x_0 = last verified token)
 *   temperature == 0: greedy. y_i = argmax_v Z[b,i,v]; n = largest k <= L-1 with
 *     x_t == y_{t-1} for t <= k; emits x_1..x_n, y_n.
 *   temperature  > 0: p_i = softmax(Z[b,i]/T). x_t is accepted when U < p_{t-1}(x_t);
 *     at the first rejection the emitted token is a draw from p_{t-1} with x_t removed
 *     and renormalised; after L-1 acceptances a bonus token is drawn from p_{L-1}.
 *     Draws: Philox4x64-10 (Salmon et al., SC'11), key (seed, 0); the accept test of
 *     position t uses counter (0, t, b, 0) word 0. The draw from row t-1 (t = L for the
 *     bonus row) takes one uniform U, counter (0, t, b, 1) word 0, and emits the first
 *     token v in vocabulary order whose cumulative weight w_0 + ... + w_v exceeds U times
 *     the row's total weight, with w_v = exp(Z[b,t-1,v] / T) for v != x_t and 0 for the
 *     removed token (if rounding leaves no such token, the last token with weight).
 *     U = ((word >> 41) + 0.5) * 2^-23 (exact in fp32).
 *   out_tokens [B, L] int32 out: the emitted tokens, then -1
 *   accept_len [B] int32 out: tokens emitted, 1..L (includes the verifier's token) */
int dfs_verify(const dfs_dims* dims, const int32_t* path, const void* target_logits,
               float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accept_len,
               void* ws, size_t ws_bytes, void* stream);

/* dfs_verify without a workspace argument, for callers that cannot allocate device memory
 * at the point where they verify: a step that is handed only its input and output tensors,
 * code whose device memory pool belongs to another component, or a host thread that must
 * not enter the CUDA allocator. The pages have no counterpart; this is a packaging of
 * dfs_verify with identical results, and no allocation happens in it.
 *   Scratch: a 4 MiB device array built into the library, held by every GPU that loads the
 *   library until the process exits. The call returns DFS_ERR_WORKSPACE when the shape
 *   needs more, roughly when 12 * B * L * ceil(V / 4096) + 4 * B bytes exceed 4 MiB
 *   (B * L up to about 9000 at V = 151936).
 *   Set-up: every call asks the runtime for the array's device address on the current
 *   device (a lookup that allocates nothing), so the address stays right even after the
 *   device's context is reset and created again. The first call on a device may also load
 *   the library's device code there; make that first call before any stream capture.
 *   Sharing: all calls use the one array, which keeps the last call's contents; each call
 *   clears the counters it needs. Calls that overlap on the GPU (other streams, other host
 *   threads) race on it: issue them one after another on one stream.
 *   Arguments: as dfs_verify; of dims only B, L, K, V and zdtype are read, and they are
 *   checked exactly as dfs_verify checks them. */
int dfs_verify_noalloc(const dfs_dims* dims, const int32_t* path, const void* target_logits,
                       float temperature, uint64_t seed, int32_t* out_tokens, int32_t* accept_len,
                       void* stream);

/* The whole step, a1..a6, fused: the LM head, gate, pair scores, path and
 * verification above in one enqueue, with the same inputs and outputs.
 * cand_ids_opt, cand_U_opt, S_opt and path_score_opt may be NULL.
 * path_mode DFS_PATH_SAMPLE with temperature > 0: the traversal draws each successor,
 *   x_t ~ q_t(c) = softmax_c(S_t(x_{t-1}, c) / T) over position t's 16 candidates (Philox
 *   counter (0, t, b, 3), word 0, against the cumulative q in candidate order), and the
 *   verification is speculative sampling against that proposal: accept x_t when
 *   U < p_{t-1}(x_t) / q_t(x_t); on the first rejection emit a draw from the residual
 *   max(0, p_{t-1} - q_t) renormalised (dfs_verify's draw with these weights); when all are
 *   accepted a bonus draw from p_{L-1}.
 *   path_score_opt is then the summed scores of the drawn path. With temperature 0 the
 *   mode is DFS_PATH_GREEDY. (dfs_path_select does not take it: it has no seed.)
 * path_mode DFS_PATH_SAMPLE_JOINT with temperature > 0: the whole path is drawn from
 *   P(x_1..x_{L-1}) proportional to exp(sum_t S_t(x_{t-1}, x_t) / T), left to right from
 *   its conditionals q_t(c | x_{t-1}) proportional to exp(S_t(x_{t-1}, c) / T + log beta_t(c)),
 *   with log beta_{L-1} = 0 and log beta_t(a) = log sum_c exp(S_{t+1}(a, c) / T +
 *   log beta_{t+1}(c)) (same counters and draw as DFS_PATH_SAMPLE), and verified by
 *   speculative sampling against those conditionals, as above. With temperature 0 the mode
 *   is DFS_PATH_VITERBI (the draw's T -> 0 limit). */
int dfs_select_verify(const dfs_dims* dims, const void* hidden, const void* W_vocab,
                      const void* W_g, const void* A, const void* Btab,
                      const int32_t* last_verified, const void* target_logits, int path_mode,
                      float temperature, uint64_t seed, int32_t* path, int32_t* out_tokens,
                      int32_t* accept_len, int32_t* cand_ids_opt, float* cand_U_opt,
                      float* S_opt, float* path_score_opt, void* ws, size_t ws_bytes,
                      void* stream);

/* ---- The LM head given quantised: E4M3 (OCP 8-bit floating point) -------------------
 * The pages run top-k candidate selection through a quantised lm_head when its weights are
 * not FP16/BF16/FP32 (the RTX 5090 NVFP4 compatibility path). Here the head is E4M3 with
 * one fp32 scale per vocabulary entry, and the draft rows are quantised per row to E4M3 with
 * a power-of-two scale (exact to apply), so the product runs on the 8-bit tensor cores:
 *   u_t[v] = s_h[t] * w_scale[v] * sum_k E4M3(hq[t][k]) * E4M3(Wq[v][k])
 * Everything after the LM head (gate, pair scores, path, verification) is the bf16 step's.
 *   Wq      the head as E4M3 bytes, packed by dfs_pack_e4m3_head (dfs_e4m3_head_bytes)
 *   w_scale [V] fp32
 *   dims: dtype DFS_BF16 (hidden states, W_g, A, B), d a multiple of 128; Wq and w_scale
 *   16-byte aligned, else DFS_ERR_UNSUPPORTED / DFS_ERR_INVALID. */

/* The packed form of an E4M3 head: Wq [V, d] (row-major bytes, each vocabulary entry's d
 * weights contiguous, as a quantised checkpoint stores it) cut into tiles of 128 vocabulary
 * rows x 128 k bytes, each tile 16 KB contiguous (its 128 rows one after another), tiles
 * ordered by vocabulary block, then k block; rows past V are zeros. The LM head then reads
 * every stage of the head as one contiguous 16 KB block.
 * dfs_e4m3_head_bytes: the packed size, ceil(V / 128) * 128 * d (0 for d not a positive
 * multiple of 128). dfs_pack_e4m3_head: one kernel on `stream` from Wq (device, 16-byte
 * aligned) into Wq_packed (device, that many bytes, not overlapping Wq). Do it once per head. */
size_t dfs_e4m3_head_bytes(int V, int d);
int dfs_pack_e4m3_head(int V, int d, const void* Wq, void* Wq_packed, void* stream);

/* The row quantisation alone: hidden [B, L, d] bf16 -> q [B*L, d] E4M3 bytes and
 * scale [B*L] fp32, per row the smallest power of two 2^e with max|h| <= 448 * 2^e (448 is
 * E4M3's largest value; 1 when max|h| < 2^-100), q = E4M3(h / 2^e) rounded to nearest
 * even. d a multiple of 8. */
int dfs_quantize_rows_e4m3(const dfs_dims* dims, const void* hidden, void* q, float* scale,
                           void* stream);

/* dfs_lmhead_topk with the E4M3 head: cand_ids / cand_U as dfs_lmhead_topk, from u above. */
int dfs_lmhead_topk_e4m3(const dfs_dims* dims, const void* hidden, const void* Wq,
                         const float* w_scale, int32_t* cand_ids, float* cand_U, void* ws,
                         size_t ws_bytes, void* stream);

/* dfs_select_verify with the E4M3 head (W_vocab replaced by Wq, w_scale); same outputs. */
int dfs_select_verify_e4m3(const dfs_dims* dims, const void* hidden, const void* Wq,
                           const float* w_scale, const void* W_g, const void* A,
                           const void* Btab, const int32_t* last_verified,
                           const void* target_logits, int path_mode, float temperature,
                           uint64_t seed, int32_t* path, int32_t* out_tokens,
                           int32_t* accept_len, int32_t* cand_ids_opt, float* cand_U_opt,
                           float* S_opt, float* path_score_opt, void* ws, size_t ws_bytes,
                           void* stream);

/* Decode-loop hand-off ([Blog] Fig. 1, one draft-verify cycle after another): for each
 * request b, next_last_verified[b] = out_tokens[b][accept_len[b] - 1], the last token the
 * cycle emitted (the target's own next token), which is the next cycle's last verified token
 * x0. out_tokens [B][L] and accept_len [B] as dfs_select_verify writes them; an accept length
 * outside 1..L gives -1. Device pointers, 16-byte aligned; next_last_verified may be the
 * buffer the next cycle passes as last_verified. One kernel on `stream`. */
int dfs_next_tokens(int B, int L, const int32_t* out_tokens, const int32_t* accept_len,
                    int32_t* next_last_verified, void* stream);

/* ---- Two-tap dynamic depthwise convolution (drafter side) ----
 * "DFlash 2: Keep Drafting Parallel" §"A lightweight local convolution" (equation, Fig. 4):
 * inserted before and after each attention and MLP sublayer of the drafter, it mixes every
 * block position with its predecessor. For block b (B blocks of L rows) and position t:
 *   out[b][t][c] = k0 * x[b][t][c] + k1 * x[b][t-1][c]        (x[b][-1] = 0: row 0 is the
 *                                                             last verified token)
 *   kj = base[j][c] + corr[b][t][j * (d/16) + c / 16]         (one correction per 16 channels)
 *   corr[b][t][n] = sum_k Wc[n][k] * x[b][t][k]               (n < d/8; a linear map of the
 *                                                             position's own hidden state)
 * x: [B][L][d] bf16; base: [2][d] fp32; Wc: [d/8][d] bf16; out: [B][L][d] bf16, all device
 * memory owned by the caller, 16-byte aligned; out must not overlap x. Correction sums are
 * fp32 (tensor cores, summed over K splits in a fixed order: results repeat bit for bit);
 * the output is rounded to bf16 once. d a multiple of 64, at most 16384; L >= 1; B*L at most
 * 2^22 (DFS_ERR_UNSUPPORTED beyond).
 * ws: dfs_conv2tap_workspace_size(B, L, d) bytes (the error word and fp32 partial sums),
 * 16-byte aligned, initialised once with dfs_workspace_init; dfs_get_device_error reads its
 * error word. Asynchronous on `stream`: two kernels, the second a programmatic dependent. */
size_t dfs_conv2tap_workspace_size(int B, int L, int d);
int dfs_conv2tap(int B, int L, int d, const void* x, const float* base, const void* Wc, void* out,
                 void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFS_H_ */
