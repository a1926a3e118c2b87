/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked KDA forward library (libkda.so).
 *
 * KDA (Kimi Delta Attention) is the delta rule with a per-channel forget gate.
 * Per value head, with state S in R^{K x V}, each token t applies
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * The library computes it chunk by chunk (chunk = 64 tokens), in the modular
 * order of cuLA REPO_LAYOUT.md (cula/kda/chunk_fwd.py, chunk_intra.py, then
 * ops/chunk_delta_h.py and ops/fwd_o.py) and of cuLA PR #131 (Summary: the
 * intra-chunk matrices, the FP32 inverse of (I + Akk), the W/U recompute):
 *   1. in-chunk inclusive cumsum of the log-gates, G;
 *   2. Aqk[r,i] = scale sum_c q_r[c] k_i[c] e^{G_r[c]-G_i[c]} (i <= r) and
 *      Akk[r,i] = beta_r sum_c k_r[c] k_i[c] e^{G_r[c]-G_i[c]} (i < r);
 *   3. Akk_inv = (I + Akk)^{-1} in FP32;
 *   4. W = Akk_inv (beta * k * e^G), U = Akk_inv (beta * v);
 *   5. per chunk in order: Delta = U - W S, O = scale (q * e^G) S + Aqk Delta,
 *      S <- Diag(e^{G_last}) S + (k * e^{G_last - G})^T Delta.
 *
 * Conventions for every entry point
 *   - Pointers marked (device) are CUDA device pointers on the current device;
 *     all tensors are dense, contiguous and token-major:
 *       q, k      bf16 [B, T, Hq, K]
 *       v         bf16 [B, T, Hv, V]
 *       g         fp32 [B, T, Hv, K]   (log-gates, already activated)
 *       beta      bf16 or fp32 [B, T, Hv]
 *       o         bf16 [B, T, Hv, V]
 *       Aqk, Akk_inv  fp32 [B, T, Hv, 64]  (row t holds row t - t0 of its
 *                     chunk's 64 x 64 matrix; columns past the chunk's valid
 *                     rows are zero)
 *       W         bf16 [B, T, Hv, K];  U bf16 [B, T, Hv, V]
 *       G         fp32 [B, T, Hv, K]   (in-chunk cumsum of g)
 *       initial_state / final_state  fp32 [N, Hv, K, V], N = B (fixed length)
 *                     or the number of packed sequences (varlen)
 *   - Packed varlen (cuLA PR #131, Summary): pass cu_seqlens (int32 [N+1],
 *     cu[0] = 0, non-decreasing, cu[N] = T) and B = 1.
 *   - Grouped-value heads: Hv % Hq == 0; value head hv reads q/k head hv / (Hv / Hq).
 *   - Supported sizes: chunk == 64; K, V in {64, 128}; T >= 0; Hq, Hv >= 1.
 *   - Every base address must be 16-byte aligned (TMA); the workspace 256-byte.
 *   - Ownership: the caller owns every buffer, outputs and workspace included.
 *     The library allocates no device memory, keeps no state between calls,
 *     and performs no host<->device synchronisation; all work is enqueued on
 *     `stream` in order.  Calls on different streams with different
 *     workspaces are independent.  The one exception is
 *     kda_chunk_fwd_static_scratch (below): its workspace is a fixed array in
 *     the library's device image, shared by every call, and the library keeps
 *     that array's address per device.  Per-device facts (compute capability,
 *     SM count, the kernels' shared memory attribute) are queried once and
 *     cached for the life of the process.
 *   - Errors: host-side argument checks return a negative kda_status before
 *     anything is enqueued.  Errors found on the device (bad cu_seqlens, a
 *     bounded wait that ran out) are written to the status word at the start
 *     of the workspace; read it with kda_get_device_status.  No entry point
 *     throws, aborts or traps.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kda_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* Gate range.  The tensor-core kernels form each decay factor e^{G_r - G_i}
 * (G the in-chunk cumulative log-gate) as the product of the operands
 * q e^{G_r} and k e^{-G_i}.  Both stay normal fp32 numbers while a chunk's
 * total log-decay on every channel, -G at its last row, is at most this
 * bound.  A (sequence, value head) chain with a chunk past it is marked by
 * those kernels and recomputed, in the same call, by an exact FP32 path that
 * takes every decay factor as one exponential of a non-positive exponent
 * (slower: it runs on CUDA cores, one CTA per marked chain), so any gate
 * gives valid outputs.  Gates of the form -softplus(x)/16 decay a few units
 * per chunk and never take that path. */
#define KDA_MAX_CHUNK_LOG_DECAY 60.0f

enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID = -1,      /* null pointer, bad dimension or inconsistent argument */
  KDA_ERR_UNSUPPORTED = -2,  /* chunk != 64, K or V outside {64, 128}, sizes past 32-bit indexing */
  KDA_ERR_MISALIGNED = -3,   /* a base address is not 16-byte aligned (256 for workspace) */
  KDA_ERR_ARCH = -4,         /* current device is not compute capability 10.3 (sm_103) */
  KDA_ERR_LAUNCH = -5,       /* a CUDA launch or tensor-map encode failed */
  KDA_ERR_WORKSPACE = -6,    /* workspace smaller than kda_workspace_size() */
  KDA_ERR_BAD_SEQLENS = -16, /* (device) cu_seqlens not 0..T and non-decreasing */
  KDA_ERR_TIMEOUT = -17,     /* (device) a bounded wait inside a kernel ran out */
  KDA_ERR_GATE_RANGE = -18,  /* reserved: no call reports it (chains past the gate range take the exact path) */
  KDA_ERR_BAD_CHUNK_TABLE = -19 /* (device) a caller-supplied chunk table does not match cu_seqlens */
};

/* Which kernels kda_chunk_fwd runs (KdaArgs.path).
 *   KDA_PATH_AUTO      the fused forward, or the two-pass forward when the TF32
 *                      option is set (only the two-pass kernels implement it).
 *   KDA_PATH_FUSED     one kernel, one CTA per (sequence, value head) chain:
 *                      the intra-chunk steps of chunk c+1 run next to the state
 *                      and output steps of chunk c on the same SM, so the
 *                      state pass's operands never reach HBM.  Chains are
 *                      sequential over chunks; the path suits N * Hv of at
 *                      least the SM count and long sequences.
 *   KDA_PATH_TWO_PASS  a persistent intra-chunk kernel over all (chunk, head)
 *                      items, then a state/output kernel over the chains; the
 *                      state pass's operands go through the workspace.
 * Both paths compute the same quantities with the same bf16/fp32 rounding
 * points; their results agree within the accuracy bars, not bit for bit. */
enum kda_path { KDA_PATH_AUTO = 0, KDA_PATH_FUSED = 1, KDA_PATH_TWO_PASS = 2 };

enum kda_dtype { KDA_DTYPE_BF16 = 0, KDA_DTYPE_FP32 = 1 };

/* Arguments of kda_chunk_fwd and kda_fwd_intra (the latter ignores the state
 * fields and o).  Output pointers that are NULL are not written. */
typedef struct KdaArgs {
  /* inputs (device) */
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  int32_t beta_dtype;          /* enum kda_dtype */
  const int32_t* cu_seqlens;   /* NULL = fixed length */
  int32_t N;                   /* number of packed sequences (ignored when cu_seqlens is NULL) */
  int32_t B, T, Hq, Hv, K, V;
  int32_t chunk;               /* must be 64 */
  float scale;
  const float* initial_state;  /* NULL = zeros */
  /* outputs (device) */
  void* o;                     /* required by kda_chunk_fwd */
  float* final_state;          /* optional */
  float* Aqk;                  /* optional for kda_chunk_fwd, required for kda_fwd_intra */
  float* Akk_inv;              /* optional for kda_chunk_fwd, required for kda_fwd_intra */
  void* W;                     /* optional for kda_chunk_fwd, required for kda_fwd_intra */
  void* U;                     /* optional for kda_chunk_fwd, required for kda_fwd_intra */
  float* G;                    /* optional (both entry points) */
  /* optional instrumentation: host array of 3 cudaEvent_t recorded on
   * `stream` (kda_chunk_fwd).  Two-pass path: before the intra-chunk kernel,
   * after it, and after the state/output kernel.  Fused path: before and after
   * the fused kernel, the third right after the second.  NULL = no events. */
  void* const* profile_events;
  /* optional output (both entry points; NULL = not written): the gated query
   * QG = q * e^G, bf16 [B, T, Hv, K], row t of value head hv from q of its
   * q/k head and the in-chunk cumsum G of the value head's gates (the
   * "optional QG" of cuLA PR #131, Summary).  Rounded from the FP32 product. */
  void* QG;
  /* Precision option of the intra-chunk products (both entry points).  0:
   * Aqk and Akk from bf16 hi/lo operand pairs in three MMA passes (relative
   * L2 error of Akk_inv near 1e-6 against FP64).  Nonzero: one MMA pass on
   * TF32 operands rounded to nearest, a few per cent faster, with Akk_inv
   * near 5e-5 and Aqk near 3e-4 (the pages' SM100 path keeps TF32 conversion
   * points, cuLA PR #131, Numerical behavior).  o, the final state, W and U
   * stay within the same bars either way. */
  int32_t intra_tf32;
  /* enum kda_path (kda_chunk_fwd; kda_fwd_intra ignores it).  Fused with the
   * TF32 option is KDA_ERR_UNSUPPORTED. */
  int32_t path;
  /* Optional varlen chunk table built earlier by kda_prepare_chunk_indices (or
   * by the caller, in its format), reused instead of being rebuilt on every call
   * (the pages cache it for the same reason, cuLA PR #135 review of
   * cula/ops/kda/index.py).  Device int32: chunk_indices [num_chunks, 2] pairs
   * (sequence, chunk within sequence) in sequence order, chunk_offsets [N + 1]
   * with chunk_offsets[N] = num_chunks.  Both NULL: built on the device into the
   * workspace.  Both set: checked on the device against cu_seqlens before any
   * kernel reads them; a mismatch sets KDA_ERR_BAD_CHUNK_TABLE and no output is
   * written.  Only one of the two set is KDA_ERR_INVALID. */
  const int32_t* chunk_indices;
  const int32_t* chunk_offsets;
  /* Intra-card context parallelism (kda_chunk_fwd; cuLA PR #135, file list:
   * cula/ops/kda/sm100/cp/pre_scan.py).  0: off.  n > 0: every sequence is cut
   * into segments of n chunks that run as chains of their own: a first pass
   * gives each segment's end state from zero, a second its K x K state
   * transition (from the identity, with v = 0), a scan over the segments
   * gives each one's start state and the sequence's final state, and a third
   * pass from those start states writes the outputs.  Three passes over the
   * data for n-fold more chains: it pays when N * Hv is far below the SM count
   * and sequences are long (one 16k-token sequence with 8 heads).  Needs
   * fixed-length input (cu_seqlens NULL), K == V, the fused path and no TF32
   * option (else KDA_ERR_UNSUPPORTED); kda_workspace_size covers its buffers
   * (three [B * segments, Hv, K, V] fp32 state arrays and two [B * T, Hv, V] bf16
   * tiles).  The device status reports the last pass. */
  int32_t cp_chunks;
} KdaArgs;

typedef KdaArgs KdaFwdArgs;
typedef KdaArgs KdaIntraArgs;

/* Bytes of device workspace a call with these arguments needs (0 on invalid
 * arguments).  Depends on the sizes and on whether W and U are NULL (the
 * workspace then holds them for the state pass), never on tensor contents. */
size_t kda_workspace_size(const KdaArgs* args);

/* Complete chunked KDA forward: o, final_state and any requested
 * intermediates.  Steps 1-5 above; the varlen chunk table is built on the
 * device (as kda_prepare_chunk_indices does) inside the workspace.  The pages'
 * own combined forward is cuLA PR #131 (Summary, sequence diagram: intra ->
 * inverse -> W/U) followed by the delta-H and output kernels of cuLA
 * REPO_LAYOUT.md. */
int kda_chunk_fwd(const KdaArgs* args, void* workspace, size_t workspace_bytes, kda_stream_t stream);

/* The standalone intra-chunk primitive (cuLA PR #135, which exposes
 * chunk_kda_fwd_intra): steps 1-4 only, writing Aqk, Akk_inv, W, U (all
 * required) and G (optional). */
int kda_fwd_intra(const KdaArgs* args, void* workspace, size_t workspace_bytes, kda_stream_t stream);

/* Varlen chunk metadata on the device (cuLA PR #135, cula/ops/kda/index.py:
 * prepare_chunk_indices).  From cu_seqlens (device int32 [N+1]) writes
 *   chunk_indices  (device int32 [T/chunk + N, 2]): pairs (sequence, chunk
 *                  within sequence) in sequence order; rows >= num_chunks are
 *                  left untouched;
 *   chunk_offsets  (device int32 [N+1]): offsets[n] = chunks in sequences < n;
 *   num_chunks     (device int32 [1]);
 *   status         (device int32 [1]): set to KDA_ERR_BAD_SEQLENS (and
 *                  num_chunks to 0) when cu[0] != 0, cu is decreasing
 *                  anywhere, or cu[N] != T; left unchanged otherwise.
 * chunk <= 0 returns KDA_ERR_INVALID (the pages reject a chunk size of None,
 * zero or below zero, cuLA PR #135 review of the index tests).  N == 0 gives
 * num_chunks = 0 and offsets = {0}. */
int kda_prepare_chunk_indices(const int32_t* cu_seqlens, int32_t N, int32_t T, int32_t chunk,
                              int32_t* chunk_indices, int32_t* chunk_offsets, int32_t* num_chunks,
                              int32_t* status, kda_stream_t stream);

/* Reads the device status word at the start of `workspace` after the work
 * enqueued on `stream` so far has finished (synchronises that stream), and
 * stores it in *status_out (KDA_OK or a device error code).  Returns KDA_OK,
 * or KDA_ERR_INVALID / KDA_ERR_LAUNCH when it could not read it. */
int kda_get_device_status(const void* workspace, kda_stream_t stream, int32_t* status_out);

/* Check of the bounded waits every kernel uses.  Launches one warp that waits
 * on a shared-memory barrier nothing ever arrives at, through the same
 * bounded wait as the kernels: after its limit (2 s) the wait gives up, the
 * warp records KDA_ERR_TIMEOUT in *device_status (device int32 [1], first error
 * kept) and returns, and the context stays usable.  Returns KDA_OK once the
 * launch is enqueued on `stream`, or KDA_ERR_INVALID / KDA_ERR_ARCH /
 * KDA_ERR_LAUNCH.  The pages have no counterpart; it exists so that the
 * failure path can be exercised without faulting the GPU. */
int kda_check_bounded_wait(int32_t* device_status, kda_stream_t stream);

/* Bytes of the fixed device scratch behind kda_chunk_fwd_static_scratch. */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/* kda_chunk_fwd without a caller-supplied workspace, for callers that cannot
 * allocate device memory: plug-ins handed only input and output buffers by a
 * host runtime that owns the device's memory pool, and latency-critical code
 * that must not allocate.  The pages have no counterpart of this entry point.
 *   - The workspace is a fixed 64 MiB (KDA_STATIC_SCRATCH_BYTES) array in the
 *     library's device image, held on every GPU that loads the library until
 *     the process exits.  Nothing is allocated per call.
 *   - Problems whose kda_workspace_size(args) exceeds KDA_STATIC_SCRATCH_BYTES
 *     are rejected with KDA_ERR_WORKSPACE before any work is enqueued.  The
 *     fused path needs only a status header and, in varlen mode, the chunk
 *     metadata (a few bytes per sequence and chunk), so any problem the other
 *     entry points accept fits; the two-pass path (KdaArgs.path, or the TF32
 *     option) keeps its state-pass operands there, which at K = V = 128 limits
 *     it to about 57,000 token-heads with W and U NULL, about 103,000 with W
 *     and U supplied.
 *   - The first call on a device looks up the array's device address (once
 *     per device, on the current device); make that first call before any
 *     stream capture.  The address is cached per process and device and does
 *     not survive a cudaDeviceReset: after a reset, do not call this entry
 *     point on that device again in the same process.
 *   - All calls share the one array, which keeps the last call's contents:
 *     calls whose GPU work overlaps (other streams, other host threads) race
 *     on it and must be serialised by the caller.  Each call resets the status
 *     word it needs before its kernels run.
 *   - device_status (optional, device int32 [1]): receives the device status
 *     word of this call (enqueued on `stream`), as kda_get_device_status would
 *     read it from a workspace.
 * Arguments, outputs and error codes are otherwise those of kda_chunk_fwd. */
int kda_chunk_fwd_static_scratch(const KdaArgs* args, int32_t* device_status, kda_stream_t stream);

/* Static text for a status code. */
const char* kda_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
