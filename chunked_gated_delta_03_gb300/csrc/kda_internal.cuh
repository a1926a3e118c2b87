// Internal declarations shared by the host API and the kernels.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "kda_ptx.cuh"

namespace kda {

constexpr int kChunk = 64;                          // rows per chunk
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // bounded waits: 2 s
constexpr uint32_t kWaitBackoffMaxNs = 64;          // longest sleep between polls of a wait
constexpr int kMaxDevicesCached = 64;               // per-device caches of launch attributes

// Sizes and chunk bookkeeping of one call, passed by value to every kernel.
struct Problem {
  int B, T, Hq, Hv, K, V;
  int N;             // sequences (B for fixed length)
  int NT;            // fixed length: chunks per sequence (ceil(T / 64)); varlen: 0
  int nc_max;        // upper bound on the chunk count (grid size)
  int varlen;        // 1 when cu_seqlens is given
  int beta_fp32;     // 1: beta is fp32, 0: bf16
  int tf32;          // 1: Aqk / Akk from TF32 operands in one MMA pass
  float scale;
  const int32_t* cu;         // varlen: cu_seqlens
  const int32_t* chunk_idx;  // varlen: [nc, 2] (sequence, chunk within sequence)
  const int32_t* chunk_off;  // varlen: [N + 1]
  const int32_t* nc_dev;     // varlen: number of chunks
  const int32_t* seq_order;  // varlen state pass: sequences by chunk count, most first
  int32_t* status;           // device status word
  int32_t* flags;            // [N * Hv]: 1 marks a chain with a chunk past the tensor-core paths' gate range
};

// One chunk: flat token row t0 (into the [B*T] token axis), L valid rows,
// its sequence n and index i within that sequence.
struct ChunkInfo {
  int n, i, t0, L;
  bool valid;
};

__device__ __forceinline__ ChunkInfo chunk_info(const Problem& P, int gc) {
  ChunkInfo c{0, 0, 0, 0, false};
  int bos, len;
  if (!P.varlen) {
    c.n = gc / P.NT;
    c.i = gc - c.n * P.NT;
    bos = c.n * P.T;
    len = P.T;
  } else {
    if (gc >= *P.nc_dev) return c;
    c.n = P.chunk_idx[2 * gc];
    c.i = P.chunk_idx[2 * gc + 1];
    bos = P.cu[c.n];
    len = P.cu[c.n + 1] - bos;
  }
  c.t0 = bos + c.i * kChunk;
  c.L = min(kChunk, len - c.i * kChunk);
  c.valid = c.L > 0;
  return c;
}

// Record the first device error (later ones are dropped).
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// Bounded mbarrier wait shared by all threads of a CTA.  After kWaitLimitNs it
// records KDA_ERR_TIMEOUT, raises the CTA's abort flag (later waits return at
// once) and returns false; the caller carries on to its normal exit.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t sleep_ns = 32;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 4; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    // back off so that waiting warps leave issue slots to working ones, but
    // briefly: a hand-off on a critical path should wake its waiter promptly
    __nanosleep(sleep_ns);
    if (sleep_ns < kWaitBackoffMaxNs) sleep_ns *= 2;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_status(status, KDA_ERR_TIMEOUT);
      return false;
    }
  }
}

// A kernel's dynamic shared memory attribute, set once per device (`dev` is
// the current device).  The cache belongs to the kernel itself (a template
// parameter), not to its type: instantiations of one kernel template share a
// type but each needs its own attribute.  It is per process and does not
// survive a cudaDeviceReset, after which the attribute would have to be set
// again.
template <auto* Kern>
cudaError_t set_smem_once(uint32_t bytes, int dev) {
  static std::atomic<uint32_t> done[kMaxDevicesCached];
  if (dev >= 0 && dev < kMaxDevicesCached && done[dev].load(std::memory_order_acquire) == bytes)
    return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevicesCached) done[dev].store(bytes, std::memory_order_release);
  return e;
}

// ---- host-side launchers (defined next to their kernels) ----
struct IntraOut {
  float* Aqk;       // fp32 [BT, Hv, 64] (may be null)
  float* Akk_inv;   // fp32 [BT, Hv, 64] (may be null)
  void* W;          // bf16 [BT, Hv, K]  (required)
  void* U;          // bf16 [BT, Hv, V]  (required)
  float* G;         // fp32 [BT, Hv, K]  (may be null)
  void* QG;         // bf16 [BT, Hv, K]: q * e^G (may be null)
  // state-pass operands (null in the standalone intra primitive)
  void* Qs;         // bf16 [BT, Hv, K]: scale * q * e^G
  void* Aqk_b;      // bf16 [BT, Hv, 64]: Aqk rounded for the output MMA
  void* Kl;         // bf16 [BT, Hv, K]: k * e^{G_last - G}, G_last of the token's chunk
  float* gamma;     // fp32 [nc_max, Hv, K]: e^{G_last}
};

struct IntraInputs {
  const void* q;     // bf16 [BT, Hq, K]
  const void* k;     // bf16 [BT, Hq, K]
  const void* v;     // bf16 [BT, Hv, V]
  const float* g;    // fp32 [BT, Hv, K]
  const void* beta;  // bf16 or fp32 [BT, Hv]
};

struct IntraMaps {
  CUtensorMap q, k, v, g;  // inputs, boxes of (D, 1, 64) rows: L2 prefetch of a whole chunk per tensor
  CUtensorMap v_sw;        // v, SWIZZLE_128B boxes of (64, 1, 64): the W/U MMA's A operand, MN-major
};

// The fused forward's maps: the intra maps' inputs plus the outputs written
// by TMA stores from token-major SWIZZLE_128B tiles, boxes of (64, 1, 64).
struct FusedMaps {
  CUtensorMap q, k, v, g, v_sw;
  CUtensorMap o, W, U;
};

struct StateMaps {
  CUtensorMap W, Qs, Aqk_b, U, Kl;
};

// Pointers of the fused forward (one kernel for the whole path).
struct FusedArgs {
  const void* q;            // bf16 [BT, Hq, K]
  const void* k;            // bf16 [BT, Hq, K]
  const float* g;           // fp32 [BT, Hv, K]
  const void* beta;         // bf16 or fp32 [BT, Hv]
  const float* h0;          // fp32 [N, Hv, K, V] or null (zeros)
  __nv_bfloat16* o;         // bf16 [BT, Hv, V]
  float* hT;                // fp32 [N, Hv, K, V] or null
  float* Aqk;               // fp32 [BT, Hv, 64] or null
  float* Akk_inv;           // fp32 [BT, Hv, 64] or null
  void* W;                  // bf16 [BT, Hv, K] or null
  void* U;                  // bf16 [BT, Hv, V] or null
  float* G;                 // fp32 [BT, Hv, K] or null
  void* QG;                 // bf16 [BT, Hv, K] or null
  int aqk_v8;               // Aqk is 32-byte aligned: its rows are written with 32-byte stores
  int o_tma, w_tma, u_tma;  // o / W / U have a store map: whole chunks leave by TMA stores
};

// Pointers of the exact path for strong gates (recomputes the flagged chains).
struct ExactArgs {
  const void* q;        // bf16 [BT, Hq, K]
  const void* k;        // bf16 [BT, Hq, K]
  const void* v;        // bf16 [BT, Hv, V]
  const float* g;       // fp32 [BT, Hv, K]
  const void* beta;     // bf16 or fp32 [BT, Hv]
  const float* h0;      // fp32 [N, Hv, K, V] or null (zeros)
  __nv_bfloat16* o;     // bf16 [BT, Hv, V] (forward only)
  float* hT;            // fp32 [N, Hv, K, V] or null
  float* Aqk;           // fp32 [BT, Hv, 64] or null
  float* Akk_inv;       // fp32 [BT, Hv, 64] or null
  void* W;              // bf16 [BT, Hv, K] or null
  void* U;              // bf16 [BT, Hv, V] or null
  float* G;             // fp32 [BT, Hv, K] or null
  void* QG;             // bf16 [BT, Hv, K] or null
  const int32_t* flags; // [N * Hv]
  int state;            // 1: the forward (o, final state); 0: the intra primitive's outputs only
};

cudaError_t launch_chunk_index(const int32_t* cu, int N, int T, int chunk, int32_t* idx, int32_t* off,
                               int32_t* nc, int32_t* status, cudaStream_t s);
cudaError_t launch_check_table(const int32_t* cu, int N, int T, int chunk, const int32_t* idx, const int32_t* off,
                               int32_t* status, cudaStream_t s);
cudaError_t launch_seq_order(const int32_t* cu, int N, int T, int chunk, int32_t* order, int32_t* status,
                             cudaStream_t s);
cudaError_t launch_intra(const Problem& P, const IntraInputs& in, const IntraOut& out, const IntraMaps& maps,
                         int dev, int sms, cudaStream_t s);
cudaError_t launch_state(const Problem& P, const StateMaps& maps, const float* gamma, const float* h0,
                         void* o, float* hT, int dev, cudaStream_t s);
cudaError_t launch_fused(const Problem& P, const FusedArgs& A, const FusedMaps& maps, int dev, cudaStream_t s);
cudaError_t launch_exact(const Problem& P, const ExactArgs& A, int dev, cudaStream_t s);
cudaError_t launch_cp_segments(int32_t* seg_cu, int B, int T, int seg_tokens, int nps, cudaStream_t s);
cudaError_t launch_cp_identity(float* h, long long nmat, int K, cudaStream_t s);
cudaError_t launch_cp_scan(const float* A, const float* Bv, const float* h0, float* S_start, float* hT, int B,
                           int nps, int Hv, int K, int dev, cudaStream_t s);

}  // namespace kda
