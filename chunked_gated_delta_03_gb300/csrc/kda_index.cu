// Varlen chunk table on the device (cuLA PR #135, cula/ops/kda/index.py:
// prepare_lens / prepare_chunk_indices): for each packed sequence n with
// len_n = cu[n+1] - cu[n], the pairs (n, i) for i < ceil(len_n / chunk), in
// sequence order, and the offsets off[n] = sum_{m<n} ceil(len_m / chunk).
// One CTA: each thread owns a contiguous run of sequences, a block scan turns
// the per-thread chunk counts into offsets, then each thread writes its pairs.
// No host synchronisation: the chunk count stays on the device.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kIndexThreads = 1024;

__global__ void __launch_bounds__(kIndexThreads)
    chunk_index_kernel(const int32_t* __restrict__ cu, int N, int T, int C, int32_t* __restrict__ idx,
                       int32_t* __restrict__ off, int32_t* __restrict__ nc, int32_t* __restrict__ status) {
  __shared__ int bad;
  __shared__ int warp_total[kIndexThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
  __syncthreads();

  const int per = (N + kIndexThreads - 1) / kIndexThreads;
  const int s0 = min(N, tid * per), s1 = min(N, s0 + per);
  int local = 0, mybad = 0;
  for (int n = s0; n < s1; ++n) {
    const int len = cu[n + 1] - cu[n];
    if (len < 0) mybad = 1;
    else local += (len + C - 1) / C;
  }
  if (mybad) atomicOr(&bad, 1);

  // block-wide exclusive scan of `local`
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_total[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_total[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      *nc = 0;
      set_status(status, KDA_ERR_BAD_SEQLENS);
    }
    return;
  }
  int acc = incl - local + (warp > 0 ? warp_total[warp - 1] : 0);
  for (int n = s0; n < s1; ++n) {
    off[n] = acc;
    const int ch = (cu[n + 1] - cu[n] + C - 1) / C;
    for (int i = 0; i < ch; ++i) {
      idx[2 * (acc + i)] = n;
      idx[2 * (acc + i) + 1] = i;
    }
    acc += ch;
  }
  if (tid == kIndexThreads - 1) {
    off[N] = acc;
    *nc = acc;
  }
}

// Check of a caller-supplied chunk table against cu_seqlens, in the same
// shape as the builder above: the block scan gives the offsets the table must
// hold; only when every offset matches (so that every index below stays
// inside the table's num_chunks = off[N] rows) are the pairs compared.  Bad
// cu_seqlens set KDA_ERR_BAD_SEQLENS, a table that differs from the one
// chunk_index_kernel would build sets KDA_ERR_BAD_CHUNK_TABLE.
__global__ void __launch_bounds__(kIndexThreads)
    check_table_kernel(const int32_t* __restrict__ cu, int N, int T, int C, const int32_t* __restrict__ idx,
                       const int32_t* __restrict__ off, int32_t* __restrict__ status) {
  __shared__ int bad;  // bit 0: cu_seqlens, bit 1: the table
  __shared__ int warp_total[kIndexThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = ((cu[0] != 0 || cu[N] != T) ? 1 : 0) | (off[0] != 0 ? 2 : 0);
  __syncthreads();
  const int per = (N + kIndexThreads - 1) / kIndexThreads;
  const int s0 = min(N, tid * per), s1 = min(N, s0 + per);
  int local = 0, mybad = 0;
  for (int n = s0; n < s1; ++n) {
    const int len = cu[n + 1] - cu[n];
    if (len < 0) mybad = 1;
    else local += (len + C - 1) / C;
  }
  if (mybad) atomicOr(&bad, 1);
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_total[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_total[lane] = w;
  }
  __syncthreads();
  if (bad & 1) {
    if (tid == 0) set_status(status, KDA_ERR_BAD_SEQLENS);
    return;
  }
  int acc = incl - local + (warp > 0 ? warp_total[warp - 1] : 0);
  int offbad = 0;
  for (int n = s0; n < s1; ++n) {
    if (off[n] != acc) offbad = 1;
    acc += (cu[n + 1] - cu[n] + C - 1) / C;
  }
  if (tid == kIndexThreads - 1 && off[N] != acc) offbad = 1;
  if (offbad) atomicOr(&bad, 2);
  __syncthreads();
  if (!bad) {
    int pairbad = 0;
    for (int n = s0; n < s1; ++n) {
      const int o = off[n], ch = off[n + 1] - o;
      for (int i = 0; i < ch; ++i)
        if (idx[2 * (o + i)] != n || idx[2 * (o + i) + 1] != i) pairbad = 1;
    }
    if (pairbad) atomicOr(&bad, 2);
  }
  __syncthreads();
  if (tid == 0 && bad) set_status(status, KDA_ERR_BAD_CHUNK_TABLE);
}

// Sequences ordered by chunk count, most first (a counting sort in one CTA),
// so that the per-chain kernels (one CTA per (sequence, head) chain) start
// their longest chains in the first wave.  Order within equal counts is
// arbitrary: chains are independent, so it changes no result.  With more
// distinct counts than shared memory holds, the order is the identity.  The
// kernel also checks cu_seqlens (cu[0] = 0, non-decreasing, cu[N] = T) and
// records KDA_ERR_BAD_SEQLENS in the status word otherwise, so that a path
// that does not build the chunk table still refuses bad metadata.
constexpr int kOrderBins = 8192;

__global__ void __launch_bounds__(kIndexThreads)
    seq_order_kernel(const int32_t* __restrict__ cu, int N, int T, int C, int maxc, int32_t* __restrict__ order,
                     int32_t* __restrict__ status) {
  __shared__ int bin[kOrderBins];
  __shared__ int warp_total[kIndexThreads / 32];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
  __syncthreads();
  for (int n = tid; n < N; n += kIndexThreads)
    if (cu[n + 1] < cu[n]) bad = 1;
  __syncthreads();
  if (bad) {
    for (int n = tid; n < N; n += kIndexThreads) order[n] = n;
    if (tid == 0 && status) set_status(status, KDA_ERR_BAD_SEQLENS);
    return;
  }
  if (maxc + 1 > kOrderBins) {
    for (int n = tid; n < N; n += kIndexThreads) order[n] = n;
    return;
  }
  const int nb = maxc + 1;
  for (int b = tid; b < nb; b += kIndexThreads) bin[b] = 0;
  __syncthreads();
  for (int n = tid; n < N; n += kIndexThreads) {
    const int len = cu[n + 1] - cu[n];
    atomicAdd(&bin[len <= 0 ? 0 : min((len + C - 1) / C, maxc)], 1);
  }
  __syncthreads();
  // bin b starts after all bins with more chunks: an exclusive scan over the
  // bins in descending order, each thread owning `per` consecutive ones
  const int per = (nb + kIndexThreads - 1) / kIndexThreads;
  const int r0 = min(nb, tid * per), r1 = min(nb, r0 + per);  // ranks r: bin nb - 1 - r
  int local = 0;
  for (int r = r0; r < r1; ++r) local += bin[nb - 1 - r];
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_total[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_total[lane] = w;
  }
  __syncthreads();
  int acc = incl - local + (warp > 0 ? warp_total[warp - 1] : 0);
  for (int r = r0; r < r1; ++r) {
    const int b = nb - 1 - r, c = bin[b];
    bin[b] = acc;
    acc += c;
  }
  __syncthreads();
  for (int n = tid; n < N; n += kIndexThreads) {
    const int len = cu[n + 1] - cu[n];
    order[atomicAdd(&bin[len <= 0 ? 0 : min((len + C - 1) / C, maxc)], 1)] = n;
  }
}

}  // namespace

cudaError_t launch_seq_order(const int32_t* cu, int N, int T, int chunk, int32_t* order, int32_t* status,
                             cudaStream_t s) {
  const int maxc = (T + chunk - 1) / chunk;
  seq_order_kernel<<<1, kIndexThreads, 0, s>>>(cu, N, T, chunk, maxc, order, status);
  return cudaGetLastError();
}

cudaError_t launch_check_table(const int32_t* cu, int N, int T, int chunk, const int32_t* idx, const int32_t* off,
                               int32_t* status, cudaStream_t s) {
  check_table_kernel<<<1, kIndexThreads, 0, s>>>(cu, N, T, chunk, idx, off, status);
  return cudaGetLastError();
}

cudaError_t launch_chunk_index(const int32_t* cu, int N, int T, int chunk, int32_t* idx, int32_t* off,
                               int32_t* nc, int32_t* status, cudaStream_t s) {
  chunk_index_kernel<<<1, kIndexThreads, 0, s>>>(cu, N, T, chunk, idx, off, nc, status);
  return cudaGetLastError();
}

}  // namespace kda
