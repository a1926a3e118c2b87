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

// Sequences ordered by chunk count, most first (a counting sort in one CTA),
// so that the state pass, one CTA per (sequence, head) chain, starts its
// longest chains in the first wave.  Order within equal counts is arbitrary:
// chains are independent, so it changes no result.  With more distinct counts
// than shared memory holds, the order is the identity.
constexpr int kOrderBins = 8192;

__global__ void __launch_bounds__(kIndexThreads)
    seq_order_kernel(const int32_t* __restrict__ cu, int N, int C, int maxc, int32_t* __restrict__ order) {
  __shared__ int bin[kOrderBins];
  __shared__ int warp_total[kIndexThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

cudaError_t launch_seq_order(const int32_t* cu, int N, int T, int chunk, int32_t* order, cudaStream_t s) {
  const int maxc = (T + chunk - 1) / chunk;
  seq_order_kernel<<<1, kIndexThreads, 0, s>>>(cu, N, chunk, maxc, order);
  return cudaGetLastError();
}

cudaError_t launch_chunk_index(const int32_t* cu, int N, int T, int chunk, int32_t* idx, int32_t* off,
                               int32_t* nc, int32_t* status, cudaStream_t s) {
  chunk_index_kernel<<<1, kIndexThreads, 0, s>>>(cu, N, T, chunk, idx, off, nc, status);
  return cudaGetLastError();
}

}  // namespace kda
