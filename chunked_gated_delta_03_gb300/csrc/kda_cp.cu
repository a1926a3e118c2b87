// Intra-card context parallelism for long chains (cuLA PR #135, file list:
// cula/ops/kda/sm100/cp/pre_scan.py): a sequence is cut into segments of a
// fixed number of chunks, each segment runs as its own chain, and the state
// each segment starts from comes from a scan over the segments.  Per chunk,
// the state update of the chunked form is affine in the state,
//   S <- Diag(e^{G_last}) S + Kl^T (U - W S) = (Diag(e^{G_last}) - Kl^T W) S + Kl^T U,
// so a segment maps its start state to its end state as S -> A S + B, with A
// the segment's K x K transition (its end state from the identity with U = 0,
// which needs K = V) and B its end state from zero.  The forward kernels
// compute both (two passes over the segments); these kernels build the
// segment table, the identity start states, and the scan
//   S_start(seg 0) = h0,  S_start(seg s + 1) = A_s S_start(s) + B_s,
// whose last value is the sequence's final state.  A third forward pass from
// the scanned start states writes the outputs.
#include "kda_internal.cuh"

namespace kda {

namespace {

// seg_cu[b * nps + s] = first token of segment s of sequence b, seg_cu[B * nps] = B T
__global__ void cp_segments_kernel(int32_t* seg_cu, int B, int T, int seg_tokens, int nps) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= B * nps; i += gridDim.x * blockDim.x) {
    const int b = i / nps, s = i - b * nps;
    seg_cu[i] = i == B * nps ? B * T : b * T + min(s * seg_tokens, T);
  }
}

// h[seg][hv] = I (K x K)
__global__ void cp_identity_kernel(float* h, long long nmat, int K) {
  const long long total = nmat * K * K;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long e = i % ((long long)K * K);
    h[i] = (e / K == e % K) ? 1.f : 0.f;
  }
}

// The scan over one (sequence, value head)'s nps segments in FP32, split by
// columns: the columns of S evolve independently (S <- A S + B mixes rows
// only), so CTA (sequence, head, column block) carries kCW columns through all
// segments.  A: [B * nps, Hv, K, K] transitions, Bv: [B * nps, Hv, K, K] end
// states from zero, h0: [B, Hv, K, K] or null; writes its columns of S_start
// [B * nps, Hv, K, K] and hT [B, Hv, K, K] (if not null).  The segment's A
// (row stride K + 4 floats) and the S columns (stride kCW + 4) live in shared
// memory; each of the 256 threads owns a TR x 2 tile of the product.
constexpr int kCW = 16;

template <int K>
__global__ void __launch_bounds__(256) cp_scan_kernel(const float* A, const float* Bv, const float* h0,
                                                      float* S_start, float* hT, int nps, int Hv) {
  constexpr int LA = K + 4, LS = kCW + 4, TR = K / 32;  // 32 row groups x 8 column pairs = 256 threads
  extern __shared__ __align__(16) float sm_f[];
  float* sA = sm_f;            // [K][LA]
  float* sS = sm_f + K * LA;   // [K][LS]
  constexpr int nblk = K / kCW;
  const int cb = blockIdx.x % nblk, bh = blockIdx.x / nblk;
  const int b = bh / Hv, hv = bh - b * Hv;
  const int col0 = cb * kCW;
  const int tid = threadIdx.x, r0 = TR * (tid >> 3), c0 = 2 * (tid & 7);
  for (int i = tid; i < K * kCW; i += blockDim.x) {
    const int r = i / kCW, c = i - r * kCW;
    sS[r * LS + c] = h0 ? h0[((size_t(b) * Hv + hv) * K + r) * K + col0 + c] : 0.f;
  }
  __syncthreads();
  for (int s = 0; s < nps; ++s) {
    const size_t m = ((size_t(b) * nps + s) * Hv + hv) * K * K;  // (segment, head) matrix
    for (int i = tid; i < K * kCW; i += blockDim.x) {
      const int r = i / kCW, c = i - r * kCW;
      S_start[m + size_t(r) * K + col0 + c] = sS[r * LS + c];
    }
    for (int i = tid; i < K * K / 4; i += blockDim.x) {
      const int r = (4 * i) / K, c = 4 * i - r * K;
      *reinterpret_cast<float4*>(sA + r * LA + c) = *reinterpret_cast<const float4*>(A + m + 4 * size_t(i));
    }
    __syncthreads();
    // columns col0 + c0, + 1 of S <- A S + B, rows r0 .. r0 + TR - 1
    float acc[TR][2];
#pragma unroll
    for (int i = 0; i < TR; ++i) {
      const float2 bv = *reinterpret_cast<const float2*>(Bv + m + size_t(r0 + i) * K + col0 + c0);
      acc[i][0] = bv.x;
      acc[i][1] = bv.y;
    }
#pragma unroll 8
    for (int jj = 0; jj < K; ++jj) {
      const float2 sv = *reinterpret_cast<const float2*>(sS + jj * LS + c0);
#pragma unroll
      for (int i = 0; i < TR; ++i) {
        const float av = sA[(r0 + i) * LA + jj];
        acc[i][0] = fmaf(av, sv.x, acc[i][0]);
        acc[i][1] = fmaf(av, sv.y, acc[i][1]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TR; ++i) *reinterpret_cast<float2*>(sS + (r0 + i) * LS + c0) = make_float2(acc[i][0], acc[i][1]);
    __syncthreads();
  }
  if (hT)
    for (int i = tid; i < K * kCW; i += blockDim.x) {
      const int r = i / kCW, c = i - r * kCW;
      hT[((size_t(b) * Hv + hv) * K + r) * K + col0 + c] = sS[r * LS + c];
    }
}

}  // namespace

cudaError_t launch_cp_segments(int32_t* seg_cu, int B, int T, int seg_tokens, int nps, cudaStream_t s) {
  cp_segments_kernel<<<1, 256, 0, s>>>(seg_cu, B, T, seg_tokens, nps);
  return cudaGetLastError();
}

cudaError_t launch_cp_identity(float* h, long long nmat, int K, cudaStream_t s) {
  if (nmat <= 0) return cudaSuccess;
  cp_identity_kernel<<<256, 256, 0, s>>>(h, nmat, K);
  return cudaGetLastError();
}

cudaError_t launch_cp_scan(const float* A, const float* Bv, const float* h0, float* S_start, float* hT, int B,
                           int nps, int Hv, int K, int dev, cudaStream_t s) {
  const int grid = B * Hv * (K / kCW);
  if (grid <= 0) return cudaSuccess;
  if (K == 128) {
    constexpr uint32_t smem = (128 * (128 + 4) + 128 * (kCW + 4)) * 4;
    cudaError_t e = set_smem_once<cp_scan_kernel<128>>(smem, dev);
    if (e != cudaSuccess) return e;
    cp_scan_kernel<128><<<grid, 256, smem, s>>>(A, Bv, h0, S_start, hT, nps, Hv);
  } else if (K == 64) {
    constexpr uint32_t smem = (64 * (64 + 4) + 64 * (kCW + 4)) * 4;
    cudaError_t e = set_smem_once<cp_scan_kernel<64>>(smem, dev);
    if (e != cudaSuccess) return e;
    cp_scan_kernel<64><<<grid, 256, smem, s>>>(A, Bv, h0, S_start, hT, nps, Hv);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kda
