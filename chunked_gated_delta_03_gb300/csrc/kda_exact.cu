// Exact path for strong gates.  The tensor-core kernels form each intra-chunk
// decay factor e^{G_r - G_i} as the product of the operands q e^{G_r} (or
// k e^{G_r}) and k e^{-G_i}; e^{-G_i} leaves the fp32 range once a chunk's
// log-decay on a channel is large, so those kernels mark the (sequence, value
// head) chain of such a chunk in a flag array instead of trusting their
// numbers.  This kernel, launched after them, recomputes every marked chain
// from its inputs in FP32 on CUDA cores, in the steps of the chunked form
// (cuLA PR #131, Summary: intra-chunk matrices, FP32 inverse of (I + Akk),
// W/U recompute; cuLA REPO_LAYOUT.md: chunk_delta_h.py, fwd_o.py) with every
// decay factor taken as one exponential of a non-positive exponent:
//   Aqk[r][i] = scale sum_c q_r[c] k_i[c] e^{G_r[c] - G_i[c]}   (i <= r)
//   Akk[r][i] = beta_r sum_c k_r[c] k_i[c] e^{G_r[c] - G_i[c]}  (i < r)
//   X = (I + Akk)^-1, W = X diag(beta) (K e^G), U = X diag(beta) V
//   Delta = U - W S,  o = scale (Q e^G) S + Aqk Delta,
//   S <- Diag(e^{G_last}) S + (K e^{G_last - G})^T Delta.
// Every factor is at most 1, so any gate gives finite numbers.  Unmarked
// chains return at once: the launch costs one flag read per CTA.
//
// One CTA of 256 threads per chain.  The chunk's q, k (fp32), G, W (then O),
// v (then U, then Delta) live in shared memory as [64][max(K,V)+1] fp32 tiles
// (the odd row stride keeps column walks conflict-free), Aqk, beta Akk and X as
// [64][65]; S stays in registers, thread (v, part) holding rows
// part * K/TP .. + K/TP of column v, TP = 256 / V threads per column.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kExactThreads = 256;

template <int K, int V>
struct ExactLayout {
  static constexpr int kS = (K > V ? K : V) + 1;  // fp32 row stride of the 64-row tiles
  static constexpr int kA = 65;                    // fp32 row stride of the 64 x 64 tiles
  static constexpr uint32_t Q = 0;                 // q, then Qg = q e^G
  static constexpr uint32_t Kt = Q + 64 * kS * 4;  // k, then Kl = k e^{G_last - G}
  static constexpr uint32_t G = Kt + 64 * kS * 4;  // G, the in-chunk inclusive cumsum of g
  static constexpr uint32_t W = G + 64 * kS * 4;   // W, then O / scale-free partial sums
  static constexpr uint32_t U = W + 64 * kS * 4;   // v, then U, then Delta
  static constexpr uint32_t AQ = U + 64 * kS * 4;  // Aqk (with scale)
  static constexpr uint32_t AK = AQ + 64 * kA * 4; // beta Akk, strictly lower
  static constexpr uint32_t X = AK + 64 * kA * 4;  // (I + beta Akk)^-1
  static constexpr uint32_t BETA = X + 64 * kA * 4;
  static constexpr uint32_t bytes = BETA + 64 * 4;
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ float bf16_at(const void* p, size_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

template <int K, int V>
__global__ void __launch_bounds__(kExactThreads, 1) exact_kernel(const Problem P, const ExactArgs A) {
  using Lay = ExactLayout<K, V>;
  constexpr int kS = Lay::kS, kA = Lay::kA;
  constexpr int TP = kExactThreads / V;  // threads per value column
  constexpr int KR = K / TP;             // state rows per thread
  static_assert(kExactThreads % V == 0 && K % TP == 0 && 64 % TP == 0, "thread split");
  const int chain = blockIdx.x;
  const int n = chain / P.Hv, hv = chain - n * P.Hv;
  // the flag and the status word are final: the kernels that write them ran
  // before this one on the stream
  if (n >= P.N || A.flags[chain] == 0 || *P.status != 0) return;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float* sQ = reinterpret_cast<float*>(smem_raw + Lay::Q);
  float* sK = reinterpret_cast<float*>(smem_raw + Lay::Kt);
  float* sG = reinterpret_cast<float*>(smem_raw + Lay::G);
  float* sW = reinterpret_cast<float*>(smem_raw + Lay::W);
  float* sU = reinterpret_cast<float*>(smem_raw + Lay::U);
  float* sAQ = reinterpret_cast<float*>(smem_raw + Lay::AQ);
  float* sAK = reinterpret_cast<float*>(smem_raw + Lay::AK);
  float* sX = reinterpret_cast<float*>(smem_raw + Lay::X);
  float* sB = reinterpret_cast<float*>(smem_raw + Lay::BETA);
  const int tid = threadIdx.x;
  const int v = tid % V, part = tid / V, kb = part * KR;
  int bos, len;
  if (P.varlen) {
    bos = P.cu[n];
    len = P.cu[n + 1] - bos;
  } else {
    bos = n * P.T;
    len = P.T;
  }
  const int hq = hv / (P.Hv / P.Hq);
  const size_t hrow = (size_t(n) * P.Hv + hv) * K;
  float S[KR];
#pragma unroll
  for (int j = 0; j < KR; ++j) S[j] = (A.state && A.h0) ? A.h0[(hrow + kb + j) * V + v] : 0.f;
  const int nch = (len + kChunk - 1) / kChunk;
  for (int c = 0; c < nch; ++c) {
    const int t0 = bos + c * kChunk, L = min(kChunk, len - c * kChunk);
    // ---- the chunk's inputs (rows past its end zero)
    for (int idx = tid; idx < 64 * K; idx += kExactThreads) {
      const int r = idx / K, cc = idx - r * K;
      float qv = 0.f, kv = 0.f, gv = 0.f;
      if (r < L) {
        const size_t tq = (size_t(t0 + r) * P.Hq + hq) * K + cc;
        qv = bf16_at(A.q, tq);
        kv = bf16_at(A.k, tq);
        gv = A.g[(size_t(t0 + r) * P.Hv + hv) * K + cc];
      }
      sQ[r * kS + cc] = qv;
      sK[r * kS + cc] = kv;
      sG[r * kS + cc] = gv;
    }
    for (int idx = tid; idx < 64 * V; idx += kExactThreads) {
      const int r = idx / V, cc = idx - r * V;
      sU[r * kS + cc] = r < L ? bf16_at(A.v, (size_t(t0 + r) * P.Hv + hv) * V + cc) : 0.f;
    }
    if (tid < 64) {
      const size_t bi = size_t(t0 + tid) * P.Hv + hv;
      sB[tid] = tid < L ? (P.beta_fp32 ? reinterpret_cast<const float*>(A.beta)[bi] : bf16_at(A.beta, bi)) : 0.f;
    }
    __syncthreads();
    // ---- inclusive cumsum of g down the chunk (rows past the end add nothing)
    for (int cc = tid; cc < K; cc += kExactThreads) {
      float acc = 0.f;
      for (int r = 0; r < 64; ++r) {
        acc += sG[r * kS + cc];
        sG[r * kS + cc] = acc;
        if (A.G && r < L) A.G[(size_t(t0 + r) * P.Hv + hv) * K + cc] = acc;
      }
    }
    __syncthreads();
    // ---- Aqk and beta Akk, each decay factor one exponential of G_r - G_i <= 0
    for (int idx = tid; idx < 64 * 64; idx += kExactThreads) {
      const int r = idx >> 6, i = idx & 63;
      float sq = 0.f, sk = 0.f;
      if (i <= r && r < L) {
        for (int cc = 0; cc < K; ++cc) {
          const float e = expf(sG[r * kS + cc] - sG[i * kS + cc]);
          const float ki = sK[i * kS + cc] * e;
          sq = fmaf(sQ[r * kS + cc], ki, sq);
          sk = fmaf(sK[r * kS + cc], ki, sk);
        }
      }
      const float aq = (i <= r && r < L) ? P.scale * sq : 0.f;
      sAQ[r * kA + i] = aq;
      sAK[r * kA + i] = (i < r && r < L) ? sB[r] * sk : 0.f;
      if (A.Aqk && r < L) A.Aqk[(size_t(t0 + r) * P.Hv + hv) * 64 + i] = aq;
    }
    __syncthreads();
    // ---- X = (I + beta Akk)^-1 by forward substitution, thread = column j
    if (tid < 64) {
      const int j = tid;
      float x[64];
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        float acc = r == j ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) acc = fmaf(-sAK[r * kA + i], x[i], acc);
        x[r] = acc;
        sX[r * kA + j] = acc;
        if (A.Akk_inv && r < L) A.Akk_inv[(size_t(t0 + r) * P.Hv + hv) * 64 + j] = acc;
      }
    }
    __syncthreads();
    // ---- W = X diag(beta) (K e^G) and U = X diag(beta) V, thread = output column
    for (int col = tid; col < K + V; col += kExactThreads) {
      const bool isw = col < K;
      const int cc = isw ? col : col - K;
      float b[64];
#pragma unroll
      for (int j = 0; j < 64; ++j)
        b[j] = sB[j] * (isw ? sK[j * kS + cc] * expf(sG[j * kS + cc]) : sU[j * kS + cc]);
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j <= r; ++j) acc = fmaf(sX[r * kA + j], b[j], acc);
        if (isw) {
          sW[r * kS + cc] = acc;
          if (A.W && r < L)
            reinterpret_cast<__nv_bfloat16*>(A.W)[(size_t(t0 + r) * P.Hv + hv) * K + cc] = __float2bfloat16_rn(acc);
        } else {
          sU[r * kS + cc] = acc;
          if (A.U && r < L)
            reinterpret_cast<__nv_bfloat16*>(A.U)[(size_t(t0 + r) * P.Hv + hv) * V + cc] = __float2bfloat16_rn(acc);
        }
      }
    }
    __syncthreads();
    // ---- the state pass's operands in place: Qg = q e^G, Kl = k e^{G_last - G}
    for (int idx = tid; idx < 64 * K; idx += kExactThreads) {
      const int r = idx / K, cc = idx - r * K;
      const float gr = sG[r * kS + cc];
      const float qg = sQ[r * kS + cc] * expf(gr);
      sQ[r * kS + cc] = qg;
      sK[r * kS + cc] *= expf(sG[63 * kS + cc] - gr);
      if (A.QG && r < L)
        reinterpret_cast<__nv_bfloat16*>(A.QG)[(size_t(t0 + r) * P.Hv + hv) * K + cc] = __float2bfloat16_rn(qg);
    }
    __syncthreads();
    if (!A.state) continue;
    // ---- Delta = U - W S: each thread's partial sums over its state rows,
    // subtracted part by part (a fixed order, so the result is deterministic)
    float p[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < KR; ++j) acc = fmaf(sW[r * kS + kb + j], S[j], acc);
      p[r] = acc;
    }
    __syncthreads();  // every W read is done before W's tile takes O below
#pragma unroll 1
    for (int ph = 0; ph < TP; ++ph) {
      if (part == ph)
#pragma unroll
        for (int r = 0; r < 64; ++r) sU[r * kS + v] -= p[r];
      __syncthreads();
    }
    // ---- O: scale (Qg S) summed part by part into W's tile, then + Aqk Delta
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < KR; ++j) acc = fmaf(sQ[r * kS + kb + j], S[j], acc);
      p[r] = acc;
    }
#pragma unroll 1
    for (int ph = 0; ph < TP; ++ph) {
      if (part == ph)
#pragma unroll
        for (int r = 0; r < 64; ++r) sW[r * kS + v] = (ph == 0 ? 0.f : sW[r * kS + v]) + p[r];
      __syncthreads();
    }
    for (int r = part; r < L; r += TP) {
      float acc = P.scale * sW[r * kS + v];
      for (int i = 0; i <= r; ++i) acc = fmaf(sAQ[r * kA + i], sU[i * kS + v], acc);
      A.o[(size_t(t0 + r) * P.Hv + hv) * V + v] = __float2bfloat16_rn(acc);
    }
    // ---- S <- Diag(e^{G_last}) S + Kl^T Delta
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      float acc = expf(sG[63 * kS + kb + j]) * S[j];
      for (int r = 0; r < 64; ++r) acc = fmaf(sK[r * kS + kb + j], sU[r * kS + v], acc);
      S[j] = acc;
    }
    __syncthreads();  // the next chunk's loads overwrite the tiles
  }
  if (A.state && A.hT) {
#pragma unroll
    for (int j = 0; j < KR; ++j) A.hT[(hrow + kb + j) * V + v] = S[j];
  }
}

template <int K, int V>
cudaError_t launch_exact_t(const Problem& P, const ExactArgs& A, int dev, cudaStream_t s) {
  constexpr uint32_t smem = ExactLayout<K, V>::bytes;
  cudaError_t e = set_smem_once<exact_kernel<K, V>>(smem, dev);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)P.N * P.Hv;
  if (grid <= 0) return cudaSuccess;
  exact_kernel<K, V><<<unsigned(grid), kExactThreads, smem, s>>>(P, A);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_exact(const Problem& P, const ExactArgs& A, int dev, cudaStream_t s) {
  if (P.K == 128 && P.V == 128) return launch_exact_t<128, 128>(P, A, dev, s);
  if (P.K == 128 && P.V == 64) return launch_exact_t<128, 64>(P, A, dev, s);
  if (P.K == 64 && P.V == 128) return launch_exact_t<64, 128>(P, A, dev, s);
  if (P.K == 64 && P.V == 64) return launch_exact_t<64, 64>(P, A, dev, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
