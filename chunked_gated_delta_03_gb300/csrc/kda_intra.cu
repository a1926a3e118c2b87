// Intra-chunk kernel: one CTA per (chunk, value head).
//
// Steps (the intra-chunk part of cuLA PR #131, Summary: the intra-chunk
// matrices, the FP32 inverse of (I + Akk), the W/U recompute):
//   1. TMA loads q, k (head hv / (Hv/Hq)), v, g (head hv) for the 64 rows of
//      the chunk; rows past the chunk's L valid rows are treated as zero.
//   2. CUDA cores: inclusive cumsum G of g down the rows (two row halves, the
//      second offset by the first half's sum), then the gated operands
//      Qg = q*e^G, Kg = k*e^G, Kd = k*e^{-G}, each split into bf16 hi + lo
//      parts, written into K-major SWIZZLE_128B tiles:
//        A1 = [Qg; Kg] (128 x K), B1 = Kd (64 x K).
//   3. tcgen05 (M=128, N=64): D1 = A1_hi B1_hi^T + A1_hi B1_lo^T + A1_lo B1_hi^T,
//      an ~FP32-accurate product (residual ~2^-17 relative).  Rows 0-63 of D1
//      are Aqk / scale, rows 64-127 are Akk / beta, both before masking.
//   4. Aqk rows: scale, causal mask (i <= r), store fp32 (optional) and a bf16
//      copy for the state pass.  Akk rows: beta_r, strict mask (i < r), to
//      shared memory; two warps invert (I + Akk) by forward substitution in
//      FP32, one column of the inverse per thread.
//   5. tcgen05 (M=128, N=64, K=64): W^T = (beta*Kg)^T Akk_inv^T and
//      U^T = (beta*v)^T Akk_inv^T, read back per channel and stored as bf16.
// For the state pass it also writes Qs = scale*q*e^G (bf16, token-major),
// Kl^T = (k*e^{G_last-G})^T (bf16, per chunk) and gamma = e^{G_last} (fp32).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kIntraThreads = 128;
constexpr int kAkkLd = 68;  // fp32 row stride of the Akk tile (conflict-free float4 rows)

template <int K, int V>
struct IntraLayout {
  static constexpr uint32_t A1_hi = 0;
  static constexpr uint32_t A1_lo = A1_hi + 128 * K * 2;
  static constexpr uint32_t B1_hi = A1_lo + 128 * K * 2;
  static constexpr uint32_t B1_lo = B1_hi + 64 * K * 2;
  static constexpr uint32_t A2 = B1_lo + 64 * K * 2;    // (beta*Kg)^T, 128 x 64
  static constexpr uint32_t A3 = A2 + 128 * 64 * 2;     // (beta*v)^T, 128 x 64
  static constexpr uint32_t stage = A3 + 128 * 64 * 2;  // TMA staging of q, k, v, g
  static constexpr uint32_t sQ = stage;
  static constexpr uint32_t sK = sQ + 64 * K * 2;
  static constexpr uint32_t sV = sK + 64 * K * 2;
  static constexpr uint32_t sG = sV + 64 * V * 2;
  static constexpr uint32_t stage_end = sG + 64 * K * 4;
  // reuse of the staging area after step 2
  static constexpr uint32_t B2 = stage;                  // Akk_inv (bf16), 64 x 64
  static constexpr uint32_t sAkk = B2 + 64 * 64 * 2;     // fp32 64 x kAkkLd
  static constexpr uint32_t sBeta = stage_end;           // 64 floats
  static constexpr uint32_t sPart = sBeta + 64 * 4;      // 2 x K floats
  static constexpr uint32_t bars = sPart + 2 * K * 4;    // 3 mbarriers
  static constexpr uint32_t tmem_slot = bars + 3 * 8;
  static constexpr uint32_t abort_slot = tmem_slot + 4;
  static constexpr uint32_t total = abort_slot + 4;
  static constexpr uint32_t bytes = total + 1024;  // slack for 1024-B alignment
  static_assert(sAkk + 64 * kAkkLd * 4 <= stage_end, "Akk tile must fit the staging area");
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void split_store(uint8_t* hi_tile, uint8_t* lo_tile, uint32_t off, float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  *reinterpret_cast<__nv_bfloat162*>(hi_tile + off) = h;
  *reinterpret_cast<__nv_bfloat162*>(lo_tile + off) = l;
}

template <int K, int V>
__global__ void __launch_bounds__(kIntraThreads, 1)
    intra_kernel(const Problem P, const __grid_constant__ IntraMaps maps, const void* __restrict__ beta,
                 const IntraOut out) {
  using Lay = IntraLayout<K, V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int hv = blockIdx.x % P.Hv;
  const int gc = blockIdx.x / P.Hv;
  if (*reinterpret_cast<volatile int32_t*>(P.status) != 0) return;
  const ChunkInfo ci = chunk_info(P, gc);
  if (!ci.valid) return;
  const int hq = hv / (P.Hv / P.Hq);
  const int L = ci.L, t0 = ci.t0;
  const int tid = threadIdx.x, warp = tid >> 5;

  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + Lay::bars);
  uint64_t* bar_mma1 = bar_tma + 1;
  uint64_t* bar_mma2 = bar_tma + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::abort_slot);
  float* sBeta = reinterpret_cast<float*>(sm + Lay::sBeta);
  float* sPart = reinterpret_cast<float*>(sm + Lay::sPart);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma1, 1);
    mbar_init(bar_mma2, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  if (tid < 64) {
    float b = 0.f;
    if (tid < L) {
      const size_t e = size_t(t0 + tid) * P.Hv + hv;
      b = P.beta_fp32 ? reinterpret_cast<const float*>(beta)[e]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(beta)[e]);
    }
    sBeta[tid] = b;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 64 * K * 2 * 2 + 64 * V * 2 + 64 * K * 4);
    tma_load_3d(sm + Lay::sQ, &maps.q, 0, hq, t0, bar_tma);
    tma_load_3d(sm + Lay::sK, &maps.k, 0, hq, t0, bar_tma);
    tma_load_3d(sm + Lay::sV, &maps.v, 0, hv, t0, bar_tma);
    tma_load_3d(sm + Lay::sG, &maps.g, 0, hv, t0, bar_tma);
  }
  wait_bar(bar_tma, 0, abort_flag, P.status);

  // ---- step 2: cumsum and gated operands (thread = channel pair x row half)
  const int p = tid & 63, h = tid >> 6;
  const int c0 = 2 * p;
  const __nv_bfloat16* sQ = reinterpret_cast<const __nv_bfloat16*>(sm + Lay::sQ);
  const __nv_bfloat16* sK = reinterpret_cast<const __nv_bfloat16*>(sm + Lay::sK);
  const __nv_bfloat16* sV = reinterpret_cast<const __nv_bfloat16*>(sm + Lay::sV);
  const float* sG = reinterpret_cast<const float*>(sm + Lay::sG);
  if (c0 < K) {
    float2 part = make_float2(0.f, 0.f);
    for (int i = 32 * h; i < min(L, 32 * h + 32); ++i) {
      const float2 gv = *reinterpret_cast<const float2*>(sG + i * K + c0);
      part.x += gv.x;
      part.y += gv.y;
    }
    sPart[h * K + c0] = part.x;
    sPart[h * K + c0 + 1] = part.y;
  }
  __syncthreads();
  const size_t head_row = size_t(gc) * P.Hv + hv;  // per-chunk buffers
  if (c0 < K) {
    float2 G = h ? make_float2(sPart[c0], sPart[c0 + 1]) : make_float2(0.f, 0.f);
    const float2 glast = make_float2(sPart[c0] + sPart[K + c0], sPart[c0 + 1] + sPart[K + c0 + 1]);
    const float2 gam = make_float2(__expf(glast.x), __expf(glast.y));
    if (out.gamma && h == 0) *reinterpret_cast<float2*>(out.gamma + head_row * K + c0) = gam;
    uint8_t* A1h = sm + Lay::A1_hi;
    uint8_t* A1l = sm + Lay::A1_lo;
    uint8_t* B1h = sm + Lay::B1_hi;
    uint8_t* B1l = sm + Lay::B1_lo;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      float a2[2][8], kl[2][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int i = 32 * h + 8 * blk + jj;
        float2 Qg = make_float2(0.f, 0.f), Kg = Qg, Kd = Qg;
        float b = 0.f;
        if (i < L) {
          const float2 gv = *reinterpret_cast<const float2*>(sG + i * K + c0);
          G.x += gv.x;
          G.y += gv.y;
          const float2 q2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sQ + i * K + c0));
          const float2 k2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sK + i * K + c0));
          const float2 eG = make_float2(__expf(G.x), __expf(G.y));
          const float2 eN = make_float2(__expf(-G.x), __expf(-G.y));
          Qg = make_float2(q2.x * eG.x, q2.y * eG.y);
          Kg = make_float2(k2.x * eG.x, k2.y * eG.y);
          Kd = make_float2(k2.x * eN.x, k2.y * eN.y);
          b = sBeta[i];
          const size_t tok = size_t(t0 + i) * P.Hv + hv;
          if (out.Qs)
            *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(out.Qs) + tok * K + c0) =
                pack_bf16x2(P.scale * Qg.x, P.scale * Qg.y);
          if (out.G) *reinterpret_cast<float2*>(out.G + tok * K + c0) = G;
        }
        split_store(A1h, A1l, sw128_offset(i, c0, 128), Qg.x, Qg.y);
        split_store(A1h, A1l, sw128_offset(64 + i, c0, 128), Kg.x, Kg.y);
        split_store(B1h, B1l, sw128_offset(i, c0, 64), Kd.x, Kd.y);
        a2[0][jj] = b * Kg.x;
        a2[1][jj] = b * Kg.y;
        kl[0][jj] = Kd.x * gam.x;
        kl[1][jj] = Kd.y * gam.y;
      }
      const int col = 32 * h + 8 * blk;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint4 pa = make_uint4(pack_bf16x2(a2[ch][0], a2[ch][1]), pack_bf16x2(a2[ch][2], a2[ch][3]),
                              pack_bf16x2(a2[ch][4], a2[ch][5]), pack_bf16x2(a2[ch][6], a2[ch][7]));
        *reinterpret_cast<uint4*>(sm + Lay::A2 + sw128_offset(c0 + ch, col, 128)) = pa;
        if (out.KlT) {
          uint4 pk = make_uint4(pack_bf16x2(kl[ch][0], kl[ch][1]), pack_bf16x2(kl[ch][2], kl[ch][3]),
                                pack_bf16x2(kl[ch][4], kl[ch][5]), pack_bf16x2(kl[ch][6], kl[ch][7]));
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.KlT) + (head_row * K + c0 + ch) * 64 +
                                    col) = pk;
        }
      }
    }
  }
  // (beta * v)^T
  if (c0 < V) {
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      float a3[2][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int i = 32 * h + 8 * blk + jj;
        float2 bv = make_float2(0.f, 0.f);
        if (i < L) {
          const float2 v2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sV + i * V + c0));
          bv = make_float2(sBeta[i] * v2.x, sBeta[i] * v2.y);
        }
        a3[0][jj] = bv.x;
        a3[1][jj] = bv.y;
      }
      const int col = 32 * h + 8 * blk;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint4 pa = make_uint4(pack_bf16x2(a3[ch][0], a3[ch][1]), pack_bf16x2(a3[ch][2], a3[ch][3]),
                              pack_bf16x2(a3[ch][4], a3[ch][5]), pack_bf16x2(a3[ch][6], a3[ch][7]));
        *reinterpret_cast<uint4*>(sm + Lay::A3 + sw128_offset(c0 + ch, col, 128)) = pa;
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- step 3: D1 = [Qg; Kg] Kd^T with the hi/lo split (TMEM columns 0-63)
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t id = idesc_bf16_f32(128, 64);
    const uint32_t a_hi = smem_u32(sm + Lay::A1_hi), a_lo = smem_u32(sm + Lay::A1_lo);
    const uint32_t b_hi = smem_u32(sm + Lay::B1_hi), b_lo = smem_u32(sm + Lay::B1_lo);
    umma_kloop(tmem, a_hi, 128, b_hi, 64, K / 16, id, 0);
    umma_kloop(tmem, a_hi, 128, b_lo, 64, K / 16, id, 1);
    umma_kloop(tmem, a_lo, 128, b_hi, 64, K / 16, id, 1);
    umma_commit(bar_mma1);
  }
  wait_bar(bar_mma1, 0, abort_flag, P.status);
  tc_fence_after();

  // ---- step 4
  if (warp < 2) {
    // Aqk rows r = tid (TMEM lanes 0-63)
    const int r = tid;
    uint32_t x[2][32];
    tmem_ld_x32(tmem_addr(tmem, 32 * warp, 0), x[0]);
    tmem_ld_x32(tmem_addr(tmem, 32 * warp, 32), x[1]);
    if (r < L) {
      const size_t tok = size_t(t0 + r) * P.Hv + hv;
      float a[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) a[c] = (c <= r) ? P.scale * __uint_as_float(x[c >> 5][c & 31]) : 0.f;
      if (out.Aqk) {
        float4* dst = reinterpret_cast<float4*>(out.Aqk + tok * 64);
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
      }
      if (out.Aqk_b) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.Aqk_b) + tok * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_uint4(pack_bf16x2(a[8 * c], a[8 * c + 1]), pack_bf16x2(a[8 * c + 2], a[8 * c + 3]),
                              pack_bf16x2(a[8 * c + 4], a[8 * c + 5]), pack_bf16x2(a[8 * c + 6], a[8 * c + 7]));
      }
    }
  } else {
    // Akk rows r = tid - 64 (TMEM lanes 64-127) -> shared fp32, then invert
    float* sAkk = reinterpret_cast<float*>(sm + Lay::sAkk);
    const int r = tid - 64;
    uint32_t x[2][32];
    tmem_ld_x32(tmem_addr(tmem, 32 * warp, 0), x[0]);
    tmem_ld_x32(tmem_addr(tmem, 32 * warp, 32), x[1]);
    const float br = sBeta[r];
    const bool rv = r < L;
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      float4 v4;
      v4.x = (rv && c + 0 < r) ? br * __uint_as_float(x[c >> 5][(c + 0) & 31]) : 0.f;
      v4.y = (rv && c + 1 < r) ? br * __uint_as_float(x[c >> 5][(c + 1) & 31]) : 0.f;
      v4.z = (rv && c + 2 < r) ? br * __uint_as_float(x[c >> 5][(c + 2) & 31]) : 0.f;
      v4.w = (rv && c + 3 < r) ? br * __uint_as_float(x[c >> 5][(c + 3) & 31]) : 0.f;
      *reinterpret_cast<float4*>(sAkk + r * kAkkLd + c) = v4;
    }
    named_bar_sync(1, 64);
    // forward substitution: thread j owns column j of X = (I + Akk)^{-1}
    const int j = r;
    float xs[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) xs[i] = 0.f;
#pragma unroll
    for (int rr = 0; rr < 64; ++rr) {
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      const float4* arow = reinterpret_cast<const float4*>(sAkk + rr * kAkkLd);
#pragma unroll
      for (int g4 = 0; g4 < (rr + 3) / 4; ++g4) {
        const float4 a4 = arow[g4];
        acc0 = fmaf(a4.x, xs[4 * g4 + 0], acc0);
        acc1 = fmaf(a4.y, xs[4 * g4 + 1], acc1);
        acc2 = fmaf(a4.z, xs[4 * g4 + 2], acc2);
        acc3 = fmaf(a4.w, xs[4 * g4 + 3], acc3);
      }
      xs[rr] = (rr == j ? 1.f : 0.f) - ((acc0 + acc1) + (acc2 + acc3));
    }
    uint8_t* B2 = sm + Lay::B2;
#pragma unroll
    for (int rr = 0; rr < 64; ++rr)
      *reinterpret_cast<__nv_bfloat16*>(B2 + sw128_offset(rr, j, 64)) = __float2bfloat16_rn(xs[rr]);
    if (out.Akk_inv) {
#pragma unroll
      for (int rr = 0; rr < 64; ++rr)
        if (rr < L) out.Akk_inv[(size_t(t0 + rr) * P.Hv + hv) * 64 + j] = xs[rr];
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();

  // ---- step 5: W^T, U^T (TMEM columns 64-127 and 128-191)
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t id = idesc_bf16_f32(128, 64);
    const uint32_t b2 = smem_u32(sm + Lay::B2);
    umma_kloop(tmem + 64, smem_u32(sm + Lay::A2), 128, b2, 64, 4, id, 0);
    umma_kloop(tmem + 128, smem_u32(sm + Lay::A3), 128, b2, 64, 4, id, 0);
    umma_commit(bar_mma2);
  }
  wait_bar(bar_mma2, 0, abort_flag, P.status);
  tc_fence_after();
  {
    const int row = tid;  // channel of k (W) or v (U)
    if (32 * warp < K) {
      uint32_t x[2][32];
      tmem_ld_x32(tmem_addr(tmem, 32 * warp, 64), x[0]);
      tmem_ld_x32(tmem_addr(tmem, 32 * warp, 96), x[1]);
      __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(out.W);
#pragma unroll
      for (int r = 0; r < 64; ++r)
        if (r < L) W[(size_t(t0 + r) * P.Hv + hv) * K + row] = __float2bfloat16_rn(__uint_as_float(x[r >> 5][r & 31]));
    }
    if (32 * warp < V) {
      uint32_t x[2][32];
      tmem_ld_x32(tmem_addr(tmem, 32 * warp, 128), x[0]);
      tmem_ld_x32(tmem_addr(tmem, 32 * warp, 160), x[1]);
      __nv_bfloat16* U = reinterpret_cast<__nv_bfloat16*>(out.U);
#pragma unroll
      for (int r = 0; r < 64; ++r)
        if (r < L) U[(size_t(t0 + r) * P.Hv + hv) * V + row] = __float2bfloat16_rn(__uint_as_float(x[r >> 5][r & 31]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int K, int V>
cudaError_t launch_intra_t(const Problem& P, const IntraMaps& maps, const void* beta, const IntraOut& out,
                           cudaStream_t s) {
  constexpr uint32_t smem = IntraLayout<K, V>::bytes;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel<K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)P.nc_max * P.Hv;
  if (grid <= 0) return cudaSuccess;
  intra_kernel<K, V><<<unsigned(grid), kIntraThreads, smem, s>>>(P, maps, beta, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Problem& P, const IntraMaps& maps, const void* beta, const IntraOut& out,
                         cudaStream_t s) {
  if (P.K == 128 && P.V == 128) return launch_intra_t<128, 128>(P, maps, beta, out, s);
  if (P.K == 128 && P.V == 64) return launch_intra_t<128, 64>(P, maps, beta, out, s);
  if (P.K == 64 && P.V == 128) return launch_intra_t<64, 128>(P, maps, beta, out, s);
  if (P.K == 64 && P.V == 64) return launch_intra_t<64, 64>(P, maps, beta, out, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
