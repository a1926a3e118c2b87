// Intra-chunk kernel: persistent, warp-specialised, one CTA per SM, looping
// over work items (chunk, value head) with stride gridDim.x.
//
// Steps (the intra-chunk part of cuLA PR #131, Summary: the intra-chunk
// matrices, the FP32 inverse of (I + Akk), the W/U recompute), spread over
// three warp groups so that consecutive items overlap:
//
//  prep  (warps 0-7, thread = channel pair x row quarter): one thread
//        prefetches item j+1's q, k, v, g chunks into L2 (four TMA tensor
//        prefetches); every thread loads its rows of q, k, v, g of item j
//        straight from global memory (coalesced, all in flight together) and
//        64 threads load the item's beta once into shared memory; inclusive
//        cumsum G of g down the rows (the quarters exchange partial sums);
//        a chunk whose log-decay on some channel passes
//        KDA_MAX_CHUNK_LOG_DECAY sets KDA_ERR_GATE_RANGE; gated operands Qg = q*e^G,
//        Kg = k*e^G, Kd = k*e^{-G}, split into bf16 hi + lo and written into
//        K-major SWIZZLE_128B tiles A1 = [Qg; Kg] (128 x K), B1 = Kd (64 x K);
//        (beta*Kg)^T and (beta*v)^T into the A2/A3 tiles of slot j%2; the
//        state-pass operands Qs, Kl^T, gamma (and G) straight to global memory.
//  mma   (lane 0 of warp 8, at the top of each item): MMA1(j):
//        D1 = A1_hi B1_hi^T + A1_hi B1_lo^T + A1_lo B1_hi^T
//        (M=128, N=64; rows 0-63 Aqk/scale, rows 64-127 Akk/beta,
//        ~FP32-accurate), then MMA2(j-1): W^T = (beta*Kg)^T Akk_inv^T and
//        U^T = (beta*v)^T Akk_inv^T (M=128, N=64, K=64).
//  epi   (warps 8-11, TMEM quadrants 0-3): W/U of item j-1 from TMEM as
//        bf16 staging tiles in its A2/A3 slot, stored by TMA; then D1(j): Aqk
//        rows (quadrants 0,1) scaled and causally masked to global (fp32
//        export and the bf16 copy for the state pass), Akk rows (quadrants
//        2,3) beta-scaled and strictly masked into shared memory, where
//        quadrants 2,3 invert (I + Akk) in FP32 by 16 x 16 blocks (forward
//        substitution on the diagonal blocks, then three block diagonals of
//        T = A X, X = -X_ii T) into the bf16 B2 tile of slot j%2 and the fp32
//        export.
//
// TMEM: D1 double-buffered at columns 0 / 64; W^T, U^T double-buffered at
// 128 / 256 (W) and +64 (U).  Shared memory: A1/B1 (single), A2/A3 and B2
// (two slots), the Akk tile and its inverse, partial sums, beta (two slots).
// Every wait is bounded.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kPrepWarps = 8;
constexpr int kEpiWarp0 = kPrepWarps;     // warps 8..11; lane 0 of warp 8 also issues the MMAs
constexpr int kIntraThreads = (kPrepWarps + 4) * 32;
constexpr int kPrepThreads = kPrepWarps * 32;
constexpr int kAkkLd = 68;  // fp32 row stride of the Akk tile (conflict-free float4 rows)
constexpr int kRowsPerThread = 16;

template <int K, int V>
struct IntraLayout {
  static constexpr uint32_t A1_hi = 0;
  static constexpr uint32_t A1_lo = A1_hi + 128 * K * 2;
  static constexpr uint32_t B1_hi = A1_lo + 128 * K * 2;
  static constexpr uint32_t B1_lo = B1_hi + 64 * K * 2;
  static constexpr uint32_t A23 = B1_lo + 64 * K * 2;   // 2 slots x [A2 | A3], each 128 x 64
  static constexpr uint32_t A23_slot = 2 * 128 * 64 * 2;
  static constexpr uint32_t B2 = A23 + 2 * A23_slot;    // 2 slots x 64 x 64 bf16
  static constexpr uint32_t B2_slot = 64 * 64 * 2;
  static constexpr uint32_t sAkk = B2 + 2 * B2_slot;    // fp32 64 x kAkkLd
  static constexpr uint32_t sX = sAkk + 64 * kAkkLd * 4;    // fp32 64 x kAkkLd: Akk_inv, row-major
  static constexpr uint32_t sT = sX + 64 * kAkkLd * 4;       // fp32 3 x 16 x 16 block temporaries
  static constexpr uint32_t sPart = sT + 3 * 16 * 16 * 4;    // 2 x 4 x K floats
  static constexpr uint32_t sBeta = sPart + 2 * 4 * K * 4;  // 2 x 64 floats: beta of the item's rows
  static constexpr uint32_t bars = sBeta + 2 * 64 * 4;
  static constexpr int kBars = 14;
  static constexpr uint32_t tmem_slot = bars + kBars * 8;
  static constexpr uint32_t abort_slot = tmem_slot + 4;
  static constexpr uint32_t total = abort_slot + 4;
  static constexpr uint32_t bytes = total + 1024;  // slack for 1024-B alignment
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

// barrier indices
enum {
  kOpndFull = 0,   // prep -> mma: A1/B1/A2/A3 of item j written          (256 arrivals)
  kA1Empty = 1,    // mma -> prep: MMA1 done reading A1/B1               (commit)
  kA23Empty = 2,   // [2] epi -> prep: A2/A3 slot free (MMA2 and the W/U staging done; 1 arrival)
  kD1Full = 4,     // [2] mma -> epi: D1 ready                           (commit)
  kD1Empty = 6,    // [2] epi -> mma: D1 read                            (128 arrivals)
  kB2Full = 8,     // [2] epi -> mma: B2 slot written                    (64 arrivals)
  kD2Full = 10,    // [2] mma -> epi: W^T/U^T ready                      (commit)
  kD2Empty = 12,   // [2] epi -> mma: W^T/U^T read                       (128 arrivals)
};

// 2^x by the MUFU ex2 instruction; e^x is taken as 2^(x log2 e).
__device__ __forceinline__ float exp2f_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), on a channel pair.
__device__ __forceinline__ void split_store2(uint8_t* hi_tile, uint8_t* lo_tile, uint32_t off, f2 x) {
  const uint32_t h = f2_to_bf16x2(x);
  const f2 lo = f2_sub(x, f2_from_bf16x2(h));
  *reinterpret_cast<uint32_t*>(hi_tile + off) = h;
  *reinterpret_cast<uint32_t*>(lo_tile + off) = f2_to_bf16x2(lo);
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// beta[i] as fp32 from an fp32 or bf16 array, through the read-only path in
// both cases (a plain load would be ordered after the kernel's own stores).
__device__ __forceinline__ float load_beta(const void* beta, int fp32, size_t i) {
  return fp32 ? __ldg(reinterpret_cast<const float*>(beta) + i)
              : __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(beta) + i));
}

// Parity of the wait for the n-th completion (n >= 0) of a barrier.
__device__ __forceinline__ uint32_t par(int n) { return uint32_t(n) & 1u; }

template <int K, int V>
__global__ void __launch_bounds__(kIntraThreads, 1)
    intra_kernel(const Problem P, const void* __restrict__ qp, const void* __restrict__ kp,
                 const void* __restrict__ vp, const float* __restrict__ gp, const void* __restrict__ beta,
                 const IntraOut out, const __grid_constant__ IntraMaps maps) {
  using Lay = IntraLayout<K, V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (*reinterpret_cast<volatile int32_t*>(P.status) != 0) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::abort_slot);
  const long long n_items = (long long)P.nc_max * P.Hv;
  const int grp = P.Hv / P.Hq;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[kOpndFull], kPrepThreads);
    mbar_init(&bar[kA1Empty], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[kA23Empty + s], 1);
      mbar_init(&bar[kD1Full + s], 1);
      mbar_init(&bar[kD1Empty + s], 128);
      mbar_init(&bar[kB2Full + s], 64);
      mbar_init(&bar[kD2Full + s], 1);
      mbar_init(&bar[kD2Empty + s], 128);
    }
    fence_mbar_init();
  }
  if (warp == kEpiWarp0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  {
    // blocks of Akk_inv above the diagonal are never written: zero them once
    float* sX = reinterpret_cast<float*>(sm + Lay::sX);
    for (int e = tid; e < 64 * kAkkLd; e += blockDim.x) sX[e] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kPrepWarps) {
    // =============================================================== prep
    const int p = tid & 63;                     // channel pair
    const int quarter = tid >> 6;               // rows 16*quarter .. +15
    const int c0 = 2 * p;
    const bool kact = c0 < K, vact = c0 < V;
    float* sPart = reinterpret_cast<float*>(sm + Lay::sPart);
    int j = 0;
    // Chunk lookups (dependent loads of the chunk table in varlen mode) run two
    // items ahead, so that neither this item's loads nor the next item's L2
    // prefetch wait for them.  Items are ordered by chunk and only the chunks
    // past the last valid one are invalid, so the loop ends at the first
    // invalid item.
    auto lookup = [&](long long it) {
      return it < n_items ? chunk_info(P, int(it / P.Hv)) : ChunkInfo{0, 0, 0, 0, false};
    };
    ChunkInfo ci = lookup(blockIdx.x);
    ChunkInfo nci = lookup(blockIdx.x + gridDim.x);
    for (long long item = blockIdx.x; item < n_items && ci.valid; item += gridDim.x) {
      const int hv = int(item % P.Hv);
      const int gc = int(item / P.Hv);
      const int hq = hv / grp;
      const int L = ci.L, t0 = ci.t0;
      const long long nitem = item + gridDim.x;
      const ChunkInfo nnci = lookup(nitem + gridDim.x);
      if (tid == 0 && nci.valid) {
        // L2 prefetch of the next item's chunk of q, k, v and g: one TMA
        // prefetch per tensor (a box of 64 token rows of one head)
        const int nhv = int(nitem % P.Hv), nhq = nhv / grp;
        tma_prefetch_l2_3d(&maps.q, 0, nhq, nci.t0);
        tma_prefetch_l2_3d(&maps.k, 0, nhq, nci.t0);
        tma_prefetch_l2_3d(&maps.v, 0, nhv, nci.t0);
        tma_prefetch_l2_3d(&maps.g, 0, nhv, nci.t0);
      }
      // ---- loads (all in flight together)
      float2 g2[kRowsPerThread];
      uint32_t q2[kRowsPerThread], k2[kRowsPerThread], v2[kRowsPerThread];
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const int i = kRowsPerThread * quarter + rr;
        g2[rr] = make_float2(0.f, 0.f);
        q2[rr] = k2[rr] = v2[rr] = 0u;
        if (i < L) {
          const size_t tq = size_t(t0 + i) * P.Hq + hq, tv = size_t(t0 + i) * P.Hv + hv;
          if (kact) {
            g2[rr] = __ldg(reinterpret_cast<const float2*>(gp + tv * K + c0));
            q2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(qp) + tq * K + c0));
            k2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(kp) + tq * K + c0));
          }
          if (vact)
            v2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(vp) + tv * V + c0));
        }
      }
      // ---- beta of the item's rows, once, as fp32 in shared memory (read by
      // every channel pair after the barrier below; two buffers, because the
      // next item's loads may start before slower threads finish this one)
      float* bt = reinterpret_cast<float*>(sm + Lay::sBeta) + (j & 1) * 64 + kRowsPerThread * quarter;
      if (tid < 64)
        bt[tid - kRowsPerThread * quarter] =
            tid < L ? load_beta(beta, P.beta_fp32, size_t(t0 + tid) * P.Hv + hv) : 0.f;
      // ---- cumsum offsets across row quarters
      float* part = sPart + (j & 1) * 4 * K;
      if (kact) {
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int rr = 0; rr < kRowsPerThread; ++rr) {
          s.x += g2[rr].x;
          s.y += g2[rr].y;
        }
        *reinterpret_cast<float2*>(part + quarter * K + c0) = s;
      }
      named_bar_sync(1, kPrepThreads);
      float btv[kRowsPerThread];  // beta of this thread's rows
#pragma unroll
      for (int q = 0; q < kRowsPerThread / 4; ++q) {
        const float4 b4 = reinterpret_cast<const float4*>(bt)[q];
        btv[4 * q] = b4.x;
        btv[4 * q + 1] = b4.y;
        btv[4 * q + 2] = b4.z;
        btv[4 * q + 3] = b4.w;
      }
      float2 G = make_float2(0.f, 0.f), glast = make_float2(0.f, 0.f);
      if (kact) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float2 s = *reinterpret_cast<const float2*>(part + qq * K + c0);
          if (qq < quarter) {
            G.x += s.x;
            G.y += s.y;
          }
          glast.x += s.x;
          glast.y += s.y;
        }
      }
      // The decay factors e^{G_r - G_i} are formed as products of q e^{G} and
      // k e^{-G}; both stay normal fp32 numbers only while the chunk's total
      // log-decay on the channel is at most KDA_MAX_CHUNK_LOG_DECAY.
      if (kact && quarter == 0 && fminf(glast.x, glast.y) < -KDA_MAX_CHUNK_LOG_DECAY)
        set_status(P.status, KDA_ERR_GATE_RANGE);
      const float2 gam = make_float2(__expf(glast.x), __expf(glast.y));
      const size_t head_row = size_t(gc) * P.Hv + hv;
      if (kact && quarter == 0 && out.gamma) *reinterpret_cast<float2*>(out.gamma + head_row * K + c0) = gam;
      // ---- wait for the operand tiles to be free
      if (j >= 1) wait_bar(&bar[kA1Empty], par(j - 1), abort_flag, P.status);
      if (j >= 2) wait_bar(&bar[kA23Empty + (j & 1)], par((j >> 1) - 1), abort_flag, P.status);
      uint8_t* A2 = sm + Lay::A23 + (j & 1) * Lay::A23_slot;
      uint8_t* A3 = A2 + 128 * 64 * 2;
      // ---- gated operands
      if (kact) {
        f2 G2 = f2_make(G.x, G.y);
        const f2 gam2 = f2_make(gam.x, gam.y);
        const f2 scale2 = f2_make(P.scale, P.scale);
        const f2 kLog2e2 = f2_make(1.4426950408889634f, 1.4426950408889634f);
        uint8_t* A1h = sm + Lay::A1_hi;
        uint8_t* A1l = sm + Lay::A1_lo;
        uint8_t* B1h = sm + Lay::B1_hi;
        uint8_t* B1l = sm + Lay::B1_lo;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float a2[2][8], kl[2][8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int rr = 8 * half + e;
            const int i = kRowsPerThread * quarter + rr;
            G2 = f2_add(G2, f2_make(g2[rr].x, g2[rr].y));
            const f2 q = f2_from_bf16x2(q2[rr]);
            const f2 k = f2_from_bf16x2(k2[rr]);
            const f2 gl = f2_mul(G2, kLog2e2);
            const float2 glv = f2_split(gl);
            const f2 eG = f2_make(exp2f_fast(glv.x), exp2f_fast(glv.y));
            const f2 eN = f2_make(exp2f_fast(-glv.x), exp2f_fast(-glv.y));
            const f2 Qg = f2_mul(q, eG);
            const f2 Kg = f2_mul(k, eG);
            const f2 Kd = f2_mul(k, eN);
            split_store2(A1h, A1l, sw128_offset(i, c0, 128), Qg);
            split_store2(A1h, A1l, sw128_offset(64 + i, c0, 128), Kg);
            split_store2(B1h, B1l, sw128_offset(i, c0, 64), Kd);
            const float2 a2v = f2_split(f2_mul(f2_make(btv[rr], btv[rr]), Kg));
            const float2 klv = f2_split(f2_mul(Kd, gam2));
            a2[0][e] = a2v.x;
            a2[1][e] = a2v.y;
            kl[0][e] = klv.x;
            kl[1][e] = klv.y;
            if (i < L) {
              const size_t tok = size_t(t0 + i) * P.Hv + hv;
              if (out.Qs)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(out.Qs) + tok * K + c0) =
                    f2_to_bf16x2(f2_mul(Qg, scale2));
              if (out.G) *reinterpret_cast<float2*>(out.G + tok * K + c0) = f2_split(G2);
            }
          }
          const int col = kRowsPerThread * quarter + 8 * half;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            *reinterpret_cast<uint4*>(A2 + sw128_offset(c0 + ch, col, 128)) = pack8(a2[ch]);
            if (out.KlT)
              *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.KlT) + (head_row * K + c0 + ch) * 64 +
                                        col) = pack8(kl[ch]);
          }
        }
      }
      if (vact) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float a3[2][8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int rr = 8 * half + e;
            const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v2[rr]));
            a3[0][e] = btv[rr] * v.x;
            a3[1][e] = btv[rr] * v.y;
          }
          const int col = kRowsPerThread * quarter + 8 * half;
          *reinterpret_cast<uint4*>(A3 + sw128_offset(c0, col, 128)) = pack8(a3[0]);
          *reinterpret_cast<uint4*>(A3 + sw128_offset(c0 + 1, col, 128)) = pack8(a3[1]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[kOpndFull]);
      ci = nci;
      nci = nnci;
      ++j;
    }
  } else {
    // ================================================================ epi
    const int q4 = warp & 3;        // TMEM lane quadrant
    const int row = 32 * q4 + lane;  // TMEM lane of this thread
    float* sAkk = reinterpret_cast<float*>(sm + Lay::sAkk);
    const bool issuer = (warp == kEpiWarp0) && lane == 0;
    constexpr uint32_t id = idesc_bf16_f32(128, 64);
    // MMA1(jj): D1 = [Qg; Kg] Kd^T with the hi/lo split
    auto mma1 = [&](int jj) {
      wait_bar(&bar[kOpndFull], par(jj), abort_flag, P.status);
      if (jj >= 2) wait_bar(&bar[kD1Empty + (jj & 1)], par((jj >> 1) - 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t a_hi = smem_u32(sm + Lay::A1_hi), a_lo = smem_u32(sm + Lay::A1_lo);
      const uint32_t b_hi = smem_u32(sm + Lay::B1_hi), b_lo = smem_u32(sm + Lay::B1_lo);
      const uint32_t d1 = tmem + 64 * (jj & 1);
      umma_kloop(d1, a_hi, 128, b_hi, 64, K / 16, id, 0);
      umma_kloop(d1, a_hi, 128, b_lo, 64, K / 16, id, 1);
      umma_kloop(d1, a_lo, 128, b_hi, 64, K / 16, id, 1);
      umma_commit(&bar[kD1Full + (jj & 1)]);
      umma_commit(&bar[kA1Empty]);
    };
    // MMA2(jj): W^T = A2 B2^T, U^T = A3 B2^T
    auto mma2 = [&](int jj) {
      const int s = jj & 1;
      wait_bar(&bar[kB2Full + s], par(jj >> 1), abort_flag, P.status);
      if (jj >= 2) wait_bar(&bar[kD2Empty + s], par((jj >> 1) - 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t a2 = smem_u32(sm + Lay::A23 + s * Lay::A23_slot);
      const uint32_t b2 = smem_u32(sm + Lay::B2 + s * Lay::B2_slot);
      const uint32_t dW = tmem + 128 + 128 * s;
      umma_kloop(dW, a2, 128, b2, 64, 4, id, 0);
      umma_kloop(dW + 64, a2 + 128 * 64 * 2, 128, b2, 64, 4, id, 0);
      umma_commit(&bar[kD2Full + s]);
    };
    // W/U of a finished item: thread `row` is channel k (W) / v (U)
    // W/U of a finished item jj (thread `row` = channel k of W / v of U).  Full
    // chunks go through the item's A2/A3 slot (free once MMA2(jj) is done) as
    // row-major staging tiles written out by TMA; the slot then returns to
    // prep.  Partial chunks take plain stores.
    auto store_wu = [&](int jj, int t0, int L, int hv) {
      const int s = jj & 1;
      wait_bar(&bar[kD2Full + s], par(jj >> 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t dW = tmem + 128 + 128 * s;
      uint8_t* stage = sm + Lay::A23 + s * Lay::A23_slot;
      const bool full_chunk = L == kChunk;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int D = part == 0 ? K : V;
        uint32_t x[64];
        tmem_ld_x64(tmem_addr(dW + 64 * part, 32 * q4, 0), x);
        if (32 * q4 < D) {
          if (full_chunk) {
            __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stage + part * 64 * K * 2) + row;
#pragma unroll
            for (int r = 0; r < 64; ++r) st[r * D] = __float2bfloat16_rn(__uint_as_float(x[r]));
          } else {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(part == 0 ? out.W : out.U) +
                                 (size_t(t0) * P.Hv + hv) * D + row;
            const size_t stride = size_t(P.Hv) * D;
#pragma unroll
            for (int r = 0; r < 64; ++r)
              if (r < L) dst[size_t(r) * stride] = __float2bfloat16_rn(__uint_as_float(x[r]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar[kD2Empty + s]);
      if (full_chunk) {
        fence_proxy_async_smem();
        named_bar_sync(4, 128);
      }
      if (issuer) {
        if (full_chunk) {
          tma_store_3d(&maps.W, stage, 0, hv, t0);
          tma_store_3d(&maps.U, stage + 64 * K * 2, 0, hv, t0);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        mbar_arrive(&bar[kA23Empty + s]);
      }
    };
    int j = 0;
    int prev_t0 = 0, prev_L = 0, prev_hv = 0;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int hv = int(item % P.Hv);
      const ChunkInfo ci = chunk_info(P, int(item / P.Hv));
      if (!ci.valid) continue;
      const int L = ci.L, t0 = ci.t0;
      if (issuer) {
        mma1(j);
        if (j >= 1) mma2(j - 1);
      }
      __syncwarp();
      if (j >= 1) store_wu(j - 1, prev_t0, prev_L, prev_hv);
      const int s = j & 1;
      wait_bar(&bar[kD1Full + s], par(j >> 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t d1 = tmem + 64 * s;
      if (q4 < 2) {
        // Aqk row r = row (lanes 0-63)
        const int r = row;
        const size_t tok = size_t(t0 + r) * P.Hv + hv;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t x[32];
          tmem_ld_x32(tmem_addr(d1, 32 * q4, 32 * h), x);
          if (r < L) {
            float a[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) a[c] = (32 * h + c <= r) ? P.scale * __uint_as_float(x[c]) : 0.f;
            if (out.Aqk) {
              float4* dst = reinterpret_cast<float4*>(out.Aqk + tok * 64 + 32 * h);
#pragma unroll
              for (int c = 0; c < 8; ++c) dst[c] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
            }
            if (out.Aqk_b) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.Aqk_b) + tok * 64 + 32 * h);
#pragma unroll
              for (int c = 0; c < 4; ++c) dst[c] = pack8(a + 8 * c);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&bar[kD1Empty + s]);
      } else {
        // Akk row r (lanes 64-127) -> shared fp32, then invert
        const int r = row - 64;
        named_bar_sync(2, 64);  // previous inverse finished reading the Akk tile
        uint32_t xa[32], xb[32];
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 0), xa);
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 32), xb);
        tc_fence_before();
        mbar_arrive(&bar[kD1Empty + s]);
        const float br = r < L ? load_beta(beta, P.beta_fp32, size_t(t0 + r) * P.Hv + hv) : 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          float4 v4;
          const uint32_t* src = c < 32 ? xa : xb;
          v4.x = (c + 0 < r) ? br * __uint_as_float(src[(c + 0) & 31]) : 0.f;
          v4.y = (c + 1 < r) ? br * __uint_as_float(src[(c + 1) & 31]) : 0.f;
          v4.z = (c + 2 < r) ? br * __uint_as_float(src[(c + 2) & 31]) : 0.f;
          v4.w = (c + 3 < r) ? br * __uint_as_float(src[(c + 3) & 31]) : 0.f;
          *reinterpret_cast<float4*>(sAkk + r * kAkkLd + c) = v4;
        }
        named_bar_sync(3, 64);
        // X = (I + Akk)^{-1} by 16 x 16 blocks.  Diagonal blocks: forward
        // substitution in registers, thread = (block d, column c).
        float* sX = reinterpret_cast<float*>(sm + Lay::sX);
        float* sT = reinterpret_cast<float*>(sm + Lay::sT);
        {
          const int d = r >> 4, c = r & 15, base = 16 * d;
          float x[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const float* arow = sAkk + (base + rr) * kAkkLd + base;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < rr; ++i) acc = fmaf(arow[i], x[i], acc);
            x[rr] = (rr == c ? 1.f : 0.f) - acc;
          }
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) sX[(base + rr) * kAkkLd + base + c] = x[rr];
        }
        named_bar_sync(3, 64);
        // Off-diagonal blocks, one block diagonal at a time:
        //   T = Akk[16i + r, 16j : 16i] X[16j : 16i, 16j + cols],  X_ij = -X_ii T.
        // Thread = (row r16, column quad cq) of each 16 x 16 block.
        const int r16 = r >> 2, cq = 4 * (r & 3);
#pragma unroll 1
        for (int lvl = 1; lvl < 4; ++lvl) {
#pragma unroll 1
          for (int jb = 0; jb + lvl < 4; ++jb) {
            const int ib = jb + lvl;
            const float* arow = sAkk + (16 * ib + r16) * kAkkLd;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int kk = 16 * jb; kk < 16 * ib; ++kk) {
              const float a = arow[kk];
              const float4 xv = *reinterpret_cast<const float4*>(sX + kk * kAkkLd + 16 * jb + cq);
              acc.x = fmaf(a, xv.x, acc.x);
              acc.y = fmaf(a, xv.y, acc.y);
              acc.z = fmaf(a, xv.z, acc.z);
              acc.w = fmaf(a, xv.w, acc.w);
            }
            *reinterpret_cast<float4*>(sT + (jb * 16 + r16) * 16 + cq) = acc;
          }
          named_bar_sync(3, 64);
#pragma unroll 1
          for (int jb = 0; jb + lvl < 4; ++jb) {
            const int ib = jb + lvl;
            const float* xrow = sX + (16 * ib + r16) * kAkkLd + 16 * ib;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const float xv = xrow[kk];
              const float4 t = *reinterpret_cast<const float4*>(sT + (jb * 16 + kk) * 16 + cq);
              acc.x = fmaf(xv, t.x, acc.x);
              acc.y = fmaf(xv, t.y, acc.y);
              acc.z = fmaf(xv, t.z, acc.z);
              acc.w = fmaf(xv, t.w, acc.w);
            }
            *reinterpret_cast<float4*>(sX + (16 * ib + r16) * kAkkLd + 16 * jb + cq) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
          }
          named_bar_sync(3, 64);
        }
        // row r of X: bf16 B2 operand row and the fp32 export row
        uint8_t* B2 = sm + Lay::B2 + s * Lay::B2_slot;
        const float* xr = sX + r * kAkkLd;
        float* inv_row = (out.Akk_inv && r < L) ? out.Akk_inv + (size_t(t0 + r) * P.Hv + hv) * 64 : nullptr;
#pragma unroll
        for (int c8 = 0; c8 < 64; c8 += 8) {
          const float4 u = *reinterpret_cast<const float4*>(xr + c8);
          const float4 w = *reinterpret_cast<const float4*>(xr + c8 + 4);
          const float f[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
          *reinterpret_cast<uint4*>(B2 + sw128_offset(r, c8, 64)) = pack8(f);
          if (inv_row) {
            *reinterpret_cast<float4*>(inv_row + c8) = u;
            *reinterpret_cast<float4*>(inv_row + c8 + 4) = w;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[kB2Full + s]);
      }
      prev_t0 = t0;
      prev_L = L;
      prev_hv = hv;
      ++j;
    }
    if (j >= 1) {
      if (issuer) mma2(j - 1);
      __syncwarp();
      store_wu(j - 1, prev_t0, prev_L, prev_hv);
    }
    if (issuer) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int K, int V>
cudaError_t launch_intra_t(const Problem& P, const IntraInputs& in, const IntraOut& out, const IntraMaps& maps,
                           cudaStream_t s) {
  constexpr uint32_t smem = IntraLayout<K, V>::bytes;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel<K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long items = (long long)P.nc_max * P.Hv;
  if (items <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = unsigned(items < sms ? items : sms);
  intra_kernel<K, V><<<grid, kIntraThreads, smem, s>>>(P, in.q, in.k, in.v, in.g, in.beta, out, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Problem& P, const IntraInputs& in, const IntraOut& out, const IntraMaps& maps,
                         cudaStream_t s) {
  if (P.K == 128 && P.V == 128) return launch_intra_t<128, 128>(P, in, out, maps, s);
  if (P.K == 128 && P.V == 64) return launch_intra_t<128, 64>(P, in, out, maps, s);
  if (P.K == 64 && P.V == 128) return launch_intra_t<64, 128>(P, in, out, maps, s);
  if (P.K == 64 && P.V == 64) return launch_intra_t<64, 64>(P, in, out, maps, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
