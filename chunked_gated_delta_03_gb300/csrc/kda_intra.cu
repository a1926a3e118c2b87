// Intra-chunk kernel: persistent, warp-specialised, one CTA per SM, looping
// over work items (chunk, value head) with stride gridDim.x.
//
// Steps (the intra-chunk part of cuLA PR #131, Summary: the intra-chunk
// matrices, the FP32 inverse of (I + Akk), the W/U recompute), spread over
// three warp groups so that consecutive items overlap:
//
//  prep  (warps 0-7, thread = channel pair x row quarter): lane 0 of warps
//        4-7 prefetch item j+1's q, k, v, g chunks into L2 (one TMA tensor
//        prefetch each); every thread loads its rows of q, k, g of item j
//        straight from global memory (coalesced, all in flight together);
//        inclusive cumsum G of g down the rows (the quarters exchange partial
//        sums); a chunk whose log-decay on some channel passes
//        KDA_MAX_CHUNK_LOG_DECAY marks its chain for the exact path; gated operands
//        Qg = q*e^G, Kg = k*e^G, Kd = k*e^{-G}, split into bf16 hi + lo and
//        written into K-major SWIZZLE_128B tiles A1 = [Qg; Kg] (128 x K, the
//        Kg rows first for odd items), B1 = Kd (64 x K); the state-pass
//        operands Qs, Kl, gamma (and G, QG) straight to global memory.  Then,
//        once MMA2 of item j-2 has freed slot j%2, the bf16 Kg rows go into
//        its A2 tile and one thread starts the TMA copy of the item's v chunk
//        into its A3 tile (both token rows, MN-major for MMA2); a tail item
//        clears the v rows past its last token once the copy has landed.
//        Last, the prep warps store W/U of item j-2 from TMEM to global
//        memory (thread = channel of its warp's TMEM lane quadrant).
//  epi   (warps 8-11, two pairs: warps 8, 9 read TMEM lanes 0-63, warps 10,
//        11 lanes 64-127).  Item j is inverted by the pair whose lanes hold
//        its Kg rows of D1 (pair 1 for even j, pair 0 for odd j): its leader
//        issues MMA1(j),
//          D1 = A1_hi B1_hi^T + A1_hi B1_lo^T + A1_lo B1_hi^T
//        (M=128, N=64, ~FP32-accurate; the Qg rows give Aqk/scale, the Kg
//        rows Akk/beta; with the TF32 option the prep writes fp32 operands
//        rounded to TF32 across the hi and lo areas instead, and MMA1 is one
//        pass of kind::tf32 MMAs); the pair copies its Akk rows, beta-scaled and
//        strictly masked, into shared memory as Akk^T, inverts (I + Akk) in
//        FP32 by 16 x 16 blocks (forward substitution on the diagonal blocks,
//        then three block diagonals of T = A X, X = -X_ii T), writes
//        B2 = Akk_inv diag(beta) as the bf16 tile of slot j%2, its leader
//        issues MMA2(j): W^T = Kg^T B2^T, U^T = v^T B2^T (M=128, N=64, K=64,
//        A MN-major), and the pair writes the fp32 Akk_inv export by whole
//        rows.  The other pair stages the Aqk rows (scale, causal mask) in its
//        idle Akk^T tile and writes them by whole rows (fp32, and the bf16 copy
//        for the state pass).  The inverses of consecutive items thus run on
//        the two pairs at once.
//
// TMEM: D1 double-buffered at columns 0 / 64; W^T, U^T double-buffered at
// 128 / 256 (W) and +64 (U).  Shared memory: A1/B1 (single), A2/A3 and B2
// (two slots), per pair the Akk^T / Akk_inv tile, the diagonal blocks of
// Akk_inv and the item's beta, partial sums.  Every wait is bounded.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kPrepWarps = 8;
constexpr int kEpiWarp0 = kPrepWarps;     // warps 8..11: two pairs, whose leaders issue the MMAs
constexpr int kIntraThreads = (kPrepWarps + 4) * 32;
constexpr int kPrepThreads = kPrepWarps * 32;
constexpr int kAkkLd = 68;  // fp32 row stride of the Akk tile (conflict-free float4 rows)
constexpr int kXdLd = 20;   // fp32 row stride of a diagonal block of Akk_inv
constexpr int kXdBlk = 16 * kXdLd + 16;  // fp32 stride between the diagonal blocks
constexpr int kRowsPerThread = 16;

template <int K, int V>
struct IntraLayout {
  static constexpr uint32_t A1_hi = 0;
  static constexpr uint32_t A1_lo = A1_hi + 128 * K * 2;
  static constexpr uint32_t B1_hi = A1_lo + 128 * K * 2;
  static constexpr uint32_t B1_lo = B1_hi + 64 * K * 2;
  // 2 slots x [A2 | A3]: Kg (hi part) and v, each as 64 token rows of up to
  // 128 channels, MN-major SWIZZLE_128B (64-channel blocks 8 KB apart)
  static constexpr uint32_t A23 = B1_lo + 64 * K * 2;
  static constexpr uint32_t A3_off = 2 * 64 * 128;
  static constexpr uint32_t A23_slot = 2 * A3_off;
  static constexpr uint32_t B2 = A23 + 2 * A23_slot;    // 2 slots x 64 x 64 bf16
  static constexpr uint32_t B2_slot = 64 * 64 * 2;
  // per epilogue pair: M (fp32 64 x kAkkLd: Akk^T in the strict upper triangle,
  // the off-diagonal blocks of Akk_inv below) and Xd (the four diagonal 16 x 16
  // blocks of Akk_inv, dense)
  static constexpr uint32_t sInv = B2 + 2 * B2_slot;
  static constexpr uint32_t sInv_M = 64 * kAkkLd * 4;
  static constexpr uint32_t sInv_pair = sInv_M + 4 * kXdBlk * 4;
  static constexpr uint32_t sPart = sInv + 2 * sInv_pair;    // 2 x 4 x K floats
  static constexpr uint32_t sBeta = sPart + 2 * 4 * K * 4;  // per epilogue pair, 64 floats: beta of the item's rows
  static constexpr uint32_t bars = sBeta + 2 * 64 * 4;
  static constexpr int kBars = 16;
  static constexpr uint32_t tmem_slot = bars + kBars * 8;
  static constexpr uint32_t abort_slot = tmem_slot + 4;
  static constexpr uint32_t total = abort_slot + 4;
  static constexpr uint32_t bytes = total + 1024;  // slack for 1024-B alignment
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

// barrier indices
enum {
  kOpndFull = 0,   // prep -> MMA1: A1/B1 of item j written              (256 arrivals)
  kA1Empty = 1,    // MMA1 done reading A1/B1 -> prep                    (commit)
  kA23Full = 2,    // [2] prep -> MMA2: A2/A3 slot written               (256 arrivals)
  kA23Empty = 4,   // [2] MMA2 done reading the A2/A3 slot -> prep       (commit)
  kD1Full = 6,     // [2] MMA1 -> epi: D1 ready                          (commit)
  kD1Empty = 8,    // [2] epi -> MMA1: D1 read                           (128 arrivals)
  kD2Full = 10,    // [2] MMA2 -> prep (W/U stores), inverting pair (B2 reuse)  (commit)
  kD2Empty = 12,   // [2] prep -> MMA2: W^T/U^T read                     (256 arrivals)
  kVFull = 14,     // [2] TMA -> MMA2: v of the item in the A3 tile      (1 arrival + bytes)
};

// 2^x by the MUFU ex2 instruction; e^x is taken as 2^(x log2 e).
__device__ __forceinline__ float exp2f_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), on a channel pair;
// returns the hi pair.
__device__ __forceinline__ uint32_t split_store2(uint8_t* hi_tile, uint8_t* lo_tile, uint32_t off, f2 x) {
  const uint32_t h = f2_to_bf16x2(x);
  const f2 lo = f2_sub(x, f2_from_bf16x2(h));
  *reinterpret_cast<uint32_t*>(hi_tile + off) = h;
  *reinterpret_cast<uint32_t*>(lo_tile + off) = f2_to_bf16x2(lo);
  return h;
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

template <int K, int V, bool kQG, bool kTF32>
__global__ void __launch_bounds__(kIntraThreads, 1)
    intra_kernel(const Problem P, const void* __restrict__ qp, const void* __restrict__ kp,
                 const void* __restrict__ vp, const float* __restrict__ gp, const void* __restrict__ beta,
                 const IntraOut out, const __grid_constant__ IntraMaps maps) {
  using Lay = IntraLayout<K, V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // an earlier error (bad cu_seqlens, another kernel's failure) stops the
  // whole CTA: one thread reads the status word, so that every thread takes
  // the same branch before the CTA's barriers
  if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<volatile int32_t*>(P.status) != 0)) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::abort_slot);
  const int grp = P.Hv / P.Hq;
  // Work items (chunk gc, value head hv) in the order gc * Hv + hv, this CTA
  // taking every gridDim.x-th: a cursor (x = hv, y = gc) stepped without division
  const int step_h = int(gridDim.x % unsigned(P.Hv)), step_g = int(gridDim.x / unsigned(P.Hv));
  auto advance = [&](int2 c) {
    c.x += step_h;
    c.y += step_g;
    if (c.x >= P.Hv) {
      c.x -= P.Hv;
      ++c.y;
    }
    return c;
  };
  const int2 first = make_int2(int(blockIdx.x % unsigned(P.Hv)), int(blockIdx.x / unsigned(P.Hv)));

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[kOpndFull], kPrepThreads);
    mbar_init(&bar[kA1Empty], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[kA23Full + s], kPrepThreads);
      mbar_init(&bar[kA23Empty + s], 1);
      mbar_init(&bar[kD1Full + s], 1);
      mbar_init(&bar[kD1Empty + s], 128);
      mbar_init(&bar[kD2Full + s], 1);
      mbar_init(&bar[kD2Empty + s], kPrepThreads);
      mbar_init(&bar[kVFull + s], 1);
    }
    fence_mbar_init();
  }
  if (warp == kEpiWarp0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
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
    // Byte offset of this thread's channel pair in row r of a SWIZZLE_128B
    // tile of 128-byte rows: the atom, row, 16-byte chunk and in-chunk fields
    // occupy disjoint bits, so the chunk's XOR with (r % 8) is one XOR with a
    // per-row constant, applied to the row's base offset.
    const uint32_t cbits = ((uint32_t(c0 & 63) >> 3) << 4) | (uint32_t(c0 & 7) << 1);
    const uint32_t rows0 = uint32_t(kRowsPerThread * quarter) * 128u;
    // (with TF32 operands A1 and B1 hold fp32 rows of 32 channels per atom)
    const uint32_t cbits32 = ((uint32_t(c0 & 31) >> 2) << 4) | (uint32_t(c0 & 3) << 2);
    const uint32_t xA = kTF32 ? uint32_t(c0 >> 5) * 128u * 128u + rows0 + cbits32
                              : uint32_t(c0 >> 6) * 128u * 128u + rows0 + cbits;  // A1, row 16*quarter
    const uint32_t xB1 = kTF32 ? uint32_t(c0 >> 5) * 64u * 128u + rows0 + cbits32
                               : uint32_t(c0 >> 6) * 64u * 128u + rows0 + cbits;  // B1, row 16*quarter
    const uint32_t xB = uint32_t(c0 >> 6) * 64u * 128u + rows0 + cbits;   // A2 and A3, row 16*quarter
    int j = 0;
    // Chunk lookups (dependent loads of the chunk table in varlen mode) run two
    // items ahead, so that neither this item's loads nor the next item's L2
    // prefetch wait for them.  Items are ordered by chunk and only the chunks
    // past the last valid one are invalid, so the loop ends at the first
    // invalid item.
    auto lookup = [&](int2 c) {
      return c.y < P.nc_max ? chunk_info(P, c.y) : ChunkInfo{0, 0, 0, 0, false};
    };
    // W/U of item jj from TMEM straight to global memory: thread = channel
    // 32*(warp%4) + lane (the warp's TMEM lane quadrant), warps 0-3 taking
    // tokens 0-31 and warps 4-7 tokens 32-63 (a warp writes 64 contiguous
    // bytes per token).  Run two items late, when MMA2 of the item is done.
    auto store_wu = [&](int jj, int3 u) {
      const int sb = jj & 1;
      wait_bar(&bar[kD2Full + sb], par(jj >> 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t dW = tmem + 128 + 128 * sb;
      const int q4 = warp & 3, th = warp >> 2;
      const int ch = 32 * q4 + lane;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int D = part == 0 ? K : V;
        uint32_t x[32];
        tmem_ld_x32(tmem_addr(dW + 64 * part + 32 * th, 32 * q4, 0), x);
        if (32 * q4 < D) {
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(part == 0 ? out.W : out.U) +
                               (size_t(u.x + 32 * th) * P.Hv + u.z) * D + ch;
          const size_t stride = size_t(P.Hv) * D;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            if (32 * th + t < u.y) *dst = __float2bfloat16_rn(__uint_as_float(x[t]));
            dst += stride;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar[kD2Empty + sb]);
    };
    int3 hist[2] = {make_int3(0, 0, 0), make_int3(0, 0, 0)};  // (t0, L, hv) of items j-2, j-1
    int2 cur = first, nxt = advance(first), nnx = advance(nxt);
    ChunkInfo ci = lookup(cur);
    ChunkInfo nci = lookup(nxt);
    while (cur.y < P.nc_max && ci.valid) {
      const int hv = cur.x;
      const int gc = cur.y;
      const int hq = hv / grp;
      const int L = ci.L, t0 = ci.t0;
      const int s = j & 1;
      const ChunkInfo nnci = lookup(nnx);
      if (lane == 0 && warp >= 4 && nci.valid) {
        // L2 prefetch of the next item's chunk of q, k, v and g: one TMA
        // prefetch per tensor (a box of 64 token rows of one head), issued by
        // lane 0 of warps 4-7
        const int nhv = nxt.x;
        const CUtensorMap* m = warp == 4 ? &maps.q : warp == 5 ? &maps.k : warp == 6 ? &maps.v : &maps.g;
        tma_prefetch_l2_3d(m, 0, warp < 6 ? nhv / grp : nhv, nci.t0);
      }
      // ---- loads (all in flight together)
      float2 g2[kRowsPerThread];
      uint32_t q2[kRowsPerThread], k2[kRowsPerThread];
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const int i = kRowsPerThread * quarter + rr;
        g2[rr] = make_float2(0.f, 0.f);
        q2[rr] = k2[rr] = 0u;
        if (i < L && kact) {
          const size_t tq = size_t(t0 + i) * P.Hq + hq, tv = size_t(t0 + i) * P.Hv + hv;
          g2[rr] = __ldg(reinterpret_cast<const float2*>(gp + tv * K + c0));
          q2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(qp) + tq * K + c0));
          k2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(kp) + tq * K + c0));
        }
      }
      // ---- cumsum offsets across row quarters
      float* part = sPart + s * 4 * K;
      if (kact) {
        float2 sum = make_float2(0.f, 0.f);
#pragma unroll
        for (int rr = 0; rr < kRowsPerThread; ++rr) {
          sum.x += g2[rr].x;
          sum.y += g2[rr].y;
        }
        *reinterpret_cast<float2*>(part + quarter * K + c0) = sum;
      }
      named_bar_sync(1, kPrepThreads);
      float2 G = make_float2(0.f, 0.f), glast = make_float2(0.f, 0.f);
      if (kact) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float2 ps = *reinterpret_cast<const float2*>(part + qq * K + c0);
          if (qq < quarter) {
            G.x += ps.x;
            G.y += ps.y;
          }
          glast.x += ps.x;
          glast.y += ps.y;
        }
      }
      // The decay factors e^{G_r - G_i} are formed as products of q e^{G} and
      // k e^{-G}; both stay normal fp32 numbers only while the chunk's total
      // log-decay on the channel is at most KDA_MAX_CHUNK_LOG_DECAY.  Past it
      // the chain is marked, and the exact path recomputes it afterwards.
      if (kact && quarter == 0 && fminf(glast.x, glast.y) < -KDA_MAX_CHUNK_LOG_DECAY)
        P.flags[size_t(ci.n) * P.Hv + hv] = 1;
      const float2 gam = make_float2(__expf(glast.x), __expf(glast.y));
      const size_t head_row = size_t(gc) * P.Hv + hv;
      if (kact && quarter == 0 && out.gamma) *reinterpret_cast<float2*>(out.gamma + head_row * K + c0) = gam;
      // ---- wait for MMA1 of the previous item to release A1/B1
      if (j >= 1) wait_bar(&bar[kA1Empty], par(j - 1), abort_flag, P.status);
      // rows of Qg and Kg in A1: the D1 rows of Kg (Akk) land in the TMEM lanes
      // of the epilogue pair that inverts this item
      const int qrow = 64 * s, krow = 64 - qrow;
      // ---- gated operands of MMA1 (and the bf16 Kg rows kept for the A2 tile)
      uint32_t kgh[kRowsPerThread];
      if (kact) {
        f2 G2 = f2_make(G.x, G.y);
        const f2 gam2 = f2_make(gam.x, gam.y);
        const f2 scale2 = f2_make(P.scale, P.scale);
        const f2 kLog2e2 = f2_make(1.4426950408889634f, 1.4426950408889634f);
        uint8_t* A1h = sm + Lay::A1_hi;
        uint8_t* A1l = sm + Lay::A1_lo;
        uint8_t* B1h = sm + Lay::B1_hi;
        uint8_t* B1l = sm + Lay::B1_lo;
        const uint32_t xq = xA + uint32_t(qrow) * 128u, xk = xA + uint32_t(krow) * 128u;
        __nv_bfloat16* qs_row = out.Qs ? reinterpret_cast<__nv_bfloat16*>(out.Qs) +
                                             (size_t(t0 + kRowsPerThread * quarter) * P.Hv + hv) * K + c0
                                       : nullptr;
        __nv_bfloat16* kl_row = out.Kl ? reinterpret_cast<__nv_bfloat16*>(out.Kl) +
                                             (size_t(t0 + kRowsPerThread * quarter) * P.Hv + hv) * K + c0
                                       : nullptr;
        const size_t qs_stride = size_t(P.Hv) * K;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
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
            const uint32_t swr = uint32_t(rr & 7) << 4, rowr = uint32_t(rr) * 128u;
            if constexpr (kTF32) {
              // fp32 tiles spanning the hi and lo areas, rounded to TF32
              *reinterpret_cast<unsigned long long*>(A1h + (xq ^ swr) + rowr) = f2_to_tf32x2(Qg);
              *reinterpret_cast<unsigned long long*>(A1h + (xk ^ swr) + rowr) = f2_to_tf32x2(Kg);
              *reinterpret_cast<unsigned long long*>(B1h + (xB1 ^ swr) + rowr) = f2_to_tf32x2(Kd);
              kgh[rr] = f2_to_bf16x2(Kg);
            } else {
              split_store2(A1h, A1l, (xq ^ swr) + rowr, Qg);
              kgh[rr] = split_store2(A1h, A1l, (xk ^ swr) + rowr, Kg);
              split_store2(B1h, B1l, (xB1 ^ swr) + rowr, Kd);
            }
            if (i < L) {
              const size_t tok = size_t(t0 + i) * P.Hv + hv;
              if (qs_row)
                *reinterpret_cast<uint32_t*>(qs_row + size_t(rr) * qs_stride) = f2_to_bf16x2(f2_mul(Qg, scale2));
              if (kl_row)
                *reinterpret_cast<uint32_t*>(kl_row + size_t(rr) * qs_stride) = f2_to_bf16x2(f2_mul(Kd, gam2));
              if (out.G) *reinterpret_cast<float2*>(out.G + tok * K + c0) = f2_split(G2);
              if constexpr (kQG)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(out.QG) + tok * K + c0) =
                    f2_to_bf16x2(Qg);
            }
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[kOpndFull]);
      // ---- A2/A3 slot s: free once MMA2 of item j - 2 has read it.  v comes
      // by TMA (MN-major, SWIZZLE_128B); the prep writes the Kg rows.
      if (j >= 2) wait_bar(&bar[kA23Empty + s], par((j >> 1) - 1), abort_flag, P.status);
      uint8_t* A2 = sm + Lay::A23 + s * Lay::A23_slot;
      uint8_t* A3 = A2 + Lay::A3_off;
      if (warp == 6 && lane == 0) {
        mbar_arrive_expect_tx(&bar[kVFull + s], uint32_t(V) * 64u * 2u);
#pragma unroll
        for (int a = 0; a < V / 64; ++a) tma_load_3d(A3 + a * 64 * 128, &maps.v_sw, a * 64, hv, t0, &bar[kVFull + s]);
      }
      if (kact) {
#pragma unroll
        for (int rr = 0; rr < kRowsPerThread; ++rr)
          *reinterpret_cast<uint32_t*>(A2 + (xB ^ (uint32_t(rr & 7) << 4)) + uint32_t(rr) * 128u) = kgh[rr];
      }
      if (L < kChunk) {
        // tail item: rows L..63 of the v box hold tokens of the next chunk or
        // sequence; clear them once the copy has landed, so that U depends on
        // this chunk's tokens alone (their W/U weights are exact zeros)
        if (vact && kRowsPerThread * quarter + kRowsPerThread > L) {
          wait_bar(&bar[kVFull + s], par(j >> 1), abort_flag, P.status);
#pragma unroll
          for (int rr = 0; rr < kRowsPerThread; ++rr)
            if (kRowsPerThread * quarter + rr >= L)
              *reinterpret_cast<uint32_t*>(A3 + (xB ^ (uint32_t(rr & 7) << 4)) + uint32_t(rr) * 128u) = 0u;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[kA23Full + s]);
      if (j >= 2) store_wu(j - 2, hist[0]);
      hist[0] = hist[1];
      hist[1] = make_int3(t0, L, hv);
      ci = nci;
      nci = nnci;
      cur = nxt;
      nxt = nnx;
      nnx = advance(nnx);
      ++j;
    }
    if (j >= 2) store_wu(j - 2, hist[0]);
    if (j >= 1) store_wu(j - 1, hist[1]);

  } else {
    // ================================================================ epi
    // Two pairs of warps: pair 0 (warps 8, 9) reads TMEM lanes 0-63, pair 1
    // (warps 10, 11) lanes 64-127.  For item j the pair whose lanes hold the
    // Kg rows of D1 (pair 1 for even j, pair 0 for odd j) inverts (I + Akk)
    // and issues MMA2(j); the other pair exports Aqk.  Then both store their
    // channels of W/U of item j-1.  Consecutive inverses thus overlap.
    const int q4 = warp & 3;                   // TMEM lane quadrant
    const int pair = (warp - kEpiWarp0) >> 1;
    const int r = lane + 32 * (q4 & 1);        // D1 row within the pair's 64 lanes
    const uint32_t pair_bar = 2 + pair;        // named barrier of the pair's 64 threads
    const bool leader = (warp & 1) == 0 && lane == 0;
    float* M = reinterpret_cast<float*>(sm + Lay::sInv + pair * Lay::sInv_pair);
    float* Xd = M + 64 * kAkkLd;
    float* sB = reinterpret_cast<float*>(sm + Lay::sBeta) + pair * 64;  // beta of the item's rows
    constexpr uint32_t id = idesc_bf16_f32(128, 64);
    // MMA1(jj), issued by the leader of the pair that inverts item jj, once
    // every prep thread has written the item's A1/B1 tiles: D1 = [Qg; Kg] Kd^T
    // with the hi/lo split (rows of Qg first for even items, of Kg for odd ones)
    auto mma1 = [&](int jj) {
      wait_bar(&bar[kOpndFull], par(jj), abort_flag, P.status);
      if (jj >= 2) wait_bar(&bar[kD1Empty + (jj & 1)], par((jj >> 1) - 1), abort_flag, P.status);
      tc_fence_after();
      const uint64_t a_hi = sdesc_kmajor_sw128(smem_u32(sm + Lay::A1_hi));
      const uint64_t a_lo = sdesc_kmajor_sw128(smem_u32(sm + Lay::A1_lo));
      const uint64_t b_hi = sdesc_kmajor_sw128(smem_u32(sm + Lay::B1_hi));
      const uint64_t b_lo = sdesc_kmajor_sw128(smem_u32(sm + Lay::B1_lo));
      const uint32_t d1 = tmem + 64 * (jj & 1);
      // atoms of 64 channels: 128 rows of A1 (1024 descriptor units apart), 64
      // rows of B1 (512 apart)
      if constexpr (kTF32) {
        // one pass on the fp32 tiles: atoms of 32 channels
        constexpr uint32_t idt = idesc_tf32_f32(128, 64);
#pragma unroll
        for (int at = 0; at < K / 32; ++at) umma_atom4_tf32(d1, a_hi + at * 1024, b_hi + at * 512, idt, at > 0);
      } else {
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(d1, a_hi + at * 1024, b_hi + at * 512, id, at > 0);
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(d1, a_hi + at * 1024, b_lo + at * 512, id, 1);
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(d1, a_lo + at * 1024, b_hi + at * 512, id, 1);
      }
      umma_commit(&bar[kD1Full + (jj & 1)]);
      umma_commit(&bar[kA1Empty]);
    };
    // MMA2(jj): W^T = Kg^T B2^T, U^T = v^T B2^T with B2 = Akk_inv diag(beta)
    // (leader of the inverting pair).  Kg and v are MN-major tiles of 64 token
    // rows (the K dimension here), 64-channel blocks 8 KB apart; a K step of
    // 16 tokens advances A by 2048 B and B2 (K-major) by 32 B.
    auto mma2 = [&](int jj) {
      const int s = jj & 1;
      wait_bar(&bar[kA23Full + s], par(jj >> 1), abort_flag, P.status);
      wait_bar(&bar[kVFull + s], par(jj >> 1), abort_flag, P.status);
      if (jj >= 2) wait_bar(&bar[kD2Empty + s], par((jj >> 1) - 1), abort_flag, P.status);
      tc_fence_after();
      constexpr uint32_t idmn = idesc_bf16_f32(128, 64) | kIdescAMajorMN;
      const uint32_t a2s = smem_u32(sm + Lay::A23 + s * Lay::A23_slot);
      const uint64_t a2 = sdesc_mnmajor_sw128(a2s, 64 * 128);
      const uint64_t a3 = sdesc_mnmajor_sw128(a2s + Lay::A3_off, 64 * 128);
      const uint64_t b2 = sdesc_kmajor_sw128(smem_u32(sm + Lay::B2 + s * Lay::B2_slot));
      const uint32_t dW = tmem + 128 + 128 * s;
      umma_k4(dW, a2, b2, idmn, 0, 2048 / 16, 2);
      umma_k4(dW + 64, a3, b2, idmn, 0, 2048 / 16, 2);
      umma_commit(&bar[kD2Full + s]);
      umma_commit(&bar[kA23Empty + s]);
    };
    int j = 0;
    for (int2 cur = first; cur.y < P.nc_max; cur = advance(cur)) {
      const int hv = cur.x;
      const ChunkInfo ci = chunk_info(P, cur.y);
      if (!ci.valid) continue;
      const int L = ci.L, t0 = ci.t0;
      const int s = j & 1;
      const bool inverts = s != pair;
      // beta of row r (inverting pair), loaded before the waits below
      const float br = (inverts && r < L) ? load_beta(beta, P.beta_fp32, size_t(t0 + r) * P.Hv + hv) : 0.f;
      if (inverts) {
        if (leader) mma1(j);
        __syncwarp();
      }
      wait_bar(&bar[kD1Full + s], par(j >> 1), abort_flag, P.status);
      tc_fence_after();
      const uint32_t d1 = tmem + 64 * s;
      if (!inverts) {
        // Aqk row r (scale, causal mask) staged in the pair's M tile, which is
        // free between the pair's inverses (the barrier below waits for the
        // last reads of its previous Akk_inv export), then written out by
        // whole rows: a warp stores full 128-byte lines instead of a 16-byte
        // piece of 32 different rows per instruction.
        uint32_t xa[32], xb[32];
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 0), xa);
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 32), xb);
        tc_fence_before();
        mbar_arrive(&bar[kD1Empty + s]);
        named_bar_sync(pair_bar, 64);
        float* mrow = M + r * kAkkLd;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          float a[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            a[e] = (c + e <= r) ? P.scale * __uint_as_float(c + e < 32 ? xa[c + e] : xb[c + e - 32]) : 0.f;
          *reinterpret_cast<float4*>(mrow + c) = make_float4(a[0], a[1], a[2], a[3]);
        }
        named_bar_sync(pair_bar, 64);
        if (out.Aqk) {
          // 16 passes of 4 rows x 16 column quads
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int row = 4 * it + (r >> 4), c4 = 4 * (r & 15);
            if (row < L)
              *reinterpret_cast<float4*>(out.Aqk + (size_t(t0 + row) * P.Hv + hv) * 64 + c4) =
                  *reinterpret_cast<const float4*>(M + row * kAkkLd + c4);
          }
        }
        if (out.Aqk_b) {
          // 8 passes of 8 rows x 8 column octets, rounded to bf16
#pragma unroll 4
          for (int it = 0; it < 8; ++it) {
            const int row = 8 * it + (r >> 3), c8 = 8 * (r & 7);
            if (row < L) {
              const float4 u = *reinterpret_cast<const float4*>(M + row * kAkkLd + c8);
              const float4 w = *reinterpret_cast<const float4*>(M + row * kAkkLd + c8 + 4);
              const float f[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
              *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.Aqk_b) +
                                        (size_t(t0 + row) * P.Hv + hv) * 64 + c8) = pack8(f);
            }
          }
        }
        named_bar_sync(pair_bar, 64);
      } else {
        // Akk row r, beta-scaled and strictly masked, into the strict upper
        // triangle of M as Akk^T (M[c][r] = Akk[r][c], c < r).  The pair's
        // previous use of M (the Aqk rows it staged for the item before)
        // ended with a barrier after its last read.
        uint32_t xa[32], xb[32];
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 0), xa);
        tmem_ld_x32(tmem_addr(d1, 32 * q4, 32), xb);
        tc_fence_before();
        mbar_arrive(&bar[kD1Empty + s]);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < r) M[c * kAkkLd + r] = br * __uint_as_float(c < 32 ? xa[c] : xb[c - 32]);
        sB[r] = br;
        named_bar_sync(pair_bar, 64);
        // X = (I + Akk)^{-1} by 16 x 16 blocks.  Diagonal blocks: forward
        // substitution in registers, thread = (block d, column c), into Xd.
        {
          const int d = r >> 4, c = r & 15, base = 16 * d;
          float x[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < rr; ++i) acc = fmaf(M[(base + i) * kAkkLd + base + rr], x[i], acc);
            x[rr] = (rr == c ? 1.f : 0.f) - acc;
          }
          float* xd = Xd + d * kXdBlk + c;
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) xd[rr * kXdLd] = x[rr];
        }
        named_bar_sync(pair_bar, 64);
        // Off-diagonal blocks, one block diagonal at a time:
        //   T = Akk[16i + r, 16j : 16i] X[16j : 16i, 16j + cols],  X_ij = -X_ii T,
        // T held in the (i, j) block of M until X_ij replaces it.
        // Thread = (row r16, column quad cq) of each 16 x 16 block.
        const int r16 = r >> 2, cq = 4 * (r & 3);
#pragma unroll 1
        for (int lvl = 1; lvl < 4; ++lvl) {
#pragma unroll 1
          for (int jb = 0; jb + lvl < 4; ++jb) {
            const int ib = jb + lvl;
            const float* acol = M + 16 * ib + r16;  // acol[kk * kAkkLd] = Akk[16 ib + r16][kk]
            const float* xdj = Xd + jb * kXdBlk + cq;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int kk = 0; kk < 16; ++kk) {
              const float a = acol[(16 * jb + kk) * kAkkLd];
              const float4 xv = *reinterpret_cast<const float4*>(xdj + kk * kXdLd);
              acc.x = fmaf(a, xv.x, acc.x);
              acc.y = fmaf(a, xv.y, acc.y);
              acc.z = fmaf(a, xv.z, acc.z);
              acc.w = fmaf(a, xv.w, acc.w);
            }
#pragma unroll 4
            for (int kk = 16 * jb + 16; kk < 16 * ib; ++kk) {
              const float a = acol[kk * kAkkLd];
              const float4 xv = *reinterpret_cast<const float4*>(M + kk * kAkkLd + 16 * jb + cq);
              acc.x = fmaf(a, xv.x, acc.x);
              acc.y = fmaf(a, xv.y, acc.y);
              acc.z = fmaf(a, xv.z, acc.z);
              acc.w = fmaf(a, xv.w, acc.w);
            }
            *reinterpret_cast<float4*>(M + (16 * ib + r16) * kAkkLd + 16 * jb + cq) = acc;
          }
          named_bar_sync(pair_bar, 64);
          float4 xn[3];
#pragma unroll
          for (int jb = 0; jb < 3; ++jb) {
            xn[jb] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (jb + lvl < 4) {
              const int ib = jb + lvl;
              const float* xrow = Xd + ib * kXdBlk + r16 * kXdLd;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int kk = 0; kk < 16; ++kk) {
                const float xv = xrow[kk];
                const float4 t = *reinterpret_cast<const float4*>(M + (16 * ib + kk) * kAkkLd + 16 * jb + cq);
                acc.x = fmaf(xv, t.x, acc.x);
                acc.y = fmaf(xv, t.y, acc.y);
                acc.z = fmaf(xv, t.z, acc.z);
                acc.w = fmaf(xv, t.w, acc.w);
              }
              xn[jb] = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
            }
          }
          named_bar_sync(pair_bar, 64);
#pragma unroll
          for (int jb = 0; jb < 3; ++jb)
            if (jb + lvl < 4) *reinterpret_cast<float4*>(M + (16 * (jb + lvl) + r16) * kAkkLd + 16 * jb + cq) = xn[jb];
          named_bar_sync(pair_bar, 64);
        }
        // row r of X: bf16 B2 operand row and the fp32 export row (blocks left
        // of the diagonal from M, the diagonal block from Xd, zeros after it)
        // (once MMA2 of the pair's previous item has finished reading the slot)
        uint8_t* B2 = sm + Lay::B2 + s * Lay::B2_slot;
        if (j >= 2) wait_bar(&bar[kD2Full + s], par((j >> 1) - 1), abort_flag, P.status);
        const int d = r >> 4;
        const float* xoff = M + r * kAkkLd;
        const float* xdia = Xd + d * kXdBlk + (r & 15) * kXdLd - 16 * d;
#pragma unroll
        for (int c8 = 0; c8 < 64; c8 += 8) {
          const int blk = c8 >> 4;
          float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = u;
          if (blk <= d) {
            const float* src = (blk < d ? xoff : xdia) + c8;
            u = *reinterpret_cast<const float4*>(src);
            w = *reinterpret_cast<const float4*>(src + 4);
          }
          // B2 = Akk_inv diag(beta): column c scaled by beta of row c
          const float4 b0 = *reinterpret_cast<const float4*>(sB + c8);
          const float4 b1 = *reinterpret_cast<const float4*>(sB + c8 + 4);
          const float f[8] = {u.x * b0.x, u.y * b0.y, u.z * b0.z, u.w * b0.w,
                              w.x * b1.x, w.y * b1.y, w.z * b1.z, w.w * b1.w};
          *reinterpret_cast<uint4*>(B2 + sw128_offset(r, c8, 64)) = pack8(f);
        }
        fence_proxy_async_smem();
        named_bar_sync(pair_bar, 64);
        if (leader) mma2(j);
        __syncwarp();
        if (out.Akk_inv) {
          // fp32 export by whole rows (16 passes of 4 rows x 16 column quads):
          // blocks left of the diagonal from M, the diagonal block from Xd,
          // zeros after it
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int row = 4 * it + (r >> 4), c4 = 4 * (r & 15);
            const int dr = row >> 4, blk = c4 >> 4;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (blk < dr) x = *reinterpret_cast<const float4*>(M + row * kAkkLd + c4);
            else if (blk == dr)
              x = *reinterpret_cast<const float4*>(Xd + dr * kXdBlk + (row & 15) * kXdLd + (c4 & 15));
            if (row < L) *reinterpret_cast<float4*>(out.Akk_inv + (size_t(t0 + row) * P.Hv + hv) * 64 + c4) = x;
          }
        }
      }
      ++j;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int K, int V, bool kQG, bool kTF32>
cudaError_t launch_intra_t(const Problem& P, const IntraInputs& in, const IntraOut& out, const IntraMaps& maps,
                           int dev, int sms, cudaStream_t s) {
  constexpr uint32_t smem = IntraLayout<K, V>::bytes;
  cudaError_t e = set_smem_once<intra_kernel<K, V, kQG, kTF32>>(smem, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)P.nc_max * P.Hv;
  if (items <= 0) return cudaSuccess;
  const unsigned grid = unsigned(items < sms ? items : sms);
  intra_kernel<K, V, kQG, kTF32><<<grid, kIntraThreads, smem, s>>>(P, in.q, in.k, in.v, in.g, in.beta, out, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Problem& P, const IntraInputs& in, const IntraOut& out, const IntraMaps& maps,
                         int dev, int sms, cudaStream_t s) {
  // The optional QG export has its own instantiations: any code added to the
  // prep's row loop changes its register allocation, so the usual path
  // carries none of it.
  // The TF32 precision option likewise.
  const bool qg = out.QG != nullptr;
  if (P.tf32) {
    if (P.K == 128 && P.V == 128)
      return qg ? launch_intra_t<128, 128, true, true>(P, in, out, maps, dev, sms, s)
                : launch_intra_t<128, 128, false, true>(P, in, out, maps, dev, sms, s);
    if (P.K == 128 && P.V == 64)
      return qg ? launch_intra_t<128, 64, true, true>(P, in, out, maps, dev, sms, s)
                : launch_intra_t<128, 64, false, true>(P, in, out, maps, dev, sms, s);
    if (P.K == 64 && P.V == 128)
      return qg ? launch_intra_t<64, 128, true, true>(P, in, out, maps, dev, sms, s)
                : launch_intra_t<64, 128, false, true>(P, in, out, maps, dev, sms, s);
    if (P.K == 64 && P.V == 64)
      return qg ? launch_intra_t<64, 64, true, true>(P, in, out, maps, dev, sms, s)
                : launch_intra_t<64, 64, false, true>(P, in, out, maps, dev, sms, s);
    return cudaErrorInvalidValue;
  }
  if (P.K == 128 && P.V == 128)
    return qg ? launch_intra_t<128, 128, true, false>(P, in, out, maps, dev, sms, s)
              : launch_intra_t<128, 128, false, false>(P, in, out, maps, dev, sms, s);
  if (P.K == 128 && P.V == 64)
    return qg ? launch_intra_t<128, 64, true, false>(P, in, out, maps, dev, sms, s)
              : launch_intra_t<128, 64, false, false>(P, in, out, maps, dev, sms, s);
  if (P.K == 64 && P.V == 128)
    return qg ? launch_intra_t<64, 128, true, false>(P, in, out, maps, dev, sms, s)
              : launch_intra_t<64, 128, false, false>(P, in, out, maps, dev, sms, s);
  if (P.K == 64 && P.V == 64)
    return qg ? launch_intra_t<64, 64, true, false>(P, in, out, maps, dev, sms, s)
              : launch_intra_t<64, 64, false, false>(P, in, out, maps, dev, sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
