// Fused chunked KDA forward: one CTA per (sequence, value head) chain runs
// every step of the chunked form for that chain, chunk after chunk, so that
// nothing but the inputs, the outputs and the requested intermediates crosses
// HBM.  The intra-chunk steps of chunk c+1 (cuLA PR #131, Summary: intra-chunk
// matrices, FP32 inverse of (I + Akk), W/U recompute) overlap the state and
// output steps of chunk c (cuLA REPO_LAYOUT.md: chunk_delta_h.py, fwd_o.py).
//
// Warp roles (16 warps; setmaxnreg gives the prep 144 registers a thread, the
// other two warpgroups 112):
//   w0-w7    prep (thread = channel pair x 16-row quarter): loads of q, k, g
//            (lanes 0 of w0-w2 prefetch the next chunk's into L2), inclusive
//            cumsum G, the gated operands Qg = q e^G, Kg = k e^G, Kd = k e^-G
//            as bf16 hi + lo pairs in registers, gamma = e^{G_last}; then the
//            hi halves into the chunk's hi buffer and the lo halves into the
//            lo area.  Thread 0 issues MMA1: D1 = [Qg; Kg] Kd^T with the hi/lo
//            split (hi*hi + lo*hi, then hi*lo once Kd's low half has replaced
//            the A operand's low half in the lo area).  A chunk past the gate
//            range marks its chain for the exact path.  While the next
//            chunk's loads are in flight, w0, w1, w4 and w5 (whose TMEM lane
//            quarters hold D1's Qg rows) write the last chunk's fp32 Aqk
//            export (scale, causal mask) straight from D1.
//   w8-w11   intra epilogue (thread = row of D1): the whole row into
//            registers, which frees D1 for the next MMA1; Aqk rows (causal
//            mask) to a bf16 operand tile; Akk rows
//            (beta, strict mask) to an fp32 scratch; the inverse
//            X = (I + Akk)^-1 by 16 x 16 blocks (diagonal blocks by
//            right-looking forward substitution, the off-diagonal products as
//            warp-level TF32 hi/lo MMAs), writing B2 = X diag(beta) as a bf16
//            tile as it goes; a tail chunk's v rows past its end are cleared;
//            then B2 is handed to MMA2 and Akk_inv leaves by whole rows.
//   w12-w15  state (thread = value channel v = TMEM lane): S^T lives in TMEM
//            in fp32 and as a bf16 copy (the A operand of its MMAs).  Per
//            chunk: w12 lane 0 issues MMA2 (W^T = Kg^T B2^T, U^T = v^T B2^T)
//            once B2 is ready; W^T from TMEM into a token-major W tile in the
//            chunk's dead Kg rows; w12 lane 0 issues P^T = S^T W^T and O^T = S^T Qg^T,
//            the next chunk's v copy and W's TMA store; the threads form
//            Delta^T = U^T - P^T into TMEM (rows past the chunk's end zero)
//            and stage U token-major; w12 lane 0 issues S^T += Delta^T Kd and
//            O^T += Delta^T Aqk^T and U's TMA store; the threads scale the
//            state by gamma
//              S <- Diag(e^{G_last}) (S + Kd^T Delta)
//                 = Diag(e^{G_last}) S + (K e^{G_last - G})^T Delta,
//            hand the hi buffer back, and stage o = scale (Qg S + (Aqk / scale)
//            Delta) token-major for its TMA store.
//
// The bf16 hi tiles of Qg, Kg and Kd are the operands of MMA1, of MMA2 (Kg as
// an MN-major A) and of the state MMAs (Qg, Kd), so they are written once and
// double-buffered by chunk parity.  Every wait is bounded.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kFusedWarps = 16;
constexpr int kFusedThreads = kFusedWarps * 32;
constexpr int kWarpIntra0 = 8, kWarpState0 = 12;
constexpr int kPrepThreadsF = 8 * 32;
constexpr int kRows = 16;  // rows per prep thread
constexpr int kLd = 68;    // fp32 row stride of the inverse's A and X tiles
constexpr uint32_t kNbPrep = 1, kNbIntra = 2, kNbState = 3;  // named barriers

// TMEM columns
constexpr uint32_t kColD1 = 0;     // MMA1: lanes 0-63 Aqk / scale, 64-127 Akk / beta (64 cols)
constexpr uint32_t kColW = 64;     // MMA2: W^T, lane = channel k (64 cols = tokens); then P^T = S^T W^T, lane = v
constexpr uint32_t kColU = 128;    // MMA2: U^T, lane = channel v
constexpr uint32_t kColDt = 192;   // Delta^T in bf16 pairs (32 cols = 64 tokens): A operand of the state MMAs
constexpr uint32_t kColO = 256;    // O^T, lane = v
constexpr uint32_t kColSb = 320;   // S^T in bf16 pairs (K / 2 cols): A operand of P^T and O^T
constexpr uint32_t kColS = 384;    // S^T in fp32, lane = v, column = k

template <int K, int V>
struct FusedLayout {
  static constexpr uint32_t kA1 = K * 256;  // [Qg; Kg]: K/64 atoms of 128 rows x 128 B
  static constexpr uint32_t kB1 = K * 128;  // Kd: K/64 atoms of 64 rows x 128 B
  static constexpr uint32_t kHi = kA1 + kB1;
  static constexpr uint32_t HI = 0;                        // 2 x (A1_hi, B1_hi)
  static constexpr uint32_t LO = HI + 2 * kHi;             // A1_lo, then Kd_lo
  static constexpr uint32_t VT = LO + kA1;                 // v: 64 token rows, 64-channel blocks 8 KB apart
  static constexpr uint32_t AQKB = VT + V * 128;           // 2 x Aqk / scale, bf16 64 x 64, K-major
  static constexpr uint32_t B2 = AQKB + 2 * 8192;          // X diag(beta), bf16 64 x 64, K-major
  static constexpr uint32_t UST = B2 + 8192;               // U staged token-major for its TMA store
  static constexpr uint32_t SCR = UST + V * 128;           // fp32 A and X of the inverse, 64 x kLd each
  static constexpr uint32_t GAM = SCR + 2 * 64 * kLd * 4;  // 2 x K floats: gamma
  static constexpr uint32_t BETA = GAM + 2 * K * 4;        // 64 floats
  static constexpr uint32_t PART = BETA + 64 * 4;          // 2 x 4 x K floats: cumsum partial sums
  static constexpr uint32_t BARS = PART + 2 * 4 * K * 4;
  static constexpr int kBars = 16;
  static constexpr uint32_t TMEM_SLOT = BARS + kBars * 8;
  static constexpr uint32_t ABORT = TMEM_SLOT + 4;
  static constexpr uint32_t total = ABORT + 4;
  static constexpr uint32_t bytes = total + 1024;  // slack for the 1024-B alignment of the base
  static_assert(LO % 1024 == 0 && VT % 1024 == 0 && AQKB % 1024 == 0 && B2 % 1024 == 0 && UST % 1024 == 0,
                "operand and staging tiles must be 1024-B aligned");
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

// barrier indices
enum {
  bLoA = 0,      // MMA1 hi*hi + lo*hi done: A1_lo may be overwritten            (commit)
  bD1Full = 1,   // MMA1 done -> intra epilogue; the lo area is free again       (commit)
  bD1Empty = 2,  // intra epilogue read D1 -> MMA1                               (128)
  bHiFree = 4,   // [2] state done with hi buffer b (and its gamma, Aqk tile)    (128)
  bVFull = 6,    // TMA: v chunk landed                                          (1 + bytes)
  bD2Full = 7,   // MMA2 done -> intra epilogue (B2 free), state                (commit)
  bB2Ready = 8,  // intra wrote B2, the v tail, the Aqk tile -> MMA2 (state)    (128)
  bPDone = 10,   // P^T = S^T W^T done -> state                                  (commit)
  bHODone = 11,  // S^T += Delta^T Kd and O^T (both parts) done                  (commit)
  bDrain = 12,   // [2] final drains of the two MMA issuers (prep, state)        (commit)
};

__device__ __forceinline__ uint32_t par(int n) { return uint32_t(n) & 1u; }

// Register budgets per warpgroup (setmaxnreg; the kernel launches with 128 a
// thread, 65536 in all): the prep warpgroups take 144, the intra and state
// warpgroups 112 each -- 2 x 128 x 144 + 2 x 128 x 112 = 65536, so the
// increase never waits for registers that are not there.
constexpr uint32_t kRegsPrep = 144, kRegsIntra = 112, kRegsState = 112;
static_assert(2 * 128 * kRegsPrep + 128 * kRegsIntra + 128 * kRegsState <= 65536, "register split");
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ float exp2f_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), on a channel pair (both
// as bf16x2): sets hi, returns lo.
__device__ __forceinline__ uint32_t split2(uint32_t& hi, f2 x) {
  hi = f2_to_bf16x2(x);
  return f2_to_bf16x2(f2_sub(x, f2_from_bf16x2(hi)));
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ float load_beta(const void* beta, int fp32, size_t i) {
  return fp32 ? __ldg(reinterpret_cast<const float*>(beta) + i)
              : __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(beta) + i));
}

// fp32 x -> (hi, lo) TF32 bit patterns with x ~ hi + lo: hi rounded to nearest
// TF32, lo the TF32 rounding of the remainder
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

// d0, d1 (16 x 8 each: the mma.m16n8k8 accumulator fragments of columns 0-7
// and 8-15) = A (16 x [k0, k1)) B ([k0, k1) x 16) on the warp's tensor cores,
// from fp32 tiles in shared memory (A row-major, stride lda; B row-major,
// stride ldb), each product as three TF32 products (hi*hi + hi*lo + lo*hi:
// close to fp32 accuracy).  The three partial products and the two column
// halves accumulate separately, so the six chains of dependent MMAs overlap.
// Fragments of the m16n8k8 TF32 shape: lane = 4 g + t holds A[g][t],
// A[g+8][t], A[g][t+4], A[g+8][t+4], B[t][g], B[t+4][g], and D[g][2t],
// D[g][2t+1], D[g+8][2t], D[g+8][2t+1].
__device__ __forceinline__ void mma_3xtf32_x2(float (&d0)[4], float (&d1)[4], const float* A, int lda,
                                              const float* B, int ldb, int k0, int k1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  float acc[6][4];
#pragma unroll
  for (int i = 0; i < 6; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#define KDA_MMA_TF32(c, a, b)                                                                                 \
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "  \
               "{%0,%1,%2,%3};"                                                                               \
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])                                              \
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]))
#pragma unroll 1
  for (int k = k0; k < k1; k += 8) {
    uint32_t ah[4], al[4], bh[2][2], bl[2][2];
    tf32_split(A[g * lda + k + t], ah[0], al[0]);
    tf32_split(A[(g + 8) * lda + k + t], ah[1], al[1]);
    tf32_split(A[g * lda + k + t + 4], ah[2], al[2]);
    tf32_split(A[(g + 8) * lda + k + t + 4], ah[3], al[3]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tf32_split(B[(k + t) * ldb + 8 * h + g], bh[h][0], bl[h][0]);
      tf32_split(B[(k + t + 4) * ldb + 8 * h + g], bh[h][1], bl[h][1]);
    }
    KDA_MMA_TF32(acc[0], ah, bh[0]);
    KDA_MMA_TF32(acc[1], ah, bh[1]);
    KDA_MMA_TF32(acc[2], ah, bl[0]);
    KDA_MMA_TF32(acc[3], ah, bl[1]);
    KDA_MMA_TF32(acc[4], al, bh[0]);
    KDA_MMA_TF32(acc[5], al, bh[1]);
  }
#undef KDA_MMA_TF32
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    d0[e] = acc[0][e] + (acc[2][e] + acc[4][e]);
    d1[e] = acc[1][e] + (acc[3][e] + acc[5][e]);
  }
}

// d (16 x 8) = A (16 x [k0, k1)) B ([k0, k1) x 8), as mma_3xtf32_x2 with one
// column half (three independent accumulation chains).
__device__ __forceinline__ void mma_3xtf32_x1(float (&d)[4], const float* A, int lda, const float* B, int ldb,
                                              int k0, int k1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  float acc[3][4];
#pragma unroll
  for (int i = 0; i < 3; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#define KDA_MMA_TF32(c, a, b)                                                                                 \
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "  \
               "{%0,%1,%2,%3};"                                                                               \
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])                                              \
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]))
#pragma unroll
  for (int k = k0; k < k1; k += 8) {
    uint32_t ah[4], al[4], bh[2], bl[2];
    tf32_split(A[g * lda + k + t], ah[0], al[0]);
    tf32_split(A[(g + 8) * lda + k + t], ah[1], al[1]);
    tf32_split(A[g * lda + k + t + 4], ah[2], al[2]);
    tf32_split(A[(g + 8) * lda + k + t + 4], ah[3], al[3]);
    tf32_split(B[(k + t) * ldb + g], bh[0], bl[0]);
    tf32_split(B[(k + t + 4) * ldb + g], bh[1], bl[1]);
    KDA_MMA_TF32(acc[0], ah, bh);
    KDA_MMA_TF32(acc[1], ah, bl);
    KDA_MMA_TF32(acc[2], al, bh);
  }
#undef KDA_MMA_TF32
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = acc[0][e] + (acc[1][e] + acc[2][e]);
}

// The fragment d (16 x 8 at rows r0.., columns c0..) scaled by s into X (fp32,
// row-major, stride kLd) and, times beta of each column, into the bf16 B2 tile.
__device__ __forceinline__ void store_x_b2(float* X, uint8_t* b2, const float* sB, int r0, int c0,
                                           const float (&d)[4], float s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int c = c0 + 2 * t;
  const float b0 = sB[c], b1 = sB[c + 1];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = r0 + g + 8 * h;
    const float x0 = s * d[2 * h], x1 = s * d[2 * h + 1];
    *reinterpret_cast<float2*>(X + r * kLd + c) = make_float2(x0, x1);
    *reinterpret_cast<uint32_t*>(b2 + sw128_offset(uint32_t(r), uint32_t(c), 64)) = pack_bf16x2(x0 * b0, x1 * b1);
  }
}

// Stores s * d (the accumulator fragment) at C (row-major, stride ldc).
__device__ __forceinline__ void store_frag(float* C, int ldc, const float (&d)[4], float s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(C + g * ldc + 2 * t) = make_float2(s * d[0], s * d[1]);
  *reinterpret_cast<float2*>(C + (g + 8) * ldc + 2 * t) = make_float2(s * d[2], s * d[3]);
}

template <int K, int V, bool kQG>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const Problem P, const FusedArgs A, const __grid_constant__ FusedMaps maps) {
  using Lay = FusedLayout<K, V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int hv = int(blockIdx.x % unsigned(P.Hv));
  const int n = P.varlen ? P.seq_order[blockIdx.x / unsigned(P.Hv)] : int(blockIdx.x / unsigned(P.Hv));
  // an earlier error (bad cu_seqlens, another kernel's failure) stops the
  // whole CTA: one thread reads the status word, so that every thread takes
  // the same branch before the CTA's barriers
  if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<volatile int32_t*>(P.status) != 0)) return;
  int bos, len;
  if (P.varlen) {
    bos = P.cu[n];
    len = P.cu[n + 1] - bos;
  } else {
    bos = n * P.T;
    len = P.T;
  }
  const int nch = (len + kChunk - 1) / kChunk;
  const int hq = hv / (P.Hv / P.Hq);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t hrow = (size_t(n) * P.Hv + hv) * K;  // row (n, hv, k = 0) of the [N, Hv, K, V] states
  if (nch == 0) {
    // an empty sequence leaves its state unchanged
    if (A.hT)
      for (int i = tid; i < K * V; i += kFusedThreads) A.hT[hrow * V + i] = A.h0 ? A.h0[hrow * V + i] : 0.f;
    return;
  }

  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::ABORT);
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[bLoA], 1);
    mbar_init(&bar[bD1Full], 1);
    mbar_init(&bar[bD1Empty], 128);
    mbar_init(&bar[bHiFree], 128);
    mbar_init(&bar[bHiFree + 1], 128);
    mbar_init(&bar[bVFull], 1);
    mbar_init(&bar[bD2Full], 1);
    mbar_init(&bar[bB2Ready], 128);
    mbar_init(&bar[bPDone], 1);
    mbar_init(&bar[bHODone], 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bar[bDrain + i], 1);
    fence_mbar_init();
  }
  if (warp == kWarpIntra0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint64_t kDrainNs = 200000000ull;  // final drains: 0.2 s, whatever the abort flag says

  if (warp < kWarpIntra0) {
    // ================================================================ prep
    regs_inc<kRegsPrep>();
    const int ptid = tid;
    const bool mma_leader = ptid == 0;  // issues MMA1
    const int p = ptid & 63, quarter = ptid >> 6, c0 = 2 * p;
    const bool kact = c0 < K;
    // byte offset of this thread's channel pair in row 16*quarter of a K-major
    // SWIZZLE_128B tile: the atom, row, 16-byte chunk and in-chunk fields are
    // disjoint bits, so the chunk's XOR with (row % 8) is one XOR per row
    const uint32_t cbits = ((uint32_t(c0 & 63) >> 3) << 4) | (uint32_t(c0 & 7) << 1);
    const uint32_t rows0 = uint32_t(kRows * quarter) * 128u;
    const uint32_t xA = uint32_t(c0 >> 6) * 16384u + rows0 + cbits;  // A1 (Qg rows 0-63, Kg rows 64-127)
    const uint32_t xB = uint32_t(c0 >> 6) * 8192u + rows0 + cbits;   // B1 (Kd rows 0-63)
    float* part_base = reinterpret_cast<float*>(sm + Lay::PART);
    float* gam_base = reinterpret_cast<float*>(sm + Lay::GAM);
    uint8_t* lo = sm + Lay::LO;
    // The fp32 Aqk export (scaled, causal mask) of chunk cc from D1's Qg rows
    // (TMEM lanes 0-63), by the prep warps whose lane quarter holds them:
    // warps 0, 1 columns 0-31, warps 4, 5 columns 32-63, thread = row
    const bool aqk_w = A.Aqk != nullptr && (warp & 2) == 0;
    auto export_aqk = [&](int cc) {
      const int tc = bos + cc * kChunk, Lc = min(kChunk, len - cc * kChunk);
      const int r = 32 * (warp & 1) + lane, cb = 32 * (warp >> 2);
      wait_bar(&bar[bD1Full], par(cc), abort_flag, P.status);
      tc_fence_after();
      float* arow = A.Aqk + (size_t(tc + r) * P.Hv + hv) * 64;
      // 8 columns at a time: the next chunk's loads hold 64 registers meanwhile
#pragma unroll 1
      for (int h = cb; h < cb + 32; h += 8) {
        uint32_t x[8];
        tmem_ld_x8(tmem_addr(tmem, 32 * (warp & 1), kColD1 + h), x);  // warp-collective
        if (r < Lc) {
          float f[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = (h + j <= r) ? P.scale * __uint_as_float(x[j]) : 0.f;
          const float4 lo4 = make_float4(f[0], f[1], f[2], f[3]), hi4 = make_float4(f[4], f[5], f[6], f[7]);
          if (A.aqk_v8) {
            st_global_v8(arow + h, lo4, hi4);  // a whole 32-byte sector per thread
          } else {
            __stcs(reinterpret_cast<float4*>(arow + h), lo4);
            __stcs(reinterpret_cast<float4*>(arow + h + 4), hi4);
          }
        }
      }
    };
    for (int c = 0; c < nch; ++c) {
      const int t0 = bos + c * kChunk, L = min(kChunk, len - c * kChunk);
      // ---- L2 prefetch of the next chunk's q, k and g (a box of 64 token rows
      // of one head each, one per thread of lanes 0 of warps 0-2), a whole
      // chunk period ahead of its loads.  (v needs none: its TMA copy is
      // issued as soon as the previous chunk's MMA2 is done.)
      if (lane == 0 && warp < 3 && c + 1 < nch) {
        const int tn = t0 + kChunk;
        const CUtensorMap* m = warp == 0 ? &maps.q : warp == 1 ? &maps.k : &maps.g;
        tma_prefetch_l2_3d(m, 0, warp < 2 ? hq : hv, tn);
      }
      // ---- loads (all in flight together)
      float2 g2[kRows];
      uint32_t q2[kRows], k2[kRows];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        const int i = kRows * quarter + rr;
        g2[rr] = make_float2(0.f, 0.f);
        q2[rr] = k2[rr] = 0u;
        if (i < L && kact) {
          const size_t tq = size_t(t0 + i) * P.Hq + hq, tv = size_t(t0 + i) * P.Hv + hv;
          g2[rr] = __ldg(reinterpret_cast<const float2*>(A.g + tv * K + c0));
          q2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(A.q) + tq * K + c0));
          k2[rr] = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(A.k) + tq * K + c0));
        }
      }
      // ---- last chunk's Aqk export while the loads are in flight (D1 holds
      // it until this iteration's MMA1)
      if (aqk_w && c >= 1) export_aqk(c - 1);
      // ---- cumsum offsets across the row quarters
      float* part = part_base + (c & 1) * 4 * K;
      if (kact) {
        float2 sum = make_float2(0.f, 0.f);
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          sum.x += g2[rr].x;
          sum.y += g2[rr].y;
        }
        *reinterpret_cast<float2*>(part + quarter * K + c0) = sum;
      }
      named_bar_sync(kNbPrep, kPrepThreadsF);
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
      // e^{G_r - G_i} is formed as the product of q e^{G_r} and k e^{-G_i}: both
      // stay normal fp32 numbers only while the chunk's log-decay on every
      // channel is at most KDA_MAX_CHUNK_LOG_DECAY.  Past it the chain is
      // marked, and the exact path recomputes it after this kernel.
      if (kact && quarter == 0 && fminf(glast.x, glast.y) < -KDA_MAX_CHUNK_LOG_DECAY)
        P.flags[size_t(n) * P.Hv + hv] = 1;
      // gated operands, all in registers before the waits: hi halves to the hi
      // tiles, lo halves to the lo area
      uint32_t qgh[kRows], kgh[kRows], kdh[kRows], qgl[kRows], kgl[kRows], kdl[kRows];
      if (kact) {
        f2 G2 = f2_make(G.x, G.y);
        const f2 kLog2e2 = f2_make(1.4426950408889634f, 1.4426950408889634f);
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int i = kRows * quarter + rr;
          G2 = f2_add(G2, f2_make(g2[rr].x, g2[rr].y));
          const f2 q = f2_from_bf16x2(q2[rr]);
          const f2 k = f2_from_bf16x2(k2[rr]);
          const float2 glv = f2_split(f2_mul(G2, kLog2e2));
          const f2 eG = f2_make(exp2f_fast(glv.x), exp2f_fast(glv.y));
          const f2 eN = f2_make(exp2f_fast(-glv.x), exp2f_fast(-glv.y));
          const f2 Qg = f2_mul(q, eG);
          const f2 Kg = f2_mul(k, eG);
          const f2 Kd = f2_mul(k, eN);
          qgl[rr] = split2(qgh[rr], Qg);
          kgl[rr] = split2(kgh[rr], Kg);
          kdl[rr] = split2(kdh[rr], Kd);
          if (i < L) {
            const size_t tok = size_t(t0 + i) * P.Hv + hv;
            if (A.G) *reinterpret_cast<float2*>(A.G + tok * K + c0) = f2_split(G2);
            if constexpr (kQG)
              *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(A.QG) + tok * K + c0) = qgh[rr];
          }
        }
      }
      // ---- hi buffer c%2 free once the state pass is done with chunk c-2; the
      // lo area once MMA1 of chunk c-1 is done
      if (c >= 2) wait_bar(&bar[bHiFree + (c & 1)], par((c >> 1) - 1), abort_flag, P.status);
      if (c >= 1) wait_bar(&bar[bD1Full], par(c - 1), abort_flag, P.status);
      __syncwarp();
      uint8_t* hi = sm + Lay::HI + (c & 1) * Lay::kHi;
      if (kact) {
        if (quarter == 0)
          *reinterpret_cast<float2*>(gam_base + (c & 1) * K + c0) = make_float2(__expf(glast.x), __expf(glast.y));
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const uint32_t swr = uint32_t(rr & 7) << 4, rowr = uint32_t(rr) * 128u;
          const uint32_t oq = (xA ^ swr) + rowr, od = (xB ^ swr) + rowr;
          *reinterpret_cast<uint32_t*>(hi + oq) = qgh[rr];
          *reinterpret_cast<uint32_t*>(hi + oq + 8192u) = kgh[rr];
          *reinterpret_cast<uint32_t*>(hi + Lay::kA1 + od) = kdh[rr];
          *reinterpret_cast<uint32_t*>(lo + oq) = qgl[rr];
          *reinterpret_cast<uint32_t*>(lo + oq + 8192u) = kgl[rr];
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();  // the Aqk export's D1 reads come before MMA1 overwrites D1
      named_bar_sync(kNbPrep, kPrepThreadsF);
      // ---- MMA1 (thread 0): hi*hi + lo*hi; atoms of 64 channels, A 128 rows
      // (1024 descriptor units apart), B 64 rows (512)
      constexpr uint32_t id = idesc_bf16_f32(128, 64);
      const uint32_t hi_addr = smem_u32(hi), lo_addr = smem_u32(lo);
      const uint64_t a_hi = sdesc_kmajor_sw128(hi_addr), b_hi = sdesc_kmajor_sw128(hi_addr + Lay::kA1);
      const uint64_t lo_d = sdesc_kmajor_sw128(lo_addr);
      if (mma_leader) {
        if (c >= 1) wait_bar(&bar[bD1Empty], par(c - 1), abort_flag, P.status);
        tc_fence_after();
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(tmem + kColD1, a_hi + at * 1024, b_hi + at * 512, id, at > 0);
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(tmem + kColD1, lo_d + at * 1024, b_hi + at * 512, id, 1);
        umma_commit(&bar[bLoA]);
      }
      __syncwarp();  // the issuer's warp-mates wait here rather than spin beside it
      // ---- Kd's low half into the area A1_lo used, once hi*hi + lo*hi is done
      wait_bar(&bar[bLoA], par(c), abort_flag, P.status);
      if (kact) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr)
          *reinterpret_cast<uint32_t*>(lo + (xB ^ (uint32_t(rr & 7) << 4)) + uint32_t(rr) * 128u) = kdl[rr];
      }
      fence_proxy_async_smem();
      named_bar_sync(kNbPrep, kPrepThreadsF);
      if (mma_leader) {
        tc_fence_after();
#pragma unroll
        for (int at = 0; at < K / 64; ++at) umma_atom4(tmem + kColD1, a_hi + at * 1024, lo_d + at * 512, id, 1);
        umma_commit(&bar[bD1Full]);
      }
      __syncwarp();
    }
    if (aqk_w && nch >= 1) export_aqk(nch - 1);
    if (mma_leader) {
      umma_commit(&bar[bDrain]);
      mbar_wait(&bar[bDrain], 0, kDrainNs);
    }

  } else if (warp < kWarpState0) {
    // ====================================================== intra epilogue
    regs_dec<kRegsIntra>();
    const int e = tid - kWarpIntra0 * 32;  // 0..127
    const int q4 = warp & 3;               // TMEM lane quadrant
    const bool akk = q4 >= 2;              // lanes 64-127: Kg rows of D1 (Akk); lanes 0-63: Qg rows (Aqk)
    const int r = 32 * (q4 & 1) + lane;    // row of the 64 x 64 matrix
    const bool leader = warp == kWarpIntra0 && lane == 0;
    float* Am = reinterpret_cast<float*>(sm + Lay::SCR);  // A = Akk (beta-scaled, strictly lower), fp32 64 x kLd
    float* Xm = Am + 64 * kLd;                            // X = (I + A)^-1
    float* sB = reinterpret_cast<float*>(sm + Lay::BETA);
    uint8_t* vt = sm + Lay::VT;
    // L2 prefetch of chunk cc's q, k, v, g (one TMA tensor prefetch each; the
    // prep warps prefetch the chunks after the first), and the TMA copy of its
    // v rows into the v tile (64-channel boxes, SWIZZLE_128B)
    auto prefetch = [&](int cc) {
      const int t = bos + cc * kChunk;
      tma_prefetch_l2_3d(&maps.q, 0, hq, t);
      tma_prefetch_l2_3d(&maps.k, 0, hq, t);
      tma_prefetch_l2_3d(&maps.v, 0, hv, t);
      tma_prefetch_l2_3d(&maps.g, 0, hv, t);
    };
    auto load_v = [&](int cc) {
      mbar_arrive_expect_tx(&bar[bVFull], uint32_t(V) * 64u * 2u);
#pragma unroll
      for (int a = 0; a < V / 64; ++a)
        tma_load_3d(vt + a * 8192, &maps.v_sw, a * 64, hv, bos + cc * kChunk, &bar[bVFull]);
    };
    if (leader) {
      prefetch(0);
      load_v(0);
    }
    // B2's entries above the diagonal are never written: clear the tile once
    for (int i = e; i < 64 * 64 * 2 / 16; i += 128)
      reinterpret_cast<uint4*>(sm + Lay::B2)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int c = 0; c < nch; ++c) {
      const int t0 = bos + c * kChunk, L = min(kChunk, len - c * kChunk);
      const float br = (akk && r < L) ? load_beta(A.beta, P.beta_fp32, size_t(t0 + r) * P.Hv + hv) : 0.f;
      wait_bar(&bar[bD1Full], par(c), abort_flag, P.status);
      tc_fence_after();
      // the whole row r of D1 (Aqk / scale or Akk / beta) into registers; D1
      // is then free for the next chunk's MMA1
      uint32_t x[64];
      tmem_ld_x64(tmem_addr(tmem, 32 * q4, kColD1), x);
      tc_fence_before();
      mbar_arrive(&bar[bD1Empty]);
      if (akk) {
        // row r of A: beta_r Akk[r][i] for i < r, zero elsewhere
        float* arow = Am + r * kLd;
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          float a4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) a4[j] = (i + j < r) ? br * __uint_as_float(x[i + j]) : 0.f;
          *reinterpret_cast<float4*>(arow + i) = make_float4(a4[0], a4[1], a4[2], a4[3]);
        }
        sB[r] = br;
      } else {
        // Aqk row r (causal mask): bf16 operand tile of O^T += Delta^T Aqk^T
        // (without scale: the state pass multiplies O by scale at the end);
        // the tile of chunk c-2 must be done
        if (c >= 2) wait_bar(&bar[bHiFree + (c & 1)], par((c >> 1) - 1), abort_flag, P.status);
        uint8_t* aqkb = sm + Lay::AQKB + (c & 1) * 8192;
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
          float f[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = (i + j <= r) ? __uint_as_float(x[i + j]) : 0.f;
          *reinterpret_cast<uint4*>(aqkb + sw128_offset(uint32_t(r), uint32_t(i), 64)) = pack8(f);
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(kNbIntra, 128);
      if (akk) {
        // ---- X = (I + A)^-1 by 16 x 16 blocks.  Diagonal blocks: forward
        // substitution, thread = (block d, column cc), on the threads that
        // wrote A; right-looking (once x[i] is final it leaves the rows below),
        // so the dependent chain is one FMA a row
        const int d = (e - 64) >> 4, cc = e & 15, base = 16 * d;
        const float* ab = Am + base * kLd + base;
        float xc[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) xc[rr] = rr == cc ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i)
#pragma unroll
          for (int rr = i + 1; rr < 16; ++rr) xc[rr] = fmaf(-ab[rr * kLd + i], xc[i], xc[rr]);
        uint8_t* b2 = sm + Lay::B2;
        const float bc = sB[base + cc];
        // MMA2 of the last chunk has read B2 (its completion is D2 full); the
        // barrier after this phase orders the R1 / R2 writers after it too
        if (c >= 1) wait_bar(&bar[bD2Full], par(c - 1), abort_flag, P.status);
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          Xm[(base + rr) * kLd + base + cc] = xc[rr];
          *reinterpret_cast<__nv_bfloat16*>(b2 + sw128_offset(uint32_t(base + rr), uint32_t(base + cc), 64)) =
              __float2bfloat16_rn(xc[rr] * bc);
        }
      }
      named_bar_sync(kNbIntra, 128);
      // The off-diagonal blocks on the warps' tensor cores (mma.m16n8k8 on
      // TF32 hi/lo pairs, fp32-accurate); each X block goes to the fp32 scratch
      // and, times beta of its columns, to the bf16 B2 tile (whose entries
      // above the diagonal are never written: zero since the kernel began).
      // 32 x 32 diagonal blocks first: X_10 = -X_11 (A_10 X_00) and
      // X_32 = -X_33 (A_32 X_22), T in the dead diagonal blocks A_00 / A_22;
      // warps 0, 1 the top block's column halves, warps 2, 3 the bottom's.
      uint8_t* b2 = sm + Lay::B2;
      {
        const int iw = warp - kWarpIntra0;
        const int co = (iw >> 1) ? 32 : 0, ro = co + 16, nb = 8 * (iw & 1);
        float d[4];
        mma_3xtf32_x1(d, Am + ro * kLd + co, kLd, Xm + co * kLd + co + nb, kLd, 0, 16);
        store_frag(Am + co * kLd + co + nb, kLd, d, 1.f);
        __syncwarp();  // the second product reads only the T columns this warp wrote
        float x[4];
        mma_3xtf32_x1(x, Xm + ro * kLd + ro, kLd, Am + co * kLd + co + nb, kLd, 0, 16);
        store_x_b2(Xm, b2, sB, ro, co + nb, x, -1.f);
      }
      named_bar_sync(kNbIntra, 128);
      // the lower-left 32 x 32 block: X_BL = -X_BR (A_BL X_TL), T_BL in the dead
      // top-left block of A.  Warp iw owns rows 16 (iw >> 1) .. + 15 and
      // columns 16 (iw & 1) .. + 15.  The blocks of X never written (above the
      // diagonal blocks) are skipped: X_TL's columns 16-31 take only the terms
      // 16-31, X_BR's rows 32-47 only the terms 32-47.
      {
        const int iw = warp - kWarpIntra0;
        const int mt = 16 * (iw >> 1), nt = 16 * (iw & 1);
        float d0[4], d1[4];
        mma_3xtf32_x2(d0, d1, Am + (32 + mt) * kLd, kLd, Xm + nt, kLd, nt, 32);
        store_frag(Am + mt * kLd + nt, kLd, d0, 1.f);
        store_frag(Am + mt * kLd + nt + 8, kLd, d1, 1.f);
        named_bar_sync(kNbIntra, 128);
        float x0[4], x1[4];
        mma_3xtf32_x2(x0, x1, Xm + (32 + mt) * kLd + 32, kLd, Am + nt, kLd, 0, mt + 16);
        store_x_b2(Xm, b2, sB, 32 + mt, nt, x0, -1.f);
        store_x_b2(Xm, b2, sB, 32 + mt, nt + 8, x1, -1.f);
      }
      // ---- v of this chunk: a tail chunk's rows past its end hold tokens of
      // the next chunk or sequence; clear them so that U depends on this
      // chunk's tokens alone
      wait_bar(&bar[bVFull], par(c), abort_flag, P.status);
      if (L < kChunk) {
        const int pieces = (kChunk - L) * 8;  // 16-byte pieces per 64-channel block
        for (int a = 0; a < V / 64; ++a)
          for (int i = e; i < pieces; i += 128)
            *reinterpret_cast<uint4*>(vt + a * 8192 + (L + (i >> 3)) * 128 + (i & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[bB2Ready]);  // B2, the v tail and the Aqk tile are ready: MMA2 may start
      named_bar_sync(kNbIntra, 128);  // every warp's X blocks are in the scratch

      // ---- Akk_inv = X (lower triangle), by whole rows from the scratch (8
      // passes of 8 rows x 16 column quads), while MMA2 runs; streaming stores
      if (A.Akk_inv) {
#pragma unroll 2
        for (int it = 0; it < 8; ++it) {
          const int row = 8 * it + (e >> 4), c4 = 4 * (e & 15);
          const float4 xv = *reinterpret_cast<const float4*>(Xm + row * kLd + c4);
          const float4 o4 = make_float4(c4 <= row ? xv.x : 0.f, c4 + 1 <= row ? xv.y : 0.f,
                                        c4 + 2 <= row ? xv.z : 0.f, c4 + 3 <= row ? xv.w : 0.f);
          if (row < L) __stcs(reinterpret_cast<float4*>(A.Akk_inv + (size_t(t0 + row) * P.Hv + hv) * 64 + c4), o4);
        }
      }
    }

  } else {
    // =============================================================== state
    regs_dec<kRegsState>();
    const int q4 = warp & 3;
    const int v = 32 * q4 + lane;  // TMEM lane: value channel v (S^T, U^T, P^T, O^T), channel k of W^T
    const bool vv = v < V, kk = v < K;
    const bool leader = warp == kWarpState0 && lane == 0;
    uint8_t* ust = sm + Lay::UST;
    const float* gam_base = reinterpret_cast<const float*>(sm + Lay::GAM);
    const uint32_t lane_base = tmem_addr(tmem, 32 * q4, 0);
    // In a token-major SWIZZLE_128B tile (64-channel atoms of 64 token rows x
    // 128 B, what a TMA store of a (64, 1, 64) box reads), this thread's
    // channel sits at byte swz[t % 8] of row t of its atom: the 16-byte chunk
    // index is XOR-ed by (row % 8).
    uint32_t swz[8];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) swz[r8] = ((uint32_t(((v & 63) >> 3) ^ r8)) << 4) | (uint32_t(v & 7) << 1);
    // 32 token rows t0 .. t0 + 31 of one channel (values x) into such a tile
    auto stage32 = [&](uint8_t* atom, int t0r, const uint32_t (&x)[32], float s) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        *reinterpret_cast<__nv_bfloat16*>(atom + (t0r + j) * 128 + swz[j & 7]) =
            __float2bfloat16_rn(s * __uint_as_float(x[j]));
    };
    // the same 32 values straight to a token-major global tensor (row stride
    // `stride` elements), rows past the chunk's end skipped
    auto store32 = [&](__nv_bfloat16* dst, size_t stride, int rows, const uint32_t (&x)[32], float s) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < rows) dst[size_t(j) * stride] = __float2bfloat16_rn(s * __uint_as_float(x[j]));
    };
    // S^T (fp32, columns j .. j + 31) into TMEM and its bf16 copy (the A operand)
    auto put_state = [&](int j, const uint32_t (&s)[32]) {
      tmem_st_x32(lane_base + kColS + j, s);
      uint32_t b[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] = pack_bf16x2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      tmem_st_x16(lane_base + kColSb + j / 2, b);
    };
    // initial state
#pragma unroll 1
    for (int j = 0; j < K; j += 32) {
      uint32_t s[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = __float_as_uint((A.h0 && vv) ? A.h0[(hrow + j + i) * V + v] : 0.f);
      put_state(j, s);
    }
    tmem_st_wait();
    tc_fence_before();
    named_bar_sync(kNbState, 128);
    constexpr uint32_t id64 = idesc_bf16_f32(128, 64);
    constexpr uint32_t idH = idesc_bf16_f32(128, K) | kIdescBMajorMN;
    for (int c = 0; c < nch; ++c) {
      const int t0 = bos + c * kChunk, L = min(kChunk, len - c * kChunk);
      const bool full = L == kChunk;  // a TMA box of 64 token rows stays inside the sequence
      uint8_t* hi = sm + Lay::HI + (c & 1) * Lay::kHi;
      const uint32_t hi_addr = smem_u32(hi);
      // ---- W^T (TMEM lane = channel k) into the W tile, token-major, in the
      // Kg rows of this chunk's A1_hi (MMA2 was their last reader): atom a at
      // hi + 16 KB a + 8 KB.  The intra warps signalled B2 ready after the
      // Aqk_b tile of chunk c was written, so D2 full also covers that tile.
      if (leader) {
        // MMA2: W^T = Kg^T B2^T, U^T = v^T B2^T (M = 128 channels, N = 64, K = 64
        // tokens), once the intra warps have written B2 (and cleared the v
        // tail); this pass is done with last chunk's W^T / U^T / P^T.  Kg is
        // read in place from the Kg rows of A1_hi as an MN-major operand (the
        // next 64 channels one A1 atom, 16 KB, further on); v from its TMA tile
        // (64-channel blocks 8 KB apart).  A K step of 16 tokens is 2048 B on the
        // A side, 32 B on B2.
        wait_bar(&bar[bB2Ready], par(c), abort_flag, P.status);
        tc_fence_after();
        constexpr uint32_t idmn = idesc_bf16_f32(128, 64) | kIdescAMajorMN;
        const uint64_t a_kg = sdesc_mnmajor_sw128(hi_addr + 8192, 16384);
        const uint64_t a_v = sdesc_mnmajor_sw128(smem_u32(sm + Lay::VT), 8192);
        const uint64_t b2 = sdesc_kmajor_sw128(smem_u32(sm + Lay::B2));
        umma_k4(tmem + kColW, a_kg, b2, idmn, 0, 2048 / 16, 2);
        umma_k4(tmem + kColU, a_v, b2, idmn, 0, 2048 / 16, 2);
        umma_commit(&bar[bD2Full]);
      }
      __syncwarp();
      wait_bar(&bar[bD2Full], par(c), abort_flag, P.status);
      tc_fence_after();
      if (leader && c + 1 < nch) {
        // MMA2 is done with the v tile: the TMA copy of the next chunk's v
        mbar_arrive_expect_tx(&bar[bVFull], uint32_t(V) * 64u * 2u);
#pragma unroll
        for (int a = 0; a < V / 64; ++a)
          tma_load_3d(sm + Lay::VT + a * 8192, &maps.v_sw, a * 64, hv, t0 + kChunk, &bar[bVFull]);
      }
      const bool w_tma = A.W && A.w_tma && full;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
        tmem_ld_x32(lane_base + kColW + 32 * h, w);
        if (kk) {
          stage32(hi + (v >> 6) * 16384 + 8192, 32 * h, w, 1.f);
          if (A.W && !w_tma)
            store32(reinterpret_cast<__nv_bfloat16*>(A.W) + (size_t(t0 + 32 * h) * P.Hv + hv) * K + v,
                    size_t(P.Hv) * K, L - 32 * h, w, 1.f);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (leader) bulk_wait_read_all();  // the last chunk's o store has read the U tile
      named_bar_sync(kNbState, 128);
      if (leader) {
        // P^T = S^T W^T into the W^T columns (read above), then O^T = S^T Qg^T;
        // A = S^T from TMEM, B = the W tile / the Qg rows (K-major, atoms 16 KB
        // apart); then the W tile's TMA store
        tc_fence_after();
        const uint64_t b_w = sdesc_kmajor_sw128(hi_addr + 8192), b_qg = sdesc_kmajor_sw128(hi_addr);
#pragma unroll
        for (int g = 0; g < K / 64; ++g) umma_ts4(tmem + kColW, tmem + kColSb + 32 * g, b_w + g * 1024, id64, g > 0, 2);
        umma_commit(&bar[bPDone]);
#pragma unroll
        for (int g = 0; g < K / 64; ++g)
          umma_ts4(tmem + kColO, tmem + kColSb + 32 * g, b_qg + g * 1024, id64, g > 0, 2);
        if (w_tma) {
#pragma unroll
          for (int a = 0; a < K / 64; ++a) tma_store_3d(&maps.W, hi + a * 16384 + 8192, a * 64, hv, t0);
          bulk_commit_group();
        }
      }
      __syncwarp();
      // ---- Delta^T row v = U^T - P^T (tokens past the chunk's end zero) into
      // TMEM as bf16 pairs; U^T to its staging tile (or straight out)
      wait_bar(&bar[bPDone], par(c), abort_flag, P.status);
      tc_fence_after();
      const bool u_tma = A.U && A.u_tma && full;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t ur[32];
        tmem_ld_x32(lane_base + kColU + 32 * h, ur);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t pr[16], dw[8];
          tmem_ld_x16(lane_base + kColW + 32 * h + 16 * q, pr);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int t = 32 * h + 16 * q + 2 * i;
            const float d0 = (vv && t < L) ? __uint_as_float(ur[16 * q + 2 * i]) - __uint_as_float(pr[2 * i]) : 0.f;
            const float d1 =
                (vv && t + 1 < L) ? __uint_as_float(ur[16 * q + 2 * i + 1]) - __uint_as_float(pr[2 * i + 1]) : 0.f;
            dw[i] = pack_bf16x2(d0, d1);
          }
          tmem_st_x8(lane_base + kColDt + 16 * h + 8 * q, dw);
        }
        if (A.U && vv) {
          if (u_tma)
            stage32(ust + (v >> 6) * 8192, 32 * h, ur, 1.f);
          else
            store32(reinterpret_cast<__nv_bfloat16*>(A.U) + (size_t(t0 + 32 * h) * P.Hv + hv) * V + v,
                    size_t(P.Hv) * V, L - 32 * h, ur, 1.f);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kNbState, 128);
      if (leader) {
        // S^T += Delta^T Kd (Kd token rows of B1_hi as an MN-major B: 64-channel
        // blocks 8 KB apart, a K step of 16 tokens 2048 B), O^T += Delta^T Aqk^T;
        // A = Delta^T from TMEM.  Then U's TMA store.
        tc_fence_after();
        const uint64_t b_kd = sdesc_mnmajor_sw128(hi_addr + Lay::kA1, 8192);
        const uint64_t b_aqk = sdesc_kmajor_sw128(smem_u32(sm + Lay::AQKB + (c & 1) * 8192));
        umma_ts4(tmem + kColS, tmem + kColDt, b_kd, idH, 1, 2048 / 16);
        umma_ts4(tmem + kColO, tmem + kColDt, b_aqk, id64, 1, 2);
        umma_commit(&bar[bHODone]);
        if (u_tma) {
#pragma unroll
          for (int a = 0; a < V / 64; ++a) tma_store_3d(&maps.U, ust + a * 8192, a * 64, hv, t0);
          bulk_commit_group();
        }
      }
      __syncwarp();
      wait_bar(&bar[bHODone], par(c), abort_flag, P.status);
      tc_fence_after();
      // ---- S <- gamma * (S + Kd^T Delta), in TMEM (fp32 and the bf16 A operand)
      const float* gm = gam_base + (c & 1) * K;
#pragma unroll 1
      for (int j = 0; j < K; j += 32) {
        uint32_t s[32];
        tmem_ld_x32(lane_base + kColS + j, s);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 g4 = *reinterpret_cast<const float4*>(gm + j + i);
          s[i] = __float_as_uint(__uint_as_float(s[i]) * g4.x);
          s[i + 1] = __float_as_uint(__uint_as_float(s[i + 1]) * g4.y);
          s[i + 2] = __float_as_uint(__uint_as_float(s[i + 2]) * g4.z);
          s[i + 3] = __float_as_uint(__uint_as_float(s[i + 3]) * g4.w);
        }
        put_state(j, s);
      }
      // ---- the W and U stores have read their tiles: the hi buffer (with its
      // gamma and Aqk tile) goes back to the prep and intra warps
      if (leader) bulk_wait_read_all();
      named_bar_sync(kNbState, 128);
      mbar_arrive(&bar[bHiFree + (c & 1)]);
      // ---- o = scale O^T, staged token-major in the U tile (its store is done)
      const bool o_tma = A.o_tma && full;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tmem_ld_x32(lane_base + kColO + 32 * h, o);
        if (vv) {
          if (o_tma)
            stage32(ust + (v >> 6) * 8192, 32 * h, o, P.scale);
          else
            store32(A.o + (size_t(t0 + 32 * h) * P.Hv + hv) * V + v, size_t(P.Hv) * V, L - 32 * h, o, P.scale);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kNbState, 128);
      if (leader && o_tma) {
#pragma unroll
        for (int a = 0; a < V / 64; ++a) tma_store_3d(&maps.o, ust + a * 8192, a * 64, hv, t0);
        bulk_commit_group();
      }
      __syncwarp();
      // (the next chunk's barrier after its W tile also orders these S^T
      // writes before its P MMA)
    }
    if (A.hT) {
#pragma unroll 1
      for (int j = 0; j < K; j += 32) {
        uint32_t s[32];
        tmem_ld_x32(lane_base + kColS + j, s);
        if (vv)
#pragma unroll
          for (int i = 0; i < 32; ++i) A.hT[(hrow + j + i) * V + v] = __uint_as_float(s[i]);
      }
    }
    if (leader) {
      // after an abort: the last v copy (issued here or by the intra leader) lands before exit
      mbar_wait(&bar[bVFull], par(nch - 1), kDrainNs);
      bulk_wait_all();
      umma_commit(&bar[bDrain + 1]);
      mbar_wait(&bar[bDrain + 1], 0, kDrainNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIntra0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int K, int V, bool kQG>
cudaError_t launch_fused_t(const Problem& P, const FusedArgs& A, const FusedMaps& maps, int dev, cudaStream_t s) {
  constexpr uint32_t smem = FusedLayout<K, V>::bytes;
  cudaError_t e = set_smem_once<fused_kernel<K, V, kQG>>(smem, dev);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)P.N * P.Hv;
  if (grid <= 0) return cudaSuccess;
  fused_kernel<K, V, kQG><<<unsigned(grid), kFusedThreads, smem, s>>>(P, A, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const Problem& P, const FusedArgs& A, const FusedMaps& maps, int dev, cudaStream_t s) {
  // The optional QG export has its own instantiations, so that the usual
  // prep loop carries none of its code.
  const bool qg = A.QG != nullptr;
  if (P.K == 128 && P.V == 128)
    return qg ? launch_fused_t<128, 128, true>(P, A, maps, dev, s) : launch_fused_t<128, 128, false>(P, A, maps, dev, s);
  if (P.K == 128 && P.V == 64)
    return qg ? launch_fused_t<128, 64, true>(P, A, maps, dev, s) : launch_fused_t<128, 64, false>(P, A, maps, dev, s);
  if (P.K == 64 && P.V == 128)
    return qg ? launch_fused_t<64, 128, true>(P, A, maps, dev, s) : launch_fused_t<64, 128, false>(P, A, maps, dev, s);
  if (P.K == 64 && P.V == 64)
    return qg ? launch_fused_t<64, 64, true>(P, A, maps, dev, s) : launch_fused_t<64, 64, false>(P, A, maps, dev, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
