// Inter-chunk state pass and output: one CTA per (sequence, value head),
// sequential over the sequence's chunks, with the K x V state on chip.
// This is the delta-H state kernel plus the output kernel of cuLA
// REPO_LAYOUT.md (ops/chunk_delta_h.py, ops/fwd_o.py), fused.
//
// Everything is computed transposed so that every MMA has M = 128 (the value
// channel v, one TMEM lane per v) and all operands are K-major SWIZZLE_128B:
//   P^T  = S^T W^T                  (M=128 v, N=64,  K=K)   TMEM cols 128b ..      (2 buffers)
//   O^T  = S^T Qs^T                 (M=128 v, N=64,  K=K)   TMEM cols 128b+64 ..
//   H^T  = Delta^T Kl               (M=128 v, N=K,   K=64)  TMEM cols 256 ..  (Kl MN-major)
//   O^T += Delta^T Aqk^T            (M=128 v, N=64,  K=64)  TMEM cols 128b+64 ..
// issued in that order, so that P and H, which gate the chunk chain, land first.
// with Delta = U - W S (rows past the chunk's L valid rows forced to 0),
// Qs = scale q e^G, Kl = k e^{G_last - G}, and the update
//   S <- Diag(e^{G_last}) S + Kl^T Delta.
// Two epilogue threads per value channel v (one per half of the columns)
// keep column v of S in fp32 registers, K/2 values each, and write their
// halves of row v of the A operand S^T for the next chunk.
//
// Warp roles: warp 0 issues TMA loads (and L2 prefetches one ring depth
// ahead, so that the stage loads hit L2), warp 1 issues the MMAs, warps 2-9
// (256 threads, two per TMEM lane quadrant) run the epilogue.  Two rings: ring A (MMA operands [W; Qs],
// Aqk, Kl as token rows; 2 stages) is released by the MMAs' own completion, so the next
// loads start mid-chunk; ring B (U and gamma, read by the epilogue; 3 stages)
// is released by the epilogue.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kEpiParts = 2;      // epilogue warps per TMEM lane quadrant (column split)
constexpr int kEpiThreads = 128 * kEpiParts;
constexpr int kStateThreads = 64 + kEpiThreads;
constexpr int kStagesA = 2;
constexpr int kStagesB = 3;

template <int K, int V>
struct StateLayout {
  // ring A stage.  W and Qs form one 128-row B operand [W; Qs]: atom a
  // (columns 64a..64a+63) holds the 64 W rows then the 64 Qs rows.
  static constexpr uint32_t WQ = 0;                       // 128 x K, K-major SW128
  static constexpr uint32_t Aqk = WQ + 128 * K * 2;       // 64 x 64
  static constexpr uint32_t Kl = Aqk + 64 * 64 * 2;       // 64 token rows x K, 64-channel blocks 8 KB apart
  static constexpr uint32_t stageA_bytes = ((Kl + K * 64 * 2) + 1023) / 1024 * 1024;
  // ring B stage
  static constexpr uint32_t U = 0;                        // 64 x V, plain row-major
  static constexpr uint32_t gam = U + 64 * V * 2;         // K floats
  static constexpr uint32_t stageB_bytes = ((gam + K * 4) + 1023) / 1024 * 1024;
  static constexpr uint32_t ringB = kStagesA * stageA_bytes;
  static constexpr uint32_t S = ringB + kStagesB * stageB_bytes;  // 128 x K, K-major SW128 (A operand S^T)
  static constexpr uint32_t D = S + 128 * K * 2;          // 128 x 64 (A operand Delta^T)
  static constexpr uint32_t bars = D + 128 * 64 * 2;      // fullA[2], emptyA[2], fullB[3], emptyB[3], P, H, sready, dready, O
  static constexpr uint32_t tmem_slot = bars + 16 * 8;
  static constexpr uint32_t abort_slot = tmem_slot + 4;
  static constexpr uint32_t total = abort_slot + 4;
  static constexpr uint32_t bytes = total + 1024;
  static constexpr uint32_t tmem_cols = 512;  // [P|O] x2 at 0 / 128, H at 256
  static constexpr uint32_t txA_bytes = 128 * K * 2 + 64 * 64 * 2 + K * 64 * 2;
  static constexpr uint32_t txB_bytes = 64 * V * 2 + K * 4;
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

// Columns k0 .. k0 + KH - 1 of row v of the A operand S^T (bf16, K-major SW128).
template <int KH>
__device__ __forceinline__ void store_state_part(uint8_t* sS, int v, int k0, const float (&S)[KH]) {
#pragma unroll
  for (int c = 0; c < KH; c += 8) {
    const uint4 pk = make_uint4(pack_bf16x2(S[c], S[c + 1]), pack_bf16x2(S[c + 2], S[c + 3]),
                                pack_bf16x2(S[c + 4], S[c + 5]), pack_bf16x2(S[c + 6], S[c + 7]));
    *reinterpret_cast<uint4*>(sS + sw128_offset(v, k0 + c, 128)) = pk;
  }
}

// Warp-collective TMEM load of N (16, 32 or 64) consecutive columns.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 64) {
    tmem_ld_x64(taddr, r);
  } else if constexpr (N == 32) {
    tmem_ld_x32(taddr, r);
  } else {
    static_assert(N == 16, "16, 32 or 64 columns");
    tmem_ld_x16(taddr, r);
  }
}

template <int K, int V>
__global__ void __launch_bounds__(kStateThreads, 1)
    state_kernel(const Problem P, const __grid_constant__ StateMaps maps, const float* __restrict__ gamma,
                 const float* __restrict__ h0, __nv_bfloat16* __restrict__ o, float* __restrict__ hT) {
  using Lay = StateLayout<K, V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int hv = blockIdx.x % P.Hv;
  const int n = P.varlen ? P.seq_order[blockIdx.x / P.Hv] : blockIdx.x / P.Hv;  // longest chains first
  // an earlier error (bad cu_seqlens, another kernel's failure) stops the
  // whole CTA: one thread reads the status word, so that every thread takes
  // the same branch before the CTA's barriers
  if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<volatile int32_t*>(P.status) != 0)) return;
  int bos, len, gc0;
  if (P.varlen) {
    bos = P.cu[n];
    len = P.cu[n + 1] - bos;
    gc0 = P.chunk_off[n];
  } else {
    bos = n * P.T;
    len = P.T;
    gc0 = n * P.NT;
  }
  const int nch = (len + kChunk - 1) / kChunk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* fullA = reinterpret_cast<uint64_t*>(sm + Lay::bars);
  uint64_t* emptyA = fullA + 2;
  uint64_t* fullB = fullA + 4;
  uint64_t* emptyB = fullA + 7;
  uint64_t* bar_P = fullA + 10;
  uint64_t* bar_H = fullA + 11;
  uint64_t* sready = fullA + 12;
  uint64_t* dready = fullA + 13;
  uint64_t* bar_O = fullA + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::tmem_slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::abort_slot);

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&emptyA[s], 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&fullB[s], 1);
      mbar_init(&emptyB[s], kEpiThreads / 32);
    }
    mbar_init(bar_P, 1);
    mbar_init(bar_H, 1);
    mbar_init(sready, kEpiThreads);
    mbar_init(dready, kEpiThreads);
    mbar_init(bar_O, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Lay::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto prefetch = [&](int c) {
        const int t0 = bos + c * kChunk;
        const int gc = gc0 + c;
#pragma unroll
        for (int a = 0; a < K / 64; ++a) {
          tma_prefetch_l2_3d(&maps.W, a * 64, hv, t0);
          tma_prefetch_l2_3d(&maps.Qs, a * 64, hv, t0);
        }
        tma_prefetch_l2_3d(&maps.Aqk_b, 0, hv, t0);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) tma_prefetch_l2_3d(&maps.Kl, a * 64, hv, t0);
        tma_prefetch_l2_3d(&maps.U, 0, hv, t0);
        bulk_prefetch_l2(gamma + (size_t(gc) * P.Hv + hv) * K, K * 4);
      };
      // L2 prefetch as far ahead as ring A is deep: the chunk whose loads this
      // slot issues next.  Further ahead, lines are evicted before their load
      // at this kernel's traffic (about 2x the DRAM reads for 5 chunks ahead).
      constexpr int kAhead = kStagesA;
      for (int c = 0; c < nch && c < kAhead; ++c) prefetch(c);
      for (int c = 0; c < nch; ++c) {
        if (c + kAhead < nch) prefetch(c + kAhead);
        const int t0 = bos + c * kChunk;
        const int gc = gc0 + c;
        const int sa = c % kStagesA, sb = c % kStagesB;
        if (c >= kStagesA) wait_bar(&emptyA[sa], (c / kStagesA - 1) & 1, abort_flag, P.status);
        uint8_t* st = sm + sa * Lay::stageA_bytes;
        mbar_arrive_expect_tx(&fullA[sa], Lay::txA_bytes);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) {
          tma_load_3d(st + Lay::WQ + a * 128 * 128, &maps.W, a * 64, hv, t0, &fullA[sa]);
          tma_load_3d(st + Lay::WQ + a * 128 * 128 + 64 * 128, &maps.Qs, a * 64, hv, t0, &fullA[sa]);
        }
        tma_load_3d(st + Lay::Aqk, &maps.Aqk_b, 0, hv, t0, &fullA[sa]);
#pragma unroll
        for (int a = 0; a < K / 64; ++a) tma_load_3d(st + Lay::Kl + a * 64 * 128, &maps.Kl, a * 64, hv, t0, &fullA[sa]);
        if (c >= kStagesB) wait_bar(&emptyB[sb], (c / kStagesB - 1) & 1, abort_flag, P.status);
        uint8_t* sbp = sm + Lay::ringB + sb * Lay::stageB_bytes;
        mbar_arrive_expect_tx(&fullB[sb], Lay::txB_bytes);
        tma_load_3d(sbp + Lay::U, &maps.U, 0, hv, t0, &fullB[sb]);
        bulk_load(sbp + Lay::gam, gamma + (size_t(gc) * P.Hv + hv) * K, K * 4, &fullB[sb]);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id64 = idesc_bf16_f32(128, 64);
      constexpr uint32_t idK = idesc_bf16_f32(128, K);
      const uint32_t sS = smem_u32(sm + Lay::S), sD = smem_u32(sm + Lay::D);
      for (int c = 0; c < nch; ++c) {
        const int sa = c % kStagesA;
        const uint32_t st = smem_u32(sm + sa * Lay::stageA_bytes);
        const uint32_t pcol = 128 * (c & 1), ocol = pcol + 64;
        wait_bar(&fullA[sa], (c / kStagesA) & 1, abort_flag, P.status);
        wait_bar(sready, c & 1, abort_flag, P.status);
        tc_fence_after();
        // P^T = S^T W^T first (it gates the chain), then O^T = S^T Qs^T: the W
        // rows are rows 0-63 and the Qs rows 64-127 of every 128-row atom.
        umma_kloop(tmem + pcol, sS, 128, st + Lay::WQ, 128, K / 16, id64, 0);
        umma_commit(bar_P);
        umma_kloop(tmem + ocol, sS, 128, st + Lay::WQ + 64 * 128, 128, K / 16, id64, 0);
        wait_bar(dready, c & 1, abort_flag, P.status);
        tc_fence_after();
        // H^T = Delta^T Kl first (it gates the next chunk), then O^T += Delta^T Aqk^T.
        // Kl is MN-major (token rows): a K step of 16 tokens is 2048 B.
        umma_k4(tmem + 256, sdesc_kmajor_sw128(sD), sdesc_mnmajor_sw128(st + Lay::Kl, 64 * 128),
                idK | kIdescBMajorMN, 0, 2, 2048 / 16);
        umma_commit(bar_H);
        umma_kloop(tmem + ocol, sD, 128, st + Lay::Aqk, 64, 4, id64, 1);
        umma_commit(bar_O);
        umma_commit(&emptyA[sa]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warps 2-9.  Warp w reads TMEM lane quadrant w % 4 (thread = value
    // channel v); the two warps on a quadrant split the columns: half 0 takes
    // tokens 0-31 of Delta and O and state channels 0 .. K/2 - 1, half 1 the rest.
    constexpr int KH = K / kEpiParts;   // state channels per thread
    constexpr int RH = 64 / kEpiParts;  // tokens of Delta and O per thread
    const int q4 = warp & 3;
    const int half = (warp - 2) >> 2;   // column part 0 .. kEpiParts - 1
    const int v = 32 * q4 + lane;
    const bool vv = v < V;
    const int k0 = KH * half, r0 = RH * half;
    uint8_t* sS = sm + Lay::S;
    uint8_t* sD = sm + Lay::D;
    float S[KH];  // S[k0 + j][v]
    const size_t hbase = (size_t(n) * P.Hv + hv) * K;
#pragma unroll
    for (int j = 0; j < KH; ++j) S[j] = (h0 && vv) ? h0[(hbase + k0 + j) * V + v] : 0.f;
    store_state_part<KH>(sS, v, k0, S);
    fence_proxy_async_smem();
    mbar_arrive(sready);
    for (int c = 0; c < nch; ++c) {
      const int sb = c % kStagesB;
      const uint8_t* st = sm + Lay::ringB + sb * Lay::stageB_bytes;
      const int t0 = bos + c * kChunk;
      const int L = min(kChunk, len - c * kChunk);
      const uint32_t pcol = 128 * (c & 1), ocol = pcol + 64;
      // Delta^T row v, tokens r0 .. r0 + 31: U[:, v] - P^T row v, rows >= L zeroed
      // U[:, v] of this part's rows is read before P lands
      wait_bar(&fullB[sb], (c / kStagesB) & 1, abort_flag, P.status);
      const __nv_bfloat16* sU = reinterpret_cast<const __nv_bfloat16*>(st + Lay::U);
      float u[RH];
#pragma unroll
      for (int e = 0; e < RH; ++e) u[e] = vv ? __bfloat162float(sU[(r0 + e) * V + v]) : 0.f;
      wait_bar(bar_P, c & 1, abort_flag, P.status);
      tc_fence_after();
      {
        uint32_t pr[RH];
        tmem_ld_n<RH>(tmem_addr(tmem + pcol, 32 * q4, r0), pr);
#pragma unroll
        for (int j = 0; j < RH; j += 8) {
          float d[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = r0 + j + e;
            d[e] = (i < L) ? u[j + e] - __uint_as_float(pr[j + e]) : 0.f;
          }
          const uint4 pk = make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                      pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7]));
          *reinterpret_cast<uint4*>(sD + sw128_offset(v, r0 + j, 128)) = pk;
        }
      }
      if (L < kChunk) {
        // tail chunk: the Kl box's rows L..63 hold tokens of the next chunk or
        // sequence; clear them before the state MMA, so that the state depends
        // on this chunk's tokens alone (their Delta rows are exact zeros)
        const int sa = c % kStagesA;
        wait_bar(&fullA[sa], (c / kStagesA) & 1, abort_flag, P.status);
        uint8_t* kl = sm + sa * Lay::stageA_bytes + Lay::Kl;
        const int tail = kChunk - L, pieces = tail * (K / 64) * 8;  // 16-byte pieces
        for (int idx = tid - 64; idx < pieces; idx += kEpiThreads) {
          const int row = idx >> 3, blk = row / tail, rw = L + row % tail;
          *reinterpret_cast<uint4*>(kl + blk * 64 * 128 + rw * 128 + (idx & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(dready);
      // state update S <- gamma * S + H on channels k0 .. k0 + KH - 1: the
      // decay is applied while the state MMA runs, H is added when it lands
      const float* sg = reinterpret_cast<const float*>(st + Lay::gam) + k0;
#pragma unroll
      for (int j = 0; j < KH; ++j) S[j] *= sg[j];
      wait_bar(bar_H, c & 1, abort_flag, P.status);
      tc_fence_after();
      {
        uint32_t hr[KH];
        tmem_ld_n<KH>(tmem_addr(tmem + 256 + k0, 32 * q4, 0), hr);
#pragma unroll
        for (int j = 0; j < KH; ++j) S[j] += __uint_as_float(hr[j]);
      }
      store_state_part<KH>(sS, v, k0, S);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(sready);
      __syncwarp();
      if (lane == 0) mbar_arrive(&emptyB[sb]);
      // O of this chunk sits in its own TMEM buffer; the next chunk writes the
      // other one, and the chunk after that waits for this thread's next
      // sready arrival, which comes after these loads.
      wait_bar(bar_O, c & 1, abort_flag, P.status);
      tc_fence_after();
      {
        uint32_t orow[RH];
        tmem_ld_n<RH>(tmem_addr(tmem + ocol, 32 * q4, r0), orow);
        if (vv) {
          __nv_bfloat16* op = o + (size_t(t0 + r0) * P.Hv + hv) * V + v;
          const size_t ostride = size_t(P.Hv) * V;
#pragma unroll
          for (int r = 0; r < RH; ++r)
            if (r0 + r < L) op[size_t(r) * ostride] = __float2bfloat16_rn(__uint_as_float(orow[r]));
        }
      }
    }
    if (hT && vv) {
#pragma unroll
      for (int j = 0; j < KH; ++j) hT[(hbase + k0 + j) * V + v] = S[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::tmem_cols);
  }
}

template <int K, int V>
cudaError_t launch_state_t(const Problem& P, const StateMaps& maps, const float* gamma, const float* h0, void* o,
                           float* hT, int dev, cudaStream_t s) {
  constexpr uint32_t smem = StateLayout<K, V>::bytes;
  cudaError_t e = set_smem_once<state_kernel<K, V>>(smem, dev);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)P.N * P.Hv;
  if (grid <= 0) return cudaSuccess;
  state_kernel<K, V><<<unsigned(grid), kStateThreads, smem, s>>>(P, maps, gamma, h0,
                                                                  reinterpret_cast<__nv_bfloat16*>(o), hT);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state(const Problem& P, const StateMaps& maps, const float* gamma, const float* h0, void* o,
                         float* hT, int dev, cudaStream_t s) {
  if (P.K == 128 && P.V == 128) return launch_state_t<128, 128>(P, maps, gamma, h0, o, hT, dev, s);
  if (P.K == 128 && P.V == 64) return launch_state_t<128, 64>(P, maps, gamma, h0, o, hT, dev, s);
  if (P.K == 64 && P.V == 128) return launch_state_t<64, 128>(P, maps, gamma, h0, o, hT, dev, s);
  if (P.K == 64 && P.V == 64) return launch_state_t<64, 64>(P, maps, gamma, h0, o, hT, dev, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
