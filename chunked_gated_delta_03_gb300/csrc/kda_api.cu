// Host side of the C ABI declared in include/kda.h: argument checks, the
// workspace layout, TMA tensor maps, and the kernel launch sequence.
// Nothing here allocates device memory or synchronises a stream, except
// kda_get_device_status, whose job is to read the status word back.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tiled map over a token-major tensor [BT, H, D] viewed as (D, H, BT), boxes
// of (box_d, 1, 64).
bool map_tokens(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int D, int H, long long BT,
                int box_d, CUtensorMapSwizzle sw) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(BT)};
  cuuint64_t strides[2] = {cuuint64_t(D) * esize, cuuint64_t(H) * D * esize};
  cuuint32_t box[3] = {cuuint32_t(box_d), 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Layout {
  size_t status = 0, nc = 4, flags = 0, flags_bytes = 0, idx = 0, off = 0, order = 0, Qs = 0, Aqk_b = 0, Kl = 0,
         gamma = 0, W = 0, U = 0, total = 0;
};

struct Shape {
  int B, T, Hq, Hv, K, V, N, varlen, NT, nc_max;
  long long BT;
};

// What a call runs: the intra-chunk primitive alone, the two-pass forward, or
// the fused forward.
enum class Mode { kIntra, kTwoPass, kFused };

// Validates the sizes (not the pointers) and fills the derived counts.
int check_shape(const KdaArgs* a, Shape* s) {
  if (!a) return KDA_ERR_INVALID;
  if (a->chunk <= 0) return KDA_ERR_INVALID;
  if (a->chunk != kChunk) return KDA_ERR_UNSUPPORTED;
  if (a->B < 1 || a->T < 0 || a->Hq < 1 || a->Hv < 1 || a->Hv % a->Hq != 0) return KDA_ERR_INVALID;
  if ((a->K != 64 && a->K != 128) || (a->V != 64 && a->V != 128)) return KDA_ERR_UNSUPPORTED;
  if (a->beta_dtype != KDA_DTYPE_BF16 && a->beta_dtype != KDA_DTYPE_FP32) return KDA_ERR_INVALID;
  if ((a->chunk_indices == nullptr) != (a->chunk_offsets == nullptr)) return KDA_ERR_INVALID;
  s->B = a->B;
  s->T = a->T;
  s->Hq = a->Hq;
  s->Hv = a->Hv;
  s->K = a->K;
  s->V = a->V;
  s->varlen = a->cu_seqlens != nullptr;
  s->BT = (long long)a->B * a->T;
  if (s->varlen) {
    if (a->B != 1 || a->N < 0) return KDA_ERR_INVALID;
    s->N = a->N;
    s->NT = 0;
    s->nc_max = s->N > 0 ? a->T / kChunk + s->N : 0;
  } else {
    s->N = a->B;
    s->NT = (a->T + kChunk - 1) / kChunk;
    s->nc_max = a->B * s->NT;
  }
  // 32-bit TMA coordinates and grid sizes
  if (s->BT >= (1ll << 31) || (long long)s->nc_max * s->Hv * s->K >= (1ll << 31) ||
      (long long)s->N * s->Hv >= (1ll << 31))
    return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// The forward's kernels for these arguments (enum kda_path).
int forward_mode(const KdaArgs* a, Mode* m) {
  switch (a->path) {
    case KDA_PATH_AUTO: *m = a->intra_tf32 ? Mode::kTwoPass : Mode::kFused; return KDA_OK;
    case KDA_PATH_FUSED:
      if (a->intra_tf32) return KDA_ERR_UNSUPPORTED;
      *m = Mode::kFused;
      return KDA_OK;
    case KDA_PATH_TWO_PASS: *m = Mode::kTwoPass; return KDA_OK;
    default: return KDA_ERR_INVALID;
  }
}

Layout make_layout(const Shape& s, const KdaArgs* a, Mode mode) {
  Layout L;
  size_t p = kAlign;  // header: status word, chunk count
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes);
    return at;
  };
  // per-chain flags of the exact path, cleared with the header by one memset
  L.flags_bytes = size_t(s.N) * s.Hv * 4;
  L.flags = take(L.flags_bytes);
  if (s.varlen && mode != Mode::kFused && !a->chunk_indices) {
    L.idx = take(size_t(s.nc_max > 0 ? s.nc_max : 1) * 2 * 4);
    L.off = take(size_t(s.N + 1) * 4);
  }
  if (s.varlen && mode != Mode::kIntra) L.order = take(size_t(s.N > 0 ? s.N : 1) * 4);
  if (mode == Mode::kTwoPass) {
    L.Qs = take(size_t(s.BT) * s.Hv * s.K * 2);
    L.Aqk_b = take(size_t(s.BT) * s.Hv * 64 * 2);
    L.Kl = take(size_t(s.BT) * s.Hv * s.K * 2);
    L.gamma = take(size_t(s.nc_max) * s.Hv * s.K * 4);
    if (!a->W) L.W = take(size_t(s.BT) * s.Hv * s.K * 2);
    if (!a->U) L.U = take(size_t(s.BT) * s.Hv * s.V * 2);
  }
  L.total = p;
  return L;
}

// Device facts queried once per device: whether it is sm_103, and its SM count.
struct DeviceInfo {
  int dev = -1, sms = 0;
};

int device_info(DeviceInfo* out) {
  static std::atomic<int> state[kMaxDevicesCached];  // 0 unknown, 1 sm_103, -1 other
  static std::atomic<int> sm_count[kMaxDevicesCached];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_ARCH;
  if (dev >= 0 && dev < kMaxDevicesCached && state[dev].load(std::memory_order_acquire) != 0) {
    if (state[dev].load(std::memory_order_relaxed) < 0) return KDA_ERR_ARCH;
    out->dev = dev;
    out->sms = sm_count[dev].load(std::memory_order_relaxed);
    return KDA_OK;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_ARCH;
  }
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < kMaxDevicesCached) {
    sm_count[dev].store(sms, std::memory_order_relaxed);
    state[dev].store(ok ? 1 : -1, std::memory_order_release);
  }
  if (!ok) return KDA_ERR_ARCH;
  out->dev = dev;
  out->sms = sms;
  return KDA_OK;
}

int check_arch() {
  DeviceInfo d;
  return device_info(&d);
}

// Inputs may be NULL only when there are no tokens (empty tensors have no storage).
int check_inputs(const KdaArgs* a, const void* ws, long long BT) {
  if (BT > 0 && (!a->q || !a->k || !a->v || !a->g || !a->beta)) return KDA_ERR_INVALID;
  const void* ptrs[] = {a->q, a->k, a->v, a->g, a->beta, a->cu_seqlens, a->initial_state, a->o,
                        a->final_state, a->Aqk, a->Akk_inv, a->W, a->U, a->G, a->QG};
  // the chunk table is read with 4-byte loads only
  if ((reinterpret_cast<uintptr_t>(a->chunk_indices) | reinterpret_cast<uintptr_t>(a->chunk_offsets)) & 3u)
    return KDA_ERR_MISALIGNED;
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return KDA_ERR_MISALIGNED;
  return KDA_OK;
}

Problem make_problem(const Shape& s, const KdaArgs* a, uint8_t* ws, const Layout& L) {
  Problem P{};
  P.B = s.B;
  P.T = s.T;
  P.Hq = s.Hq;
  P.Hv = s.Hv;
  P.K = s.K;
  P.V = s.V;
  P.N = s.N;
  P.NT = s.NT;
  P.nc_max = s.nc_max;
  P.varlen = s.varlen;
  P.beta_fp32 = a->beta_dtype == KDA_DTYPE_FP32;
  P.tf32 = a->intra_tf32 != 0;
  P.scale = a->scale;
  P.cu = a->cu_seqlens;
  P.status = reinterpret_cast<int32_t*>(ws + L.status);
  P.flags = reinterpret_cast<int32_t*>(ws + L.flags);
  if (s.varlen) {
    if (a->chunk_indices) {
      P.chunk_idx = a->chunk_indices;
      P.chunk_off = a->chunk_offsets;
      P.nc_dev = a->chunk_offsets + s.N;  // chunk_offsets[N] = number of chunks
    } else if (L.idx) {
      P.chunk_idx = reinterpret_cast<const int32_t*>(ws + L.idx);
      P.chunk_off = reinterpret_cast<const int32_t*>(ws + L.off);
      P.nc_dev = reinterpret_cast<const int32_t*>(ws + L.nc);
    }
    if (L.order) P.seq_order = reinterpret_cast<const int32_t*>(ws + L.order);
  }
  return P;
}

// Shared front half of the entry points: checks, status reset, varlen chunk
// metadata.  kIntra (kda_fwd_intra) needs its four outputs; the forward modes
// need o.  Outputs may be NULL only when there are no tokens.
int prologue(const KdaArgs* a, void* workspace, size_t ws_bytes, cudaStream_t st, Mode mode, Shape* s, Layout* L,
             DeviceInfo* d) {
  int rc = check_shape(a, s);
  if (rc) return rc;
  if (!workspace) return KDA_ERR_INVALID;
  if (s->BT > 0 && (mode != Mode::kIntra ? !a->o : (!a->Aqk || !a->Akk_inv || !a->W || !a->U)))
    return KDA_ERR_INVALID;
  rc = check_inputs(a, workspace, s->BT);
  if (rc) return rc;
  *L = make_layout(*s, a, mode);
  if (ws_bytes < L->total) return KDA_ERR_WORKSPACE;
  rc = device_info(d);
  if (rc) return rc;
  if (!encode_fn()) return KDA_ERR_LAUNCH;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(ws, 0, L->flags + L->flags_bytes, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (s->varlen && s->N > 0) {
    int32_t* status = reinterpret_cast<int32_t*>(ws + L->status);
    if (a->chunk_indices) {
      if (launch_check_table(a->cu_seqlens, s->N, s->T, kChunk, a->chunk_indices, a->chunk_offsets, status, st) !=
          cudaSuccess)
        return KDA_ERR_LAUNCH;
    } else if (mode != Mode::kFused) {
      if (launch_chunk_index(a->cu_seqlens, s->N, s->T, kChunk, reinterpret_cast<int32_t*>(ws + L->idx),
                             reinterpret_cast<int32_t*>(ws + L->off), reinterpret_cast<int32_t*>(ws + L->nc), status,
                             st) != cudaSuccess)
        return KDA_ERR_LAUNCH;
    }
    if (mode != Mode::kIntra &&
        launch_seq_order(a->cu_seqlens, s->N, s->T, kChunk, reinterpret_cast<int32_t*>(ws + L->order), status,
                         st) != cudaSuccess)
      return KDA_ERR_LAUNCH;
  }
  return KDA_OK;
}

bool make_intra_maps(const Shape& s, const KdaArgs* a, IntraMaps* m) {
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
  return map_tokens(&m->q, a->q, bf, 2, s.K, s.Hq, s.BT, s.K, none) &&
         map_tokens(&m->k, a->k, bf, 2, s.K, s.Hq, s.BT, s.K, none) &&
         map_tokens(&m->v, a->v, bf, 2, s.V, s.Hv, s.BT, s.V, none) &&
         map_tokens(&m->g, a->g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.K, s.Hv, s.BT, s.K, none) &&
         map_tokens(&m->v_sw, a->v, bf, 2, s.V, s.Hv, s.BT, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

int run_intra(const Shape& s, const KdaArgs* a, const Problem& P, const IntraOut& out, const DeviceInfo& d,
              cudaStream_t st) {
  const IntraInputs in{a->q, a->k, a->v, a->g, a->beta};
  IntraMaps m;
  if (!make_intra_maps(s, a, &m)) return KDA_ERR_LAUNCH;
  return launch_intra(P, in, out, m, d.dev, d.sms, st) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// No tokens: the final state is the initial state.
int empty_forward(const Shape& s, const KdaArgs* a, cudaStream_t st) {
  if (!a->final_state) return KDA_OK;
  const size_t bytes = size_t(s.N) * s.Hv * s.K * s.V * 4;
  const cudaError_t e = a->initial_state
                            ? cudaMemcpyAsync(a->final_state, a->initial_state, bytes, cudaMemcpyDeviceToDevice, st)
                            : cudaMemsetAsync(a->final_state, 0, bytes, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// The exact path: recomputes the chains the tensor-core kernels marked (a
// chunk past the gate range); a chain left unmarked costs one flag read.
int run_exact(const KdaArgs* a, const Problem& P, const DeviceInfo& d, bool state, cudaStream_t st) {
  ExactArgs x{};
  x.q = a->q;
  x.k = a->k;
  x.v = a->v;
  x.g = a->g;
  x.beta = a->beta;
  x.h0 = a->initial_state;
  x.o = reinterpret_cast<__nv_bfloat16*>(a->o);
  x.hT = a->final_state;
  x.Aqk = a->Aqk;
  x.Akk_inv = a->Akk_inv;
  x.W = a->W;
  x.U = a->U;
  x.G = a->G;
  x.QG = a->QG;
  x.flags = P.flags;
  x.state = state ? 1 : 0;
  return launch_exact(P, x, d.dev, st) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

int two_pass_forward(const Shape& s, const KdaArgs* a, uint8_t* ws, const Layout& L, const DeviceInfo& d,
                     cudaEvent_t const* ev, cudaStream_t st) {
  const Problem P = make_problem(s, a, ws, L);
  IntraOut out{};
  out.Aqk = a->Aqk;
  out.Akk_inv = a->Akk_inv;
  out.W = a->W ? a->W : ws + L.W;
  out.U = a->U ? a->U : ws + L.U;
  out.G = a->G;
  out.QG = a->QG;
  out.Qs = ws + L.Qs;
  out.Aqk_b = ws + L.Aqk_b;
  out.Kl = ws + L.Kl;
  out.gamma = reinterpret_cast<float*>(ws + L.gamma);
  int rc = run_intra(s, a, P, out, d, st);
  if (rc) return rc;
  if (ev && cudaEventRecord(ev[1], st) != cudaSuccess) return KDA_ERR_LAUNCH;
  StateMaps m;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!map_tokens(&m.W, out.W, bf, 2, s.K, s.Hv, s.BT, 64, sw) ||
      !map_tokens(&m.Qs, out.Qs, bf, 2, s.K, s.Hv, s.BT, 64, sw) ||
      !map_tokens(&m.Aqk_b, out.Aqk_b, bf, 2, 64, s.Hv, s.BT, 64, sw) ||
      !map_tokens(&m.U, out.U, bf, 2, s.V, s.Hv, s.BT, s.V, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !map_tokens(&m.Kl, out.Kl, bf, 2, s.K, s.Hv, s.BT, 64, sw))
    return KDA_ERR_LAUNCH;
  if (launch_state(P, m, out.gamma, a->initial_state, a->o, a->final_state, d.dev, st) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  if (ev && cudaEventRecord(ev[2], st) != cudaSuccess) return KDA_ERR_LAUNCH;
  return run_exact(a, P, d, true, st);
}

int fused_forward(const Shape& s, const KdaArgs* a, uint8_t* ws, const Layout& L, const DeviceInfo& d,
                  cudaEvent_t const* ev, cudaStream_t st) {
  const Problem P = make_problem(s, a, ws, L);
  IntraMaps im;
  if (!make_intra_maps(s, a, &im)) return KDA_ERR_LAUNCH;
  FusedMaps m;
  m.q = im.q;
  m.k = im.k;
  m.v = im.v;
  m.g = im.g;
  m.v_sw = im.v_sw;
  FusedArgs f{};
  // outputs whose base and strides a TMA store map accepts (16-byte alignment)
  // leave by TMA stores of whole chunks; the others by per-thread stores
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  f.o_tma = aligned16(a->o) && map_tokens(&m.o, a->o, bf, 2, s.V, s.Hv, s.BT, 64, sw);
  f.w_tma = a->W && aligned16(a->W) && map_tokens(&m.W, a->W, bf, 2, s.K, s.Hv, s.BT, 64, sw);
  f.u_tma = a->U && aligned16(a->U) && map_tokens(&m.U, a->U, bf, 2, s.V, s.Hv, s.BT, 64, sw);
  f.q = a->q;
  f.k = a->k;
  f.g = a->g;
  f.beta = a->beta;
  f.h0 = a->initial_state;
  f.o = reinterpret_cast<__nv_bfloat16*>(a->o);
  f.hT = a->final_state;
  f.Aqk = a->Aqk;
  f.Akk_inv = a->Akk_inv;
  f.W = a->W;
  f.U = a->U;
  f.G = a->G;
  f.QG = a->QG;
  f.aqk_v8 = (reinterpret_cast<uintptr_t>(a->Aqk) & 31u) == 0;
  if (launch_fused(P, f, m, d.dev, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (ev && (cudaEventRecord(ev[1], st) != cudaSuccess || cudaEventRecord(ev[2], st) != cudaSuccess))
    return KDA_ERR_LAUNCH;
  return run_exact(a, P, d, true, st);
}

}  // namespace
}  // namespace kda

namespace kda {
namespace {

// ---- intra-card context parallelism (KdaArgs.cp_chunks): the segmented view
// of a fixed-length batch runs as a packed batch of B * nps sequences through
// the public entry point, three times (kda_cp.cu has the scan and the reason).

int cp_check(const KdaArgs* a, const Shape& s) {
  if (a->cp_chunks < 0) return KDA_ERR_INVALID;
  if (a->cu_seqlens || a->K != a->V || a->path == KDA_PATH_TWO_PASS || a->intra_tf32 || a->chunk_indices ||
      a->chunk_offsets)
    return KDA_ERR_UNSUPPORTED;
  (void)s;
  return KDA_OK;
}

// segments per sequence (1: nothing to split)
int cp_segments(const KdaArgs* a, const Shape& s) { return (s.NT + a->cp_chunks - 1) / a->cp_chunks; }

KdaArgs cp_sub_args(const KdaArgs* a, int nps, const int32_t* seg_cu) {
  KdaArgs x = *a;
  x.cu_seqlens = seg_cu;
  x.N = a->B * nps;
  x.T = a->B * a->T;
  x.B = 1;
  x.path = KDA_PATH_FUSED;
  x.cp_chunks = 0;
  x.profile_events = nullptr;
  return x;
}

struct CpLayout {
  size_t sub = 0, seg = 0, hs = 0, A = 0, Bs = 0, vz = 0, oz = 0, total = 0;
  int nps = 1;
};

CpLayout cp_layout(const KdaArgs* a, const Shape& s) {
  CpLayout c;
  c.nps = cp_segments(a, s);
  // any aligned non-null address stands for the segment table here: the
  // size query dereferences no pointer
  const KdaArgs sub = cp_sub_args(a, c.nps, reinterpret_cast<const int32_t*>(uintptr_t(1) << 20));
  c.sub = align_up(kda_workspace_size(&sub));
  size_t p = c.sub;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes);
    return at;
  };
  const size_t nseg = size_t(s.B) * c.nps;
  const size_t smat = nseg * s.Hv * s.K * s.V * 4;
  c.seg = take((nseg + 1) * 4);
  c.hs = take(smat);  // identity start states, then the scanned start states
  c.A = take(smat);   // segment transitions
  c.Bs = take(smat);  // segment end states from zero, then the last pass's (unused) end states
  c.vz = take(size_t(s.BT) * s.Hv * s.V * 2);  // v = 0 for the transition pass
  c.oz = take(size_t(s.BT) * s.Hv * s.V * 2);  // o of the first two passes (discarded)
  c.total = p;
  return c;
}

int cp_forward(const KdaArgs* a, const Shape& s, uint8_t* ws, size_t ws_bytes, cudaStream_t st) {
  const CpLayout c = cp_layout(a, s);
  if (ws_bytes < c.total) return KDA_ERR_WORKSPACE;
  DeviceInfo d;
  int rc = device_info(&d);
  if (rc) return rc;
  const int nseg = s.B * c.nps;
  int32_t* seg = reinterpret_cast<int32_t*>(ws + c.seg);
  float* hs = reinterpret_cast<float*>(ws + c.hs);
  float* Am = reinterpret_cast<float*>(ws + c.A);
  float* Bm = reinterpret_cast<float*>(ws + c.Bs);
  kda_stream_t stream = reinterpret_cast<kda_stream_t>(st);
  if (launch_cp_segments(seg, s.B, s.T, a->cp_chunks * kChunk, c.nps, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  // pass 1: each segment's end state from zero (o discarded)
  KdaArgs p1 = cp_sub_args(a, c.nps, seg);
  p1.initial_state = nullptr;
  p1.o = ws + c.oz;
  p1.final_state = Bm;
  p1.Aqk = p1.Akk_inv = nullptr;
  p1.W = p1.U = nullptr;
  p1.G = nullptr;
  p1.QG = nullptr;
  rc = kda_chunk_fwd(&p1, ws, c.sub, stream);
  if (rc) return rc;
  // pass 2: each segment's transition, its end state from the identity with v = 0
  if (launch_cp_identity(hs, (long long)nseg * s.Hv, s.K, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (cudaMemsetAsync(ws + c.vz, 0, size_t(s.BT) * s.Hv * s.V * 2, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  KdaArgs p2 = p1;
  p2.v = ws + c.vz;
  p2.initial_state = hs;
  p2.final_state = Am;
  rc = kda_chunk_fwd(&p2, ws, c.sub, stream);
  if (rc) return rc;
  // the scan: start states of the segments, final states of the sequences
  if (launch_cp_scan(Am, Bm, a->initial_state, hs, a->final_state, s.B, c.nps, s.Hv, s.K, d.dev, st) !=
      cudaSuccess)
    return KDA_ERR_LAUNCH;
  // pass 3: the outputs, from the scanned start states
  KdaArgs p3 = cp_sub_args(a, c.nps, seg);
  p3.initial_state = hs;
  p3.final_state = Bm;
  return kda_chunk_fwd(&p3, ws, c.sub, stream);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_workspace_size(const KdaArgs* a) {
  Shape s;
  Mode mode;
  if (check_shape(a, &s) != KDA_OK || forward_mode(a, &mode) != KDA_OK) return 0;
  // the larger of the forward's and the intra primitive's needs
  size_t fwd = make_layout(s, a, mode).total;
  const size_t intra = make_layout(s, a, Mode::kIntra).total;
  if (a->cp_chunks != 0) {
    if (cp_check(a, s) != KDA_OK) return 0;
    if (cp_segments(a, s) > 1) fwd = cp_layout(a, s).total;
  }
  return fwd > intra ? fwd : intra;
}

extern "C" int kda_chunk_fwd(const KdaArgs* a, void* workspace, size_t ws_bytes, kda_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!a) return KDA_ERR_INVALID;
  if (a->cp_chunks != 0) {
    Shape s;
    int rc = check_shape(a, &s);
    if (rc) return rc;
    rc = cp_check(a, s);
    if (rc) return rc;
    if (cp_segments(a, s) > 1 && s.BT > 0) {
      if (!workspace) return KDA_ERR_INVALID;
      // the profiling events bracket the whole call (all passes and the scan)
      cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->profile_events);
      if (ev && cudaEventRecord(ev[0], st) != cudaSuccess) return KDA_ERR_LAUNCH;
      rc = cp_forward(a, s, static_cast<uint8_t*>(workspace), ws_bytes, st);
      if (rc == KDA_OK && ev &&
          (cudaEventRecord(ev[1], st) != cudaSuccess || cudaEventRecord(ev[2], st) != cudaSuccess))
        return KDA_ERR_LAUNCH;
      return rc;
    }
    KdaArgs one = *a;  // a single segment: the plain forward
    one.cp_chunks = 0;
    return kda_chunk_fwd(&one, workspace, ws_bytes, stream);
  }
  Mode mode;
  int rc = forward_mode(a, &mode);
  if (rc) return rc;
  Shape s;
  Layout L;
  DeviceInfo d;
  rc = prologue(a, workspace, ws_bytes, st, mode, &s, &L, &d);
  if (rc) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->profile_events);
  if (ev && cudaEventRecord(ev[0], st) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (s.BT == 0 || s.nc_max == 0) return empty_forward(s, a, st);
  return mode == Mode::kFused ? fused_forward(s, a, ws, L, d, ev, st) : two_pass_forward(s, a, ws, L, d, ev, st);
}

extern "C" int kda_fwd_intra(const KdaArgs* a, void* workspace, size_t ws_bytes, kda_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Shape s;
  Layout L;
  DeviceInfo d;
  int rc = prologue(a, workspace, ws_bytes, st, Mode::kIntra, &s, &L, &d);
  if (rc) return rc;
  if (s.BT == 0 || s.nc_max == 0) return KDA_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const Problem P = make_problem(s, a, ws, L);
  IntraOut out{};
  out.Aqk = a->Aqk;
  out.Akk_inv = a->Akk_inv;
  out.W = a->W;
  out.U = a->U;
  out.G = a->G;
  out.QG = a->QG;
  rc = run_intra(s, a, P, out, d, st);
  return rc ? rc : run_exact(a, P, d, false, st);
}

extern "C" int kda_prepare_chunk_indices(const int32_t* cu_seqlens, int32_t N, int32_t T, int32_t chunk,
                                         int32_t* chunk_indices, int32_t* chunk_offsets, int32_t* num_chunks,
                                         int32_t* status, kda_stream_t stream) {
  if (chunk <= 0 || N < 0 || T < 0) return KDA_ERR_INVALID;
  if (!cu_seqlens || !chunk_offsets || !num_chunks || !status || (N > 0 && !chunk_indices))
    return KDA_ERR_INVALID;
  const int rc = check_arch();
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_chunk_index(cu_seqlens, N, T, chunk, chunk_indices, chunk_offsets, num_chunks, status, st) ==
                 cudaSuccess
             ? KDA_OK
             : KDA_ERR_LAUNCH;
}

extern "C" int kda_get_device_status(const void* workspace, kda_stream_t stream, int32_t* status_out) {
  if (!workspace || !status_out) return KDA_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_LAUNCH;
  *status_out = v;
  return KDA_OK;
}

namespace kda {
namespace {

// One warp waits on a barrier that no thread arrives at: the bounded wait of
// every kernel must give up, record the timeout and return.
__global__ void bounded_wait_check_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  wait_bar(&bar, 0, &abort_flag, status);
}

}  // namespace
}  // namespace kda

extern "C" int kda_check_bounded_wait(int32_t* device_status, kda_stream_t stream) {
  if (!device_status) return KDA_ERR_INVALID;
  const int rc = kda::check_arch();
  if (rc) return rc;
  kda::bounded_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(device_status);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported size (chunk must be 64; K, V in {64, 128})";
    case KDA_ERR_MISALIGNED: return "misaligned pointer (16 B for tensors, 256 B for the workspace)";
    case KDA_ERR_ARCH: return "device is not sm_103 (the library is built for sm_103a)";
    case KDA_ERR_LAUNCH: return "CUDA launch or tensor-map encode failed";
    case KDA_ERR_WORKSPACE: return "workspace smaller than kda_workspace_size()";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens must start at 0, be non-decreasing and end at T";
    case KDA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case KDA_ERR_GATE_RANGE:
      return "reserved (chains past the gate range are recomputed by the exact path)";
    case KDA_ERR_BAD_CHUNK_TABLE: return "the supplied chunk_indices / chunk_offsets do not match cu_seqlens";
    default: return "unknown status";
  }
}
