// kda_chunk_fwd for callers that cannot allocate device memory.
//
// Some callers only ever hold the input and output buffers they were handed:
// plug-ins inside a host runtime or inference engine that owns all device
// memory through its own pool (a cudaMalloc there fails once the pool has
// reserved the device, or fragments it), and latency-critical code that must
// not pay for, or risk the failure of, an allocation in the middle of a
// request.  This entry point runs the same kernels as kda_chunk_fwd, but its
// workspace is a fixed array that lives in the library's device image: every
// GPU that loads the library holds kStaticScratchBytes for it until the
// process exits, and nothing is allocated per call.
//
// Host code cannot use the array's name as a device address (on the host it
// is only a stand-in symbol), so the device address is looked up with
// cudaGetSymbolAddress, while that device is current, on the first call made
// with it, and reused afterwards.  The cache is per process and per device
// ordinal: it does not survive a cudaDeviceReset (the library's module, and
// with it the array, is loaded again at a new address), so a process that
// resets a device must not call this entry point on it afterwards.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static_assert(kStaticScratchBytes == KDA_STATIC_SCRATCH_BYTES, "header and library must agree");

static __device__ __align__(256) unsigned char g_kda_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_kda_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return KDA_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no pending error behind for the caller's next CUDA call
      return KDA_ERR_LAUNCH;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

// Compute capability 10.3, as kda_chunk_fwd checks, but before the symbol
// lookup, so that a device without the library's sm_103a image reports
// KDA_ERR_ARCH rather than a failed lookup.
int is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_ARCH;
  }
  return (major == 10 && minor == 3) ? KDA_OK : KDA_ERR_ARCH;
}

}  // namespace

extern "C" int kda_chunk_fwd_static_scratch(const KdaArgs* args, int32_t* device_status, kda_stream_t stream) {
  const size_t need = kda_workspace_size(args);
  // need == 0 means the sizes are invalid: kda_chunk_fwd reports why, before
  // touching the scratch.
  if (need > kStaticScratchBytes) return KDA_ERR_WORKSPACE;
  if (need > 0) {
    int rc = is_sm103();
    if (rc != KDA_OK) return rc;
  }
  void* ws = nullptr;
  int rc = need > 0 ? scratch_address(&ws) : KDA_OK;
  if (rc != KDA_OK) return rc;
  // kda_chunk_fwd zeroes the status word and chunk count at the start of the
  // scratch before its kernels run; nothing else needs to start at zero.  With
  // invalid sizes it returns its error before touching the (null) workspace.
  rc = kda_chunk_fwd(args, ws, kStaticScratchBytes, stream);
  if (rc != KDA_OK) return rc;
  if (device_status &&
      cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  return KDA_OK;
}
