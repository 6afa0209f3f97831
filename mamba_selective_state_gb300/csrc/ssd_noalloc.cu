// ssd_noalloc.cu -- ssd_fwd_noalloc: the forward pass with its workspace in a
// device array owned by the library instead of caller memory.
//
// Some callers cannot allocate device memory where they call the layer: a
// plain C host that has no handle on the framework's caching allocator, or
// a latency-critical loop where an allocation (and the synchronisation that
// cudaMalloc implies) is not allowed.  They still pass inputs and outputs;
// the workspace lives in g_noalloc_scratch, a file-scope __device__ array of
// SSD_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
// the process exits.
#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// In host code the array's name is only a host-side stand-in: its device
// address is looked up once per device, with that device current, and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_fwd_noalloc(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
                               const float* A, const void* B, const void* C, const float* D,
                               const float* initial_states, const int32_t* seq_idx, void* y,
                               float* final_states, ssd_stream_t stream) {
  const size_t need = ssd_fwd_workspace_bytes(prob);
  if (need == 0) return SSD_ERR_INVALID_ARGUMENT;
  if (need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const int rc = ssd::scratch_address(&ws);
  if (rc != SSD_OK) return rc;
  // ssd_fwd validates the rest; its first kernel re-zeroes the parts of the
  // workspace that must start at zero (scan flags, tickets, status word).
  return ssd_fwd(prob, x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, y, final_states, ws,
                 (size_t)SSD_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word of the last ssd_fwd_noalloc call sits at the start of the
// library-owned array, whose address the caller never sees: this reads it
// there, exactly as ssd_read_device_status reads a caller workspace.
extern "C" int ssd_fwd_noalloc_read_device_status(ssd_stream_t stream) {
  void* ws = nullptr;
  const int rc = ssd::scratch_address(&ws);
  if (rc != SSD_OK) return rc;
  return ssd_read_device_status(ws, stream);
}
