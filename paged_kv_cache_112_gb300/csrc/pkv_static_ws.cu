// Decode attention that needs no caller-side scratch buffer and allocates
// nothing.
//
// Who needs this: code that must not allocate device memory at the point it
// runs decode.  Examples are plugins and custom operators whose host
// framework owns every byte of device memory and forbids cudaMalloc during
// execution, serving loops that cannot afford the device-wide synchronisation
// a cudaMalloc/cudaFree can cause, and plain C callers that have no allocator
// to hand a workspace from.  They pass only inputs and outputs; the split-K
// partial results live in a fixed array compiled into this library.
//
// The array is a file-scope __device__ variable of PKV_STATIC_WORKSPACE_BYTES
// bytes.  Every GPU on which the library's module is loaded holds that much
// memory until the process exits.  Host code cannot use the array's name as a
// device address (on the host it names a stand-in object), so each call made
// outside stream capture, with its device current, asks the runtime for the
// real device address with cudaGetSymbolAddress and keeps it for that device.
// A call inside stream capture uses the kept address, so the first call on a
// device must come before any stream capture (a captured first call returns
// PKV_ERR_CUDA).  cudaDeviceReset unloads the module; the next uncaptured
// call looks the address up again.
//
// All calls share the one array, and it keeps whatever the last call left in
// it.  Nothing in it has to start at zero: every partial result the reduce
// kernel reads is written earlier in the same call.  Two calls whose kernels
// overlap on the GPU (different streams, or different host threads on the
// same device) race on the array; callers must order such calls.
//
// The paged-attention pages have no counterpart of this entry point; it is a
// deployment convenience on top of pkv_decode_attention, which it calls with
// the array as the workspace.
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_pkv_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 256;
void* g_workspace_addr[kMaxDevices] = {};
std::mutex g_workspace_mutex;

// Device address of the array on the current device.  The address is looked
// up again on every call made outside stream capture, so a module reloaded
// after cudaDeviceReset is picked up; during capture (where the lookup is not
// wanted) the address from the device's last uncaptured call is used, and a
// device that has had no uncaptured call yet is refused.
pkv_status static_workspace_address(cudaStream_t stream, void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_workspace_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_static_workspace) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    g_workspace_addr[dev] = p;
  } else if (!g_workspace_addr[dev]) {
    return PKV_ERR_CUDA;
  }
  *addr = g_workspace_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_static_workspace(
    void* out, const void* q, const void* k_pool, const void* v_pool, int64_t block_stride, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, float scale, int partition_size, int max_context_len,
    pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status, void* stream) {
  const size_t need =
      pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, partition_size);
  if (need > static_cast<size_t>(PKV_STATIC_WORKSPACE_BYTES)) return PKV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    const pkv_status st = static_workspace_address(static_cast<cudaStream_t>(stream), &ws);
    if (st != PKV_OK) return st;
  }
  return pkv_decode_attention(out, q, k_pool, v_pool, block_stride, block_tables, max_blocks_per_seq, context_lens,
                              num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                              max_context_len, ws, need > 0 ? static_cast<size_t>(PKV_STATIC_WORKSPACE_BYTES) : 0,
                              kv_dtype, out_dtype, dev_status, stream);
}
