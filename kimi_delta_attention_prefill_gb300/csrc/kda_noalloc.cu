// kda_noalloc.cu -- kda_prefill_noalloc: prefill for callers that may not allocate device
// memory.
//
// Some callers cannot hand the library a workspace.  A plugin loaded into a serving
// framework that owns every byte of device memory (it passes in only the input and
// output tensors, and gives the plugin no allocator), or a latency-critical path where a
// cudaMalloc -- which may synchronise the device -- is not allowed, cannot obtain the
// scratch buffer that the sequence split of kda_prefill needs.  This entry point takes
// that scratch from a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ object of kNoallocScratchBytes (32 MiB): every GPU
// on which the module holding it is loaded keeps it until the process exits.  Host code
// cannot use the array's name as a device address, so each device's address is looked
// up once with cudaGetSymbolAddress (on the first call made while that device is
// current, whatever the problem's size) and cached.  Under the CUDA runtime's default lazy
// module loading that lookup is also what loads the module on the device, so the driver
// reserves the array's memory then: the first call belongs in the caller's set-up.
#include <cuda_runtime.h>
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(KDA_NOALLOC_SCRATCH_BYTES);
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).
kda_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no failed lookup pending in the runtime's error state
      return KDA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                                          const float* beta, const float* S_in, const int32_t* cu_seqlens, int n_seq,
                                          int64_t total_tokens, const int32_t* ckpt_off, const int32_t* ckpt_pos,
                                          int64_t n_ckpt, kda_bf16* o, float* S_out, float* ckpts, int H, int d,
                                          int n_segments, int* dev_status, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_seq < 0 || H < 0 || total_tokens < 0 || n_segments < 0) return KDA_ERR_INVALID_ARG;
  // set-up on the first call on this device, whatever the problem (an empty one included)
  void* scratch = nullptr;
  const kda_status st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  size_t need = 0;
  if (n_seq > 0 && H > 0) {
    need = kda_prefill_workspace_size(n_seq, H, d, total_tokens, n_segments);
    if (need > kNoallocScratchBytes) return KDA_ERR_WORKSPACE;  // larger than the built-in scratch
  }
  if (need == 0) scratch = nullptr;
  return kda_prefill(q, k, v, g, beta, S_in, cu_seqlens, n_seq, total_tokens, ckpt_off, ckpt_pos, n_ckpt, o, S_out,
                     ckpts, H, d, n_segments, scratch, need, dev_status, stream);
}
