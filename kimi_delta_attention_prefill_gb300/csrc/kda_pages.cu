// kda_pages.cu -- page-table checks of the paged entry points.
//
// The prefix cache of "部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景" (section 3)
// keeps each head's state as one 64 KiB block and shares a cached checkpoint between the
// requests that hit it; such a shared block is read, never written (copy on hit: the
// continuation's state goes to a fresh page).  Before a paged call runs, these two kernels
// verify that contract over the caller's page tables with an owner table in the workspace:
//   claim  every written page is claimed by its writer; a second claim is an error;
//   reads  a read page must be unclaimed or claimed by its own unit's final state (in place).
// Both are grid-stride loops over the table entries (a few thousand to a few million).
#include <cuda_runtime.h>
#include <cstdint>

#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kCheckThreads = 256;

__device__ __forceinline__ void page_fail(int* fail, int* status) {
  atomicExch(fail, 1);
  report_status(status, 7 /* KDA_ERR_DEVICE_CHECK */);
}

__global__ void claim_pages_kernel(const int32_t* __restrict__ out, int64_t n_units, const int32_t* __restrict__ ckpt,
                                   int64_t n_ck, int64_t n_pages, int* __restrict__ owner, int* __restrict__ fail,
                                   int* __restrict__ status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_units + n_ck; i += stride) {
    const int32_t pg = i < n_units ? (out ? out[i] : -1) : ckpt[i - n_units];
    if (pg == -1) continue;
    if (pg < -1 || pg >= n_pages) { page_fail(fail, status); continue; }
    if (atomicCAS(&owner[pg], -1, static_cast<int>(i)) != -1) page_fail(fail, status);
  }
}

__global__ void check_reads_kernel(const int32_t* __restrict__ in, int64_t n_units, int64_t n_pages,
                                   const int* __restrict__ owner, int* __restrict__ fail, int* __restrict__ status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_units; i += stride) {
    const int32_t pg = in[i];
    if (pg == -1) continue;
    if (pg < -1 || pg >= n_pages) { page_fail(fail, status); continue; }
    const int w = owner[pg];
    if (w != -1 && w != static_cast<int>(i)) page_fail(fail, status);
  }
}

unsigned grid_for(int64_t n) {
  const int64_t b = (n + kCheckThreads - 1) / kCheckThreads;
  return static_cast<unsigned>(b < 1 ? 1 : (b > 4096 ? 4096 : b));
}

}  // namespace

cudaError_t launch_page_check(const int32_t* in, const int32_t* out, int64_t n_units, const int32_t* ckpt,
                              int64_t n_ckpt_entries, int64_t n_pages, void* ws, int* status, cudaStream_t stream) {
  int* fail = static_cast<int*>(ws);
  int* owner = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + 256);
  cudaError_t e = cudaMemsetAsync(fail, 0, 256, stream);
  if (e == cudaSuccess && n_pages > 0) e = cudaMemsetAsync(owner, 0xff, 4 * static_cast<size_t>(n_pages), stream);
  if (e != cudaSuccess) return e;
  const int64_t n_w = n_units + (ckpt ? n_ckpt_entries : 0);
  if (n_w > 0) {
    claim_pages_kernel<<<grid_for(n_w), kCheckThreads, 0, stream>>>(out, n_units, ckpt, ckpt ? n_ckpt_entries : 0,
                                                                    n_pages, owner, fail, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (in && n_units > 0) {
    check_reads_kernel<<<grid_for(n_units), kCheckThreads, 0, stream>>>(in, n_units, n_pages, owner, fail, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
