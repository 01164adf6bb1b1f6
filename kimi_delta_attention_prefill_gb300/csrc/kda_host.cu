// kda_host.cu -- kda_prefill_host: prefill from host buffers with the transfers overlapped.
//
// A prefill whose inputs start in host memory spends most of its time on the host link
// (about 210 GB/s each way on a GB300 against ~1.4 TB/s of kernel traffic).  This executor
// cuts the packed token stream into blocks and pipelines them over three streams:
//
//   h2d stream      block j's rows of q, k, v, g, beta (one contiguous copy per tensor)
//   caller's stream block j's prefill, once its rows have landed
//   d2h stream      block j's rows of o, once its prefill is done; the final states last
//
// so block j + 1 uploads while block j computes and block j - 1 downloads.  Block borders
// sit on the chunk grid of the sequence they cut (a multiple of 64 tokens from its start),
// and each block runs as an ordinary packed prefill whose sequences start from the running
// states, kept in one device array [n_seq, H, d, d] and updated in place: a sequence cut
// into blocks goes through exactly the chunks, and the fp32 states, of one call.  The
// per-block cu_seqlens are built on the device from one copy of the caller's offsets.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kMaxHostBlocks = 64;
constexpr int64_t kTailTokens = 256;  // size of the last block when the final stretch allows

struct HostBlock {
  int64_t a, e;  // token rows [a, e)
  int s0, s1;    // sequences s0 .. s1 - 1 (contiguous)
};

struct BlockTable {
  HostBlock blk[kMaxHostBlocks];
  int64_t cu_off[kMaxHostBlocks];  // start of block j's cu array in the device buffer
  int n;
};

// Block j's cu array: cu_j[i] = clamp(cu[s0 + i], a, e) - a, i = 0 .. s1 - s0.
__global__ void block_cu_kernel(const int32_t* __restrict__ cu, const BlockTable t, int32_t* __restrict__ out) {
  const HostBlock b = t.blk[blockIdx.x];
  int32_t* dst = out + t.cu_off[blockIdx.x];
  for (int i = threadIdx.x; i <= b.s1 - b.s0; i += blockDim.x) {
    const int64_t c = cu[b.s0 + i];
    dst[i] = static_cast<int32_t>((c < b.a ? b.a : (c > b.e ? b.e : c)) - b.a);
  }
}

// Block borders: about `target` tokens each, the last one about kTailTokens; a border
// that falls inside a sequence moves down to that sequence's chunk grid (a multiple of 64
// tokens from its start), or up when that would leave the block empty.
bool plan_borders(const int32_t* cu, int n_seq, int64_t T, int64_t target, std::vector<int64_t>& border) {
  border.assign(1, 0);
  int k = 0;
  for (int64_t a = 0; a < T;) {
    // the last block's compute and download are the part no upload overlaps: a final stretch
    // longer than 2 kTailTokens ends with a block of about kTailTokens
    const int64_t left = T - a;
    int64_t e = (left <= target && left > 2 * kTailTokens) ? T - kTailTokens : std::min(a + target, T);
    while (k < n_seq && cu[k + 1] <= e) ++k;  // first sequence ending after e: the one e may cut
    if (e < T && k < n_seq && cu[k] < e) {
      const int64_t base = cu[k];
      int64_t cut = base + (e - base) / kChunk * kChunk;
      if (cut <= a) cut = std::min<int64_t>(base + (e - base + kChunk - 1) / kChunk * kChunk, cu[k + 1]);
      e = cut;
    }
    border.push_back(e);
    if (static_cast<int>(border.size()) > kMaxHostBlocks + 1) return false;
    a = e;
  }
  if (T == 0) border.push_back(0);
  return true;
}

// Block j = rows [border[j], border[j + 1]) with the sequences whose rows it holds, plus the
// empty sequences positioned in it (those at T in the last block): a contiguous range.
bool plan_blocks(const int32_t* cu, int n_seq, int64_t T, int64_t target, std::vector<HostBlock>& out) {
  std::vector<int64_t> border;
  if (!plan_borders(cu, n_seq, T, target, border)) return false;
  const int n = static_cast<int>(border.size()) - 1;
  out.resize(n);
  int s0 = 0;
  for (int j = 0; j < n; ++j) {
    const int64_t a = border[j], e = border[j + 1];
    const bool last = j + 1 == n;
    while (s0 < n_seq && cu[s0 + 1] <= a && !(cu[s0] == cu[s0 + 1] && cu[s0] == a)) ++s0;
    int s1 = s0;
    while (s1 < n_seq && (cu[s1] < e || (last && cu[s1] <= T))) ++s1;
    out[j] = HostBlock{a, e, s0, s1};
  }
  return true;
}

// Streams and events of the executor, per device, created by the first call on that device
// and kept for the life of the process (a call used to create and destroy about 2 + 2 x
// blocks of them).  A call holds the device's lock while it enqueues: an event is recorded
// again only by a later call, after every wait on its previous record has been enqueued
// (cudaStreamWaitEvent waits for the record current when it is called), so calls may
// overlap on the GPU.  Two calls' transfers share the two streams and run in call order.
constexpr int kMaxExecDevices = 64;
struct ExecCache {
  std::mutex mu;
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, done = nullptr, fail_up = nullptr, fail_down = nullptr;
  cudaEvent_t landed[kMaxHostBlocks] = {}, computed[kMaxHostBlocks] = {};

  cudaError_t init() {  // creates what is still missing (a failed earlier attempt keeps its part)
    if (ready) return cudaSuccess;
    cudaError_t r = cudaSuccess;
    for (cudaStream_t* st : {&up, &down})
      if (r == cudaSuccess && !*st) r = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
    auto ev = [&](cudaEvent_t* e) {
      if (r == cudaSuccess && !*e) r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    };
    for (cudaEvent_t* e : {&start, &done, &fail_up, &fail_down}) ev(e);
    for (int j = 0; j < kMaxHostBlocks; ++j) { ev(&landed[j]); ev(&computed[j]); }
    if (r == cudaSuccess) ready = true;
    return r;
  }
};
ExecCache g_exec[kMaxExecDevices];

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct HostLayout {
  size_t off_cu = 0, off_bcu = 0, off_q = 0, off_k = 0, off_v = 0, off_g = 0, off_beta = 0, off_o = 0, off_S = 0,
         off_split = 0, bytes = 0;
};

HostLayout host_layout(int n_seq, int H, int64_t T, size_t split_bytes) {
  HostLayout L;
  const size_t row = static_cast<size_t>(T) * H * kHeadDim;
  L.off_cu = 0;
  L.off_bcu = up256(L.off_cu + 4 * static_cast<size_t>(n_seq + 1));
  L.off_q = up256(L.off_bcu + 4 * static_cast<size_t>(n_seq + 2 * kMaxHostBlocks));
  L.off_k = up256(L.off_q + 2 * row);
  L.off_v = up256(L.off_k + 2 * row);
  L.off_g = up256(L.off_v + 2 * row);
  L.off_beta = up256(L.off_g + 4 * row);
  L.off_o = up256(L.off_beta + 4 * static_cast<size_t>(T) * H);
  L.off_S = up256(L.off_o + 2 * row);
  L.off_split = up256(L.off_S + 4 * static_cast<size_t>(n_seq) * H * kHeadDim * kHeadDim);
  L.bytes = L.off_split + split_bytes;
  return L;
}

int64_t default_block(int64_t T) {
  int64_t b = (T / 8 + kChunk - 1) / kChunk * kChunk;
  return std::max<int64_t>(b, 1024);
}

// The split path's workspace bound over the blocks: the planner sees a block as a packed
// prefill of at most n_seq sequences and at most `block` + 64 n_seq tokens.
size_t split_bound(int n_seq, int H, int64_t T, int64_t block, int sms) {
  const int64_t tok = std::min<int64_t>(T, block + static_cast<int64_t>(kChunk) * n_seq);
  return prefill_workspace_bytes(n_seq, H, tok, 0, sms);
}

}  // namespace

}  // namespace kda

extern "C" {

int kda_prefill_host_blocks(const int32_t* cu_seqlens, int n_seq, int64_t total_tokens, int64_t block_tokens,
                            int64_t* borders, int max_borders) {
  if (!cu_seqlens || n_seq < 0 || total_tokens < 0 || block_tokens < 0 || (block_tokens % kda::kChunk) != 0)
    return -1;
  if (n_seq == 0) return 0;
  if (cu_seqlens[0] != 0 || cu_seqlens[n_seq] != total_tokens) return -1;
  for (int s = 0; s < n_seq; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  std::vector<int64_t> border;
  if (!kda::plan_borders(cu_seqlens, n_seq, total_tokens,
                         block_tokens > 0 ? block_tokens : kda::default_block(total_tokens), border))
    return -1;
  const int n = static_cast<int>(border.size()) - 1;
  for (int i = 0; i < static_cast<int>(border.size()) && i < max_borders; ++i) borders[i] = border[i];
  return n;
}

size_t kda_prefill_host_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int64_t block_tokens) {
  if (d != KDA_HEAD_DIM || n_seq < 0 || H <= 0 || total_tokens < 0 || block_tokens < 0) return 0;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  const int64_t blk = block_tokens > 0 ? block_tokens : kda::default_block(total_tokens);
  return kda::host_layout(n_seq, H, total_tokens, kda::split_bound(n_seq, H, total_tokens, blk, sms)).bytes;
}

kda_status kda_prefill_host(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                            const float* beta, const float* S_in, const int32_t* cu_seqlens, int n_seq,
                            int64_t total_tokens, kda_bf16* o, float* S_out, int H, int d, int64_t block_tokens,
                            void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  using namespace kda;
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_seq < 0 || H < 0 || total_tokens < 0 || block_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0x7fffffffLL || static_cast<int64_t>(n_seq) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (n_seq == 0 || H == 0) return KDA_OK;
  if (!cu_seqlens || !S_out || (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)))
    return KDA_ERR_INVALID_ARG;
  if (block_tokens > 0 && block_tokens % kChunk != 0) return KDA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return KDA_ERR_ALIGNMENT;
  // the host offsets are read here to plan the blocks: they must describe a valid packing
  if (cu_seqlens[0] != 0 || cu_seqlens[n_seq] != total_tokens) return KDA_ERR_INVALID_ARG;
  for (int s = 0; s < n_seq; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return KDA_ERR_INVALID_ARG;
  const int64_t T = total_tokens;
  const int64_t blk = block_tokens > 0 ? block_tokens : default_block(T);
  std::vector<HostBlock> blocks;
  if (!plan_blocks(cu_seqlens, n_seq, T, blk, blocks)) return KDA_ERR_UNSUPPORTED;  // more than 64 blocks
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  const size_t split = split_bound(n_seq, H, T, blk, sms);
  const HostLayout L = host_layout(n_seq, H, T, split);
  if (!workspace || workspace_bytes < L.bytes) return KDA_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* d_cu = reinterpret_cast<int32_t*>(ws + L.off_cu);
  int32_t* d_bcu = reinterpret_cast<int32_t*>(ws + L.off_bcu);
  kda_bf16* d_q = reinterpret_cast<kda_bf16*>(ws + L.off_q);
  kda_bf16* d_k = reinterpret_cast<kda_bf16*>(ws + L.off_k);
  kda_bf16* d_v = reinterpret_cast<kda_bf16*>(ws + L.off_v);
  float* d_g = reinterpret_cast<float*>(ws + L.off_g);
  float* d_beta = reinterpret_cast<float*>(ws + L.off_beta);
  kda_bf16* d_o = reinterpret_cast<kda_bf16*>(ws + L.off_o);
  float* d_S = reinterpret_cast<float*>(ws + L.off_S);
  void* d_split = split > 0 ? ws + L.off_split : nullptr;

  BlockTable tab;
  tab.n = static_cast<int>(blocks.size());
  int64_t off = 0;
  for (int j = 0; j < tab.n; ++j) {
    tab.blk[j] = blocks[j];
    tab.cu_off[j] = off;
    off += blocks[j].s1 - blocks[j].s0 + 1;
  }
  if (off > n_seq + 2 * kMaxHostBlocks) return KDA_ERR_UNSUPPORTED;

  if (dev < 0 || dev >= kMaxExecDevices) return KDA_ERR_UNSUPPORTED;
  ExecCache& ex = g_exec[dev];
  std::lock_guard<std::mutex> lock(ex.mu);
  if (ex.init() != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  cudaStream_t up = ex.up, down = ex.down;
  cudaEvent_t start = ex.start, done = ex.done;
  const cudaEvent_t* landed = ex.landed;
  const cudaEvent_t* computed = ex.computed;

  // On a failure after the first enqueue, the work already queued on the two internal
  // streams may still run: the caller's stream is made to wait for it before returning, so
  // that synchronising `stream` still means no transfer touches the caller's buffers.
  auto fail = [&](kda_status code) {
    if (cudaEventRecord(ex.fail_up, up) == cudaSuccess) cudaStreamWaitEvent(stream, ex.fail_up, 0);
    if (cudaEventRecord(ex.fail_down, down) == cudaSuccess) cudaStreamWaitEvent(stream, ex.fail_down, 0);
    return code;
  };
  const size_t HD = static_cast<size_t>(H) * kHeadDim;
  const size_t state_bytes = static_cast<size_t>(n_seq) * HD * kHeadDim * sizeof(float);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // the workspace may still be in use by the caller's earlier work
  if (!ok(cudaEventRecord(start, stream)) || !ok(cudaStreamWaitEvent(up, start, 0)) ||
      !ok(cudaStreamWaitEvent(down, start, 0)))
    return fail(KDA_ERR_CUDA);
  if (!ok(cudaMemcpyAsync(d_cu, cu_seqlens, 4 * static_cast<size_t>(n_seq + 1), cudaMemcpyHostToDevice, up)))
    return fail(KDA_ERR_CUDA);
  block_cu_kernel<<<tab.n, 128, 0, up>>>(d_cu, tab, d_bcu);
  if (!ok(cudaGetLastError())) return fail(KDA_ERR_CUDA);
  if (!ok(S_in ? cudaMemcpyAsync(d_S, S_in, state_bytes, cudaMemcpyHostToDevice, up)
               : cudaMemsetAsync(d_S, 0, state_bytes, up)))
    return fail(KDA_ERR_CUDA);
  for (int j = 0; j < tab.n; ++j) {
    const HostBlock& b = tab.blk[j];
    const size_t r0 = static_cast<size_t>(b.a), nr = static_cast<size_t>(b.e - b.a);
    if (nr > 0) {
      const size_t e2 = r0 * HD, n2 = nr * HD;
      if (!ok(cudaMemcpyAsync(d_q + e2, q + e2, 2 * n2, cudaMemcpyHostToDevice, up)) ||
          !ok(cudaMemcpyAsync(d_k + e2, k + e2, 2 * n2, cudaMemcpyHostToDevice, up)) ||
          !ok(cudaMemcpyAsync(d_v + e2, v + e2, 2 * n2, cudaMemcpyHostToDevice, up)) ||
          !ok(cudaMemcpyAsync(d_g + e2, g + e2, 4 * n2, cudaMemcpyHostToDevice, up)) ||
          !ok(cudaMemcpyAsync(d_beta + r0 * H, beta + r0 * H, 4 * nr * H, cudaMemcpyHostToDevice, up)))
        return fail(KDA_ERR_CUDA);
    }
    if (!ok(cudaEventRecord(landed[j], up)) || !ok(cudaStreamWaitEvent(stream, landed[j], 0))) return fail(KDA_ERR_CUDA);
    // block j: its sequences start from (and end in) the running states, in place
    float* Sj = d_S + static_cast<size_t>(b.s0) * HD * kHeadDim;
    const size_t e2 = r0 * HD;
    const kda_status st =
        kda_prefill(d_q + e2, d_k + e2, d_v + e2, d_g + e2, d_beta + r0 * H, Sj, d_bcu + tab.cu_off[j],
                    b.s1 - b.s0, b.e - b.a, nullptr, nullptr, 0, d_o + e2, Sj, nullptr, H, d, 0, d_split, split,
                    dev_status, stream);
    if (st != KDA_OK) return fail(st);
    if (!ok(cudaEventRecord(computed[j], stream)) || !ok(cudaStreamWaitEvent(down, computed[j], 0)))
      return fail(KDA_ERR_CUDA);
    if (nr > 0 && !ok(cudaMemcpyAsync(o + e2, d_o + e2, 2 * nr * HD, cudaMemcpyDeviceToHost, down)))
      return fail(KDA_ERR_CUDA);
  }
  if (!ok(cudaMemcpyAsync(S_out, d_S, state_bytes, cudaMemcpyDeviceToHost, down)) ||
      !ok(cudaEventRecord(done, down)) || !ok(cudaStreamWaitEvent(stream, done, 0)))
    return fail(KDA_ERR_CUDA);
  return KDA_OK;
}

}  // extern "C"
