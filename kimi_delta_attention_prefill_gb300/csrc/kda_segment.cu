// kda_segment.cu -- the SM-level sequence split: planner and entry-state scan.
//
// "部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景", sections 1.2 and 2: a
// segment's effect on the state is the pair (M, S~) of its cumulative transition
// M = prod_r (I - beta_r k_r k_r^T) Diag(alpha_r) and its zero-start state S~; the exit
// state for entry S_in is S~ + M S_in, and pairs compose associatively, so the entry
// state of every segment follows from a prefix scan over the preceding pairs.
//
// On one GPU the split runs as:
//   plan   (1 thread)   per sequence: segment count (plan_segments), chunk ranges, work
//                        items for the two prefill passes, workspace slots;
//   pass 1 (prefill)     segment 0 in full from S_in (its exit state is exact), and for
//                        each middle segment k its S~_k (zero entry) and M_k (identity
//                        entry, V = 0) as two state-only items;
//   scan   (this file)   entry_1 = exit_0, entry_{k+1} = S~_k + M_k entry_k, column blocks
//                        of 16 in parallel, fp32;
//   pass 3 (prefill)     segments 1.. from their entry states: outputs, checkpoints, S_out.
#include <cuda_runtime.h>
#include <cstdint>

#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanCols = 16;

__global__ void split_plan_kernel(const int32_t* __restrict__ cu, int n_seq, int64_t total_tokens, int H,
                                  int num_sms, int n_segments, int4* __restrict__ items1,
                                  int4* __restrict__ items3, int2* __restrict__ seginfo, int* __restrict__ counts,
                                  int64_t max1, int64_t max3, int64_t max_slots, int* __restrict__ status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int64_t n1 = 0, n3 = 0, slot = 0;
  for (int s = 0; s < n_seq; ++s) {
    const int64_t a = cu[s], b = cu[s + 1];
    const bool ok = a >= 0 && b >= a && b <= total_tokens && (s != 0 || a == 0) &&
                    (s != n_seq - 1 || b == total_tokens);
    if (!ok) {
      report_status(status, 7 /* KDA_ERR_DEVICE_CHECK */);
      seginfo[s] = make_int2(-1, 0);
      continue;
    }
    const int len = static_cast<int>(b - a);
    const int nch = (len + kChunk - 1) / kChunk;
    const int ns = plan_segments(len, H, num_sms, n_segments);
    if (ns <= 1) {
      if (n1 >= max1) { report_status(status, 4); continue; }
      items1[n1++] = make_int4(s, 0, nch, kModeFull);
      seginfo[s] = make_int2(-1, 1);
      continue;
    }
    if (slot + ns > max_slots || n1 + 2 * ns - 3 > max1 || n3 + ns - 1 > max3) {
      report_status(status, 4 /* KDA_ERR_WORKSPACE: bound violated (cannot happen) */);
      seginfo[s] = make_int2(-1, 0);
      continue;
    }
    const int base = static_cast<int>(slot);
    slot += ns;
    const int w0 = n_segments > 0 ? 1 : split_pass1_waves(ns, H, num_sms);
    auto cb = [&](int k) { return segment_boundary(k, ns, nch, w0); };
    items1[n1++] = make_int4(s, 0, cb(1), kModeFirst | (base << 3));
    for (int k = 1; k + 1 < ns; ++k) {
      items1[n1++] = make_int4(s, cb(k), cb(k + 1), kModeZero | ((base + k) << 3));
      items1[n1++] = make_int4(s, cb(k), cb(k + 1), kModeTrans | ((base + k) << 3));
    }
    for (int k = 1; k < ns; ++k) items3[n3++] = make_int4(s, cb(k), cb(k + 1), kModeTail | ((base + k) << 3));
    seginfo[s] = make_int2(base, ns);
  }
  counts[0] = static_cast<int>(n1);
  counts[1] = static_cast<int>(n3);
}

// Slot buffer b (0: exit / S~, 1: M, 2: entry) of (slot, head).
__device__ __forceinline__ float* slot_buf(float* slots, int slot, int H, int h, int b) {
  return slots + ((static_cast<int64_t>(slot) * H + h) * 3 + b) * (kHeadDim * kHeadDim);
}

// One CTA per (sequence, head, 16-column block): the entry states of segments 1..n-1.
// Columns of the state evolve independently under left-multiplication by M.
__global__ void __launch_bounds__(kScanThreads) split_scan_kernel(const int2* __restrict__ seginfo,
                                                                  float* __restrict__ slots, int H) {
  const int s = blockIdx.x, h = blockIdx.y, c_base = blockIdx.z * kScanCols;
  const int2 info = seginfo[s];
  if (info.y < 2) return;
  const int base = info.x, ns = info.y;
  __shared__ float E[kHeadDim][kScanCols];
  const int tid = threadIdx.x, i = tid >> 1, c0 = (tid & 1) * 8;
  {
    const float* x0 = slot_buf(slots, base, H, h, 0) + i * kHeadDim + c_base + c0;
    float* e1 = slot_buf(slots, base + 1, H, h, 2) + i * kHeadDim + c_base + c0;
    const float4 a = *reinterpret_cast<const float4*>(x0), b = *reinterpret_cast<const float4*>(x0 + 4);
    *reinterpret_cast<float4*>(&E[i][c0]) = a;
    *reinterpret_cast<float4*>(&E[i][c0 + 4]) = b;
    *reinterpret_cast<float4*>(e1) = a;
    *reinterpret_cast<float4*>(e1 + 4) = b;
  }
  __syncthreads();
  for (int k = 1; k + 1 < ns; ++k) {
    const float* St = slot_buf(slots, base + k, H, h, 0) + i * kHeadDim + c_base + c0;
    const float* Mrow = slot_buf(slots, base + k, H, h, 1) + i * kHeadDim;
    float acc[8];
    {
      const float4 a = *reinterpret_cast<const float4*>(St), b = *reinterpret_cast<const float4*>(St + 4);
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
#pragma unroll 4
    for (int m4 = 0; m4 < kHeadDim; m4 += 4) {
      const float4 mv = *reinterpret_cast<const float4*>(Mrow + m4);
      const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 e0 = *reinterpret_cast<const float4*>(&E[m4 + u][c0]);
        const float4 e1 = *reinterpret_cast<const float4*>(&E[m4 + u][c0 + 4]);
        acc[0] += mm[u] * e0.x; acc[1] += mm[u] * e0.y; acc[2] += mm[u] * e0.z; acc[3] += mm[u] * e0.w;
        acc[4] += mm[u] * e1.x; acc[5] += mm[u] * e1.y; acc[6] += mm[u] * e1.z; acc[7] += mm[u] * e1.w;
      }
    }
    __syncthreads();  // every thread has read E
    *reinterpret_cast<float4*>(&E[i][c0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(&E[i][c0 + 4]) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    float* en = slot_buf(slots, base + k + 1, H, h, 2) + i * kHeadDim + c_base + c0;
    *reinterpret_cast<float4*>(en) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(en + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
  }
}

// Cross-device KCP combine ("部署 Kimi K3 ..." section 2: after the all-gather, a rank
// folds the preceding ranks' pairs in order): one CTA per (sequence, head, 16-column
// block), E <- S~_r + M_r E for r = 0 .. n_pairs - 1 from E = S_in, fp32.
__global__ void __launch_bounds__(kScanThreads) combine_pairs_kernel(const float* __restrict__ M,
                                                                     const float* __restrict__ St, int n_pairs,
                                                                     const float* __restrict__ S_in,
                                                                     float* __restrict__ entry, int n_seq, int H) {
  const int s = blockIdx.x, h = blockIdx.y, c_base = blockIdx.z * kScanCols;
  const int64_t unit = static_cast<int64_t>(s) * H + h, units = static_cast<int64_t>(n_seq) * H;
  __shared__ float E[kHeadDim][kScanCols];
  const int tid = threadIdx.x, i = tid >> 1, c0 = (tid & 1) * 8;
  {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (S_in) {
      const float* x0 = S_in + unit * kStateFloats + i * kHeadDim + c_base + c0;
      a = *reinterpret_cast<const float4*>(x0);
      b = *reinterpret_cast<const float4*>(x0 + 4);
    }
    *reinterpret_cast<float4*>(&E[i][c0]) = a;
    *reinterpret_cast<float4*>(&E[i][c0 + 4]) = b;
  }
  __syncthreads();
  for (int r = 0; r < n_pairs; ++r) {
    const int64_t base = (static_cast<int64_t>(r) * units + unit) * kStateFloats;
    const float* Sr = St + base + i * kHeadDim + c_base + c0;
    const float* Mrow = M + base + i * kHeadDim;
    float acc[8];
    {
      const float4 a = *reinterpret_cast<const float4*>(Sr), b = *reinterpret_cast<const float4*>(Sr + 4);
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
#pragma unroll 4
    for (int m4 = 0; m4 < kHeadDim; m4 += 4) {
      const float4 mv = *reinterpret_cast<const float4*>(Mrow + m4);
      const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 e0 = *reinterpret_cast<const float4*>(&E[m4 + u][c0]);
        const float4 e1 = *reinterpret_cast<const float4*>(&E[m4 + u][c0 + 4]);
        acc[0] += mm[u] * e0.x; acc[1] += mm[u] * e0.y; acc[2] += mm[u] * e0.z; acc[3] += mm[u] * e0.w;
        acc[4] += mm[u] * e1.x; acc[5] += mm[u] * e1.y; acc[6] += mm[u] * e1.z; acc[7] += mm[u] * e1.w;
      }
    }
    __syncthreads();  // every thread has read E
    *reinterpret_cast<float4*>(&E[i][c0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(&E[i][c0 + 4]) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
  }
  float* dst = entry + unit * kStateFloats + i * kHeadDim + c_base + c0;
  *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(&E[i][c0]);
  *reinterpret_cast<float4*>(dst + 4) = *reinterpret_cast<const float4*>(&E[i][c0 + 4]);
}

}  // namespace

cudaError_t launch_combine_pairs(const float* M, const float* S_tilde, int n_pairs, const float* S_in, float* entry,
                                 int n_seq, int H, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(n_seq), static_cast<unsigned>(H), kHeadDim / kScanCols);
  combine_pairs_kernel<<<grid, kScanThreads, 0, stream>>>(M, S_tilde, n_pairs, S_in, entry, n_seq, H);
  return cudaGetLastError();
}

cudaError_t launch_split_plan(const PrefillArgs& a, const SplitLayout& L, int num_sms) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  split_plan_kernel<<<1, 32, 0, a.stream>>>(
      a.cu_seqlens, a.n_seq, a.total_tokens, a.H, num_sms, a.n_segments,
      reinterpret_cast<int4*>(ws + L.off_items1), reinterpret_cast<int4*>(ws + L.off_items3),
      reinterpret_cast<int2*>(ws + L.off_seginfo), reinterpret_cast<int*>(ws), L.max1, L.max3, L.n_slots, a.status);
  return cudaGetLastError();
}

cudaError_t launch_split_scan(const PrefillArgs& a, const SplitLayout& L) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  dim3 grid(static_cast<unsigned>(a.n_seq), static_cast<unsigned>(a.H), kHeadDim / kScanCols);
  split_scan_kernel<<<grid, kScanThreads, 0, a.stream>>>(reinterpret_cast<const int2*>(ws + L.off_seginfo),
                                                         reinterpret_cast<float*>(ws + L.off_slots), a.H);
  return cudaGetLastError();
}

}  // namespace kda
