// kda_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace kda {

constexpr int kHeadDim = 128;
constexpr int kChunk = 64;
constexpr int kMaxDecodeTokens = 4;

// Device-side error report: the first non-zero code wins.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

constexpr int64_t kStateFloats = static_cast<int64_t>(kHeadDim) * kHeadDim;  // one page / one head's state

// Paged state: a pool of pages, each one head's 128 x 128 fp32 state (64 KiB, row = d_k),
// addressed through int32 page tables; -1 = no page (a zero entry state, or no write).
struct PageTables {
  float* pool = nullptr;  // nullptr: contiguous addressing
  int64_t n_pages = 0;
  const int32_t* in = nullptr;    // [units] entry / read page
  const int32_t* out = nullptr;   // [units] final / written page
  const int32_t* ckpt = nullptr;  // [n_ckpt * H] checkpoint pages (prefill)
  const int* fail = nullptr;      // set by the page check: the kernels then do nothing
};

// Workspace of the page check: a failure word, then an owner table of n_pages int32.
__host__ inline size_t page_check_bytes(int64_t n_pages) { return 256 + 4 * static_cast<size_t>(n_pages); }

// Claims every written page for its writer (a page may be written once per call) and
// then checks every read page: it may be written only by its own unit (in place).
// Writers: out[u] is writer u, ckpt[j] writer n_units + j.  On a violation or a page
// outside [-1, n_pages) it sets the failure word and reports KDA_ERR_DEVICE_CHECK.
cudaError_t launch_page_check(const int32_t* in, const int32_t* out, int64_t n_units, const int32_t* ckpt,
                              int64_t n_ckpt_entries, int64_t n_pages, void* ws, int* status, cudaStream_t stream);

constexpr int kMaxConvWidth = 4;

// Decode front end (kda_decode_fused): the step starts from projected inputs.
struct FrontEnd {
  const void* qp = nullptr;  // [B, n, H, d] bf16 projected inputs before the short convolution
  const void* kp = nullptr;
  const void* vp = nullptr;
  const float* conv_w = nullptr;  // [3, H, d, W] depthwise filters of q, k, v (tap j: j steps back)
  float* conv_cache = nullptr;    // [B, H, 3, W - 1, d] the W - 1 inputs before the step, oldest first
  int W = 1;
  int act = 0;                    // 0: none, 1: SiLU after the convolution
  const float* z = nullptr;       // [B, n, H, d] decay-gate pre-activations
  const float* a_log = nullptr;   // [H]
  float g_min = -5.f;
  const float* b = nullptr;       // [B, n, H] beta logits
  const void* gate = nullptr;     // [B, n, H, d] bf16 output-gate logits, or nullptr
  const float* norm_weight = nullptr;
  float eps = 0.f;
};

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, float* S,
                          const int32_t* n_commit, float* o, int B, int n_tok, int H, int* status,
                          cudaStream_t stream, const PageTables& pages = PageTables());
cudaError_t launch_decode_fused(const FrontEnd& fe, float* S, const int32_t* n_commit, float* o, int B, int n_tok,
                                int H, int* status, cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S_in;
  const int32_t* cu_seqlens;
  int n_seq;
  int64_t total_tokens;
  const int32_t* ckpt_off;
  const int32_t* ckpt_pos;
  int64_t n_ckpt;
  void* o;
  // output stage (kda_prefill_gated): gate logits [T, H, d] bf16 or nullptr for plain o
  const void* gate = nullptr;
  const float* norm_weight = nullptr;  // [d] or nullptr for ones
  float eps = 0.f;
  float* S_out;
  float* ckpts;
  PageTables pages;  // paged S_in / S_out / checkpoints when pages.pool is set
  int stall_chunk = -1;  // test hook (kda_debug_stall_next_prefill): a withheld hand-off
  int H;
  int n_segments;  // 0 = planner, k >= 1 forced
  void* workspace;
  size_t workspace_bytes;
  int* status;
  cudaStream_t stream;
};

// ----------------------------------------------------------------- sequence split
// Planner rule ("部署 Kimi K3 ..." section 1.2: split a sequence over the SMs when its
// rank holds few heads).  A function of the sequence's own length, H, the SM count and
// the caller's request only, so a sequence is split the same way packed or alone.
//   n_segments > 0 : min(n_segments, chunks) segments of equal length
//   n_segments = 0 : the count with the least chain time in a wave model (one CTA per SM,
//     S SMs): with n segments pass 1 runs the first segment and two state-only items per
//     middle segment, H (2n - 3) items in w1 = ceil(H (2n - 3) / S) waves, and pass 3 the
//     n - 1 later segments, H (n - 1) items in w3 waves.  The first segment, which needs no
//     state-only items, is made w1 times as long as the others (it runs through all of
//     pass 1's waves, launched first), so a segment is 1 / (n - 1 + w1) of the chain and the
//     time is (w1 + w3) / (n - 1 + w1) of the unsplit chain; n = 1 costs 1 and ties keep the
//     smaller n.  Candidates: n <= S / H + 1, and segments of at least kMinSegChunks chunks.
constexpr int kMinSegChunks = 64;  // segments shorter than 4096 tokens do not pay for the extra passes

// Pass 1's waves for n segments (1 when there are no middle segments).
__host__ __device__ inline int split_pass1_waves(int n, int H, int num_sms) {
  if (n < 3) return 1;
  const int64_t h = H > 0 ? H : 1, S = num_sms > 0 ? num_sms : 1;
  return static_cast<int>((h * (2 * n - 3) + S - 1) / S);
}

__host__ __device__ inline int plan_segments(int len, int H, int num_sms, int n_segments) {
  const int nch = (len + kChunk - 1) / kChunk;
  if (nch <= 1) return 1;
  if (n_segments > 0) return n_segments < nch ? n_segments : nch;
  const int h = H > 0 ? H : 1, S = num_sms > 0 ? num_sms : 1;
  const int nmax = S / h + 1;
  int best = 1;
  int64_t best_w = 1, best_n = 1;  // cost best_w / best_n, compared as cross products
  for (int n = 2; n <= nmax; ++n) {
    const int w1 = split_pass1_waves(n, h, S);
    const int64_t parts = n - 1 + w1;  // the chain in parts of one later segment each
    if (parts * kMinSegChunks > nch) break;
    const int64_t w = w1 + (static_cast<int64_t>(h) * (n - 1) + S - 1) / S;
    if (w * best_n < best_w * parts) { best = n; best_w = w; best_n = parts; }
  }
  return best;
}

// Chunk boundary k (0 <= k <= ns) of a sequence of nch chunks split into ns segments; the
// first segment has weight w0 (split_pass1_waves for the planner's own count, 1 when the
// caller forces the count), the others weight 1.
__host__ __device__ inline int segment_boundary(int k, int ns, int nch, int w0) {
  if (k <= 0) return 0;
  const int64_t parts = ns - 1 + w0;
  return static_cast<int>(((w0 + k - 1) * static_cast<int64_t>(nch)) / parts);
}

// Work-item modes of the prefill kernel.
enum : int {
  kModeFull = 0,   // whole sequence from S_in: outputs, checkpoints, S_out
  kModeFirst = 1,  // first segment from S_in: outputs, checkpoints, exit state -> slot A
  kModeZero = 2,   // middle segment from a zero state, no outputs: S~ -> slot A
  kModeTrans = 3,  // middle segment from the identity with V = 0: M -> slot B
  kModeTail = 4    // segment 1.. from the entry state in slot C: outputs, checkpoints, S_out if last
};

// Workspace of the split path (all offsets 256-byte aligned):
//   [0, 256)       int counts[2]  (pass-1 items, pass-3 items)
//   items1[max1]   int4 {seq, chunk begin, chunk end, mode | slot << 3}
//   items3[max3]   int4
//   seginfo[n_seq] int2 {first slot, segment count}
//   slots          [n_slots][H][3][128][128] fp32 (A: exit or S~, B: M, C: entry)
struct SplitLayout {
  int64_t extra = 0;  // bound on the total number of extra segments (0: no split)
  int64_t max1 = 0, max3 = 0, n_slots = 0;
  size_t off_items1 = 0, off_items3 = 0, off_seginfo = 0, off_slots = 0, bytes = 0;
};

__host__ inline SplitLayout split_layout(int n_seq, int H, int64_t total_tokens, int n_segments, int num_sms) {
  SplitLayout L;
  int64_t extra = 0;
  if (n_segments > 1) {
    const int64_t a = static_cast<int64_t>(n_seq) * (n_segments - 1);
    const int64_t b = total_tokens / kChunk + n_seq;
    extra = a < b ? a : b;
  } else if (n_segments == 0) {
    // the planner's count only grows with the length: a sequence of all the tokens bounds it
    const int most = plan_segments(total_tokens < (int64_t{1} << 30) ? static_cast<int>(total_tokens) : (1 << 30), H,
                                   num_sms, 0);
    if (most >= 2) {
      const int64_t a = static_cast<int64_t>(n_seq) * (most - 1);
      const int64_t b = total_tokens / (static_cast<int64_t>(kChunk) * kMinSegChunks);
      extra = a < b ? a : b;
    }
  }
  if (extra <= 0) return L;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  L.extra = extra;
  L.max1 = n_seq + 2 * extra;
  L.max3 = extra;
  L.n_slots = (2 * extra < n_seq + extra) ? 2 * extra : n_seq + extra;
  L.off_items1 = 256;
  L.off_items3 = up(L.off_items1 + 16 * static_cast<size_t>(L.max1));
  L.off_seginfo = up(L.off_items3 + 16 * static_cast<size_t>(L.max3));
  L.off_slots = up(L.off_seginfo + 8 * static_cast<size_t>(n_seq));
  L.bytes = L.off_slots + static_cast<size_t>(L.n_slots) * H * 3 * kHeadDim * kHeadDim * sizeof(float);
  return L;
}

// Workspace bytes for the segment split; 0 when it cannot be taken.
size_t prefill_workspace_bytes(int n_seq, int H, int64_t total_tokens, int n_segments, int num_sms);
cudaError_t launch_prefill(const PrefillArgs& a, int num_sms);

// Pair mode of the prefill kernel: per (sequence, head) the zero-entry state S~ and the
// transition M of the sequence's rows, into [n_seq][H][128][128] each.
cudaError_t launch_prefill_pairs(const PrefillArgs& a, float* M, float* S_tilde, int num_sms);
// entry = fold over r < n_pairs of E <- S~_r + M_r E, from E = S_in (zeros when null).
cudaError_t launch_combine_pairs(const float* M, const float* S_tilde, int n_pairs, const float* S_in, float* entry,
                                 int n_seq, int H, cudaStream_t stream);

// The split path's helper kernels (kda_segment.cu).
cudaError_t launch_split_plan(const PrefillArgs& a, const SplitLayout& L, int num_sms);
cudaError_t launch_split_scan(const PrefillArgs& a, const SplitLayout& L);

}  // namespace kda
