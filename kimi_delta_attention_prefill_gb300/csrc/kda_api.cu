// kda_api.cu -- the C ABI (include/kda.h): host-side validation and launch.
//
// Nothing here allocates device memory or keeps per-call state; the only cached
// values are per-device properties (compute capability, SM count).
#include <cuda_runtime.h>
#include <cmath>
#include <atomic>
#include <cstdint>

#include "kda.h"
#include "kda_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_cc[kMaxDevices];   // 0 = unknown, else major*10+minor
std::atomic<int> g_dev_sms[kMaxDevices];

// Returns KDA_OK when the current device is an sm_103 part; fills its SM count.
kda_status current_device(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_CUDA;
  int cc = dev < kMaxDevices ? g_dev_cc[dev].load(std::memory_order_relaxed) : 0;
  int n = dev < kMaxDevices ? g_dev_sms[dev].load(std::memory_order_relaxed) : 0;
  if (cc == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KDA_ERR_CUDA;
    cc = major * 10 + minor;
    if (dev < kMaxDevices) {
      g_dev_sms[dev].store(n, std::memory_order_relaxed);
      g_dev_cc[dev].store(cc, std::memory_order_relaxed);
    }
  }
  if (sms) *sms = n;
  return cc == 103 ? KDA_OK : KDA_ERR_UNSUPPORTED;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// kda_debug_stall_next_prefill: consumed by the next prefill launch
std::atomic<int> g_stall_chunk{-1};

}  // namespace

extern "C" {

const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_ALIGNMENT: return "KDA_ERR_ALIGNMENT";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
    default: return "KDA_ERR_UNKNOWN";
  }
}

int kda_version(void) { return 100; }

kda_status kda_decode(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g, const float* beta,
                      float* S_state, const int32_t* n_commit, float* o, int B, int n_tok, int H, int d,
                      int* dev_status, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_tok < 1 || n_tok > KDA_MAX_DECODE_TOKENS) return KDA_ERR_UNSUPPORTED;
  if (B < 0 || H < 0) return KDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta || !S_state || !o) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(S_state, 16) ||
      !aligned(o, 16) || !aligned(beta, 4) || !aligned(n_commit, 4) || !aligned(dev_status, 4))
    return KDA_ERR_ALIGNMENT;
  kda_status st = current_device(nullptr);
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_decode(q, k, v, g, beta, S_state, n_commit, o, B, n_tok, H, dev_status, stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_prefill_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int n_segments) {
  if (d != KDA_HEAD_DIM || n_seq < 0 || H <= 0 || total_tokens < 0 || n_segments < 0) return 0;
  int sms = 0;
  if (current_device(&sms) != KDA_OK) sms = 152;
  return kda::prefill_workspace_bytes(n_seq, H, total_tokens, n_segments, sms);
}

}  // extern "C"

namespace {
size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Host checks shared by the paged entry points.
kda_status check_pool(const float* pool, int64_t n_pages) {
  if (n_pages < 0 || n_pages > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (n_pages > 0 && !pool) return KDA_ERR_INVALID_ARG;
  return aligned(pool, 16) ? KDA_OK : KDA_ERR_ALIGNMENT;
}

// `pages` is nullptr for contiguous states; otherwise S_in / S_out / ckpts are unused and
// the page check runs in the workspace after the split path's part.
kda_status prefill_impl(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g, const float* beta,
                        const kda_bf16* gate, const float* norm_weight, float eps, const float* S_in,
                        const int32_t* cu_seqlens, int n_seq, int64_t total_tokens, const int32_t* ckpt_off,
                        const int32_t* ckpt_pos, int64_t n_ckpt, kda_bf16* o, float* S_out, float* ckpts, int H,
                        int d, int n_segments, void* workspace, size_t workspace_bytes, int* dev_status,
                        cudaStream_t stream, const kda::PageTables* pages = nullptr) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_seq < 0 || H < 0 || total_tokens < 0 || n_ckpt < 0 || n_segments < 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0x7fffffffLL || static_cast<int64_t>(n_seq) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (n_seq == 0 || H == 0) return KDA_OK;
  if (H > 65535) return KDA_ERR_UNSUPPORTED;  // heads index the grid's y dimension
  if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
  if (ckpt_off == nullptr && n_ckpt != 0) return KDA_ERR_INVALID_ARG;
  if (ckpt_off != nullptr && n_ckpt > 0 && (!ckpt_pos || !(pages ? pages->ckpt != nullptr : ckpts != nullptr)))
    return KDA_ERR_INVALID_ARG;
  if (pages && (static_cast<int64_t>(n_seq) + n_ckpt) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(o, 16) ||
      !aligned(S_in, 16) || !aligned(S_out, 16) || !aligned(ckpts, 16) || !aligned(beta, 4) ||
      !aligned(cu_seqlens, 4) || !aligned(ckpt_off, 4) || !aligned(ckpt_pos, 4) || !aligned(dev_status, 4) ||
      !aligned(workspace, 256))
    return KDA_ERR_ALIGNMENT;
  // the page check's part of the workspace does not depend on the device
  if (pages && (workspace == nullptr || workspace_bytes < kda::page_check_bytes(pages->n_pages)))
    return KDA_ERR_WORKSPACE;
  int sms = 0;
  kda_status st = current_device(&sms);
  if (st != KDA_OK) return st;
  const size_t split = kda::prefill_workspace_bytes(n_seq, H, total_tokens, n_segments, sms);
  const size_t need = pages ? up256(split) + kda::page_check_bytes(pages->n_pages) : split;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  kda::PrefillArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S_in = S_in;
  a.cu_seqlens = cu_seqlens; a.n_seq = n_seq; a.total_tokens = total_tokens;
  a.ckpt_off = (ckpt_off && n_ckpt > 0) ? ckpt_off : nullptr;
  a.ckpt_pos = ckpt_pos; a.n_ckpt = n_ckpt;
  a.o = o; a.S_out = S_out; a.ckpts = ckpts; a.H = H; a.n_segments = n_segments;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes; a.status = dev_status; a.stream = stream;
  a.gate = gate; a.norm_weight = norm_weight; a.eps = eps;
  if (g_stall_chunk.load(std::memory_order_relaxed) >= 0) a.stall_chunk = g_stall_chunk.exchange(-1);
  if (pages) {
    void* pws = static_cast<uint8_t*>(workspace) + up256(split);
    a.pages = *pages;
    a.pages.ckpt = a.ckpt_off ? pages->ckpt : nullptr;
    a.pages.fail = static_cast<const int*>(pws);
    a.S_in = nullptr; a.S_out = nullptr; a.ckpts = nullptr;
    cudaError_t e = kda::launch_page_check(pages->in, pages->out, static_cast<int64_t>(n_seq) * H, a.pages.ckpt,
                                           n_ckpt * H, pages->n_pages, pws, dev_status, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
  }
  cudaError_t e = kda::launch_prefill(a, sms);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

extern "C" {

kda_status kda_prefill(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g, const float* beta,
                       const float* S_in, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                       const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt, kda_bf16* o,
                       float* S_out, float* ckpts, int H, int d, int n_segments, void* workspace,
                       size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  return prefill_impl(q, k, v, g, beta, nullptr, nullptr, 0.f, S_in, cu_seqlens, n_seq, total_tokens, ckpt_off,
                      ckpt_pos, n_ckpt, o, S_out, ckpts, H, d, n_segments, workspace, workspace_bytes, dev_status,
                      stream);
}

kda_status kda_prefill_gated(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const kda_bf16* gate, const float* norm_weight, float eps,
                             const float* S_in, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                             const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt, kda_bf16* y,
                             float* S_out, float* ckpts, int H, int d, int n_segments, void* workspace,
                             size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  if (!(eps >= 0.f) || !std::isfinite(eps)) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && n_seq > 0 && H > 0 && !gate) return KDA_ERR_INVALID_ARG;
  if (!aligned(gate, 16) || !aligned(norm_weight, 16)) return KDA_ERR_ALIGNMENT;
  return prefill_impl(q, k, v, g, beta, gate, norm_weight, eps, S_in, cu_seqlens, n_seq, total_tokens, ckpt_off,
                      ckpt_pos, n_ckpt, y, S_out, ckpts, H, d, n_segments, workspace, workspace_bytes, dev_status,
                      stream);
}

void kda_debug_stall_next_prefill(int chunk) { g_stall_chunk.store(chunk < 0 ? -1 : chunk); }

size_t kda_prefill_paged_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int n_segments,
                                        int64_t n_pages) {
  if (d != KDA_HEAD_DIM || n_seq < 0 || H <= 0 || total_tokens < 0 || n_segments < 0 || n_pages < 0) return 0;
  int sms = 0;
  if (current_device(&sms) != KDA_OK) sms = 152;
  return up256(kda::prefill_workspace_bytes(n_seq, H, total_tokens, n_segments, sms)) + kda::page_check_bytes(n_pages);
}

kda_status kda_prefill_paged(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const kda_bf16* gate, const float* norm_weight, float eps,
                             float* state_pool, int64_t n_pages, const int32_t* s_in_page,
                             const int32_t* s_out_page, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                             const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt,
                             const int32_t* ckpt_page, kda_bf16* o, int H, int d, int n_segments, void* workspace,
                             size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  kda_status st = check_pool(state_pool, n_pages);
  if (st != KDA_OK) return st;
  if (!aligned(s_in_page, 4) || !aligned(s_out_page, 4) || !aligned(ckpt_page, 4)) return KDA_ERR_ALIGNMENT;
  if (gate) {
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KDA_ERR_INVALID_ARG;
    if (!aligned(gate, 16) || !aligned(norm_weight, 16)) return KDA_ERR_ALIGNMENT;
  }
  kda::PageTables pt;
  pt.pool = state_pool; pt.n_pages = n_pages; pt.in = s_in_page; pt.out = s_out_page; pt.ckpt = ckpt_page;
  return prefill_impl(q, k, v, g, beta, gate, gate ? norm_weight : nullptr, gate ? eps : 0.f, nullptr, cu_seqlens,
                      n_seq, total_tokens, ckpt_off, ckpt_pos, n_ckpt, o, nullptr, nullptr, H, d, n_segments,
                      workspace, workspace_bytes, dev_status, stream, &pt);
}

size_t kda_decode_paged_workspace_size(int64_t n_pages) {
  return n_pages < 0 ? 0 : kda::page_check_bytes(n_pages);
}

kda_status kda_decode_paged(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                            const float* beta, float* state_pool, int64_t n_pages, const int32_t* s_in_page,
                            const int32_t* s_out_page, const int32_t* n_commit, float* o, int B, int n_tok, int H,
                            int d, void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_tok < 1 || n_tok > KDA_MAX_DECODE_TOKENS) return KDA_ERR_UNSUPPORTED;
  if (B < 0 || H < 0) return KDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  kda_status st = check_pool(state_pool, n_pages);
  if (st != KDA_OK) return st;
  if (B == 0 || H == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta || !o || !s_in_page) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(o, 16) ||
      !aligned(beta, 4) || !aligned(n_commit, 4) || !aligned(dev_status, 4) || !aligned(s_in_page, 4) ||
      !aligned(s_out_page, 4) || !aligned(workspace, 256))
    return KDA_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < kda::page_check_bytes(n_pages)) return KDA_ERR_WORKSPACE;
  if ((st = current_device(nullptr)) != KDA_OK) return st;
  const int64_t units = static_cast<int64_t>(B) * H;
  // in place (no out table): every unit writes its own entry page
  cudaError_t e = kda::launch_page_check(s_in_page, s_out_page ? s_out_page : s_in_page, units, nullptr, 0, n_pages,
                                         workspace, dev_status, stream);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  kda::PageTables pt;
  pt.pool = state_pool; pt.n_pages = n_pages; pt.in = s_in_page; pt.out = s_out_page;
  pt.fail = static_cast<const int*>(workspace);
  e = kda::launch_decode(q, k, v, g, beta, nullptr, n_commit, o, B, n_tok, H, dev_status, stream, pt);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode_fused(const kda_bf16* qp, const kda_bf16* kp, const kda_bf16* vp, const float* conv_w,
                            float* conv_cache, int conv_width, int conv_act, const float* z, const float* a_log,
                            float g_min, const float* b, const kda_bf16* gate, const float* norm_weight, float eps,
                            float* S_state, const int32_t* n_commit, float* o, int B, int n_tok, int H, int d,
                            int* dev_status, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_tok < 1 || n_tok > KDA_MAX_DECODE_TOKENS) return KDA_ERR_UNSUPPORTED;
  if (conv_width < 1 || conv_width > kda::kMaxConvWidth) return KDA_ERR_UNSUPPORTED;
  if (conv_act != 0 && conv_act != 1) return KDA_ERR_INVALID_ARG;
  if (!(g_min < 0.f) || !std::isfinite(g_min)) return KDA_ERR_INVALID_ARG;
  if (gate && (!(eps >= 0.f) || !std::isfinite(eps))) return KDA_ERR_INVALID_ARG;
  if (B < 0 || H < 0) return KDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return KDA_OK;
  if (!qp || !kp || !vp || !conv_w || !z || !a_log || !b || !S_state || !o) return KDA_ERR_INVALID_ARG;
  if (conv_width > 1 && !conv_cache) return KDA_ERR_INVALID_ARG;
  if (!aligned(S_state, 16) || !aligned(o, 16) || !aligned(qp, 2) || !aligned(kp, 2) || !aligned(vp, 2) ||
      !aligned(gate, 2) || !aligned(conv_w, 4) || !aligned(conv_cache, 4) || !aligned(z, 4) || !aligned(a_log, 4) ||
      !aligned(b, 4) || !aligned(norm_weight, 4) || !aligned(n_commit, 4) || !aligned(dev_status, 4))
    return KDA_ERR_ALIGNMENT;
  kda_status st = current_device(nullptr);
  if (st != KDA_OK) return st;
  kda::FrontEnd fe;
  fe.qp = qp; fe.kp = kp; fe.vp = vp; fe.conv_w = conv_w; fe.conv_cache = conv_cache; fe.W = conv_width;
  fe.act = conv_act; fe.z = z; fe.a_log = a_log; fe.g_min = g_min; fe.b = b;
  fe.gate = gate; fe.norm_weight = gate ? norm_weight : nullptr; fe.eps = gate ? eps : 0.f;
  cudaError_t e = kda::launch_decode_fused(fe, S_state, n_commit, o, B, n_tok, H, dev_status, stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_prefill_pairs(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens, float* M,
                             float* S_tilde, int H, int d, int* dev_status, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_seq < 0 || H < 0 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0x7fffffffLL || static_cast<int64_t>(n_seq) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (n_seq == 0 || H == 0) return KDA_OK;
  if (H > 65535 || n_seq > 0x7fffffff / 2) return KDA_ERR_UNSUPPORTED;  // grid: (2 n_seq, H)
  if (!cu_seqlens || !M || !S_tilde) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta)) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(M, 16) ||
      !aligned(S_tilde, 16) || !aligned(beta, 4) || !aligned(cu_seqlens, 4) || !aligned(dev_status, 4))
    return KDA_ERR_ALIGNMENT;
  int sms = 0;
  kda_status st = current_device(&sms);
  if (st != KDA_OK) return st;
  kda::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu_seqlens = cu_seqlens; a.n_seq = n_seq;
  a.total_tokens = total_tokens; a.H = H; a.status = dev_status; a.stream = stream;
  cudaError_t e = kda::launch_prefill_pairs(a, M, S_tilde, sms);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_combine_pairs(const float* M, const float* S_tilde, int n_pairs, const float* S_in, float* entry,
                             int n_seq, int H, int d, cudaStream_t stream) {
  if (d != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (n_pairs < 0 || n_seq < 0 || H < 0) return KDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_seq) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (n_seq == 0 || H == 0) return KDA_OK;
  if (H > 65535) return KDA_ERR_UNSUPPORTED;
  if (!entry || (n_pairs > 0 && (!M || !S_tilde))) return KDA_ERR_INVALID_ARG;
  if (!aligned(M, 16) || !aligned(S_tilde, 16) || !aligned(S_in, 16) || !aligned(entry, 16)) return KDA_ERR_ALIGNMENT;
  kda_status st = current_device(nullptr);
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_combine_pairs(M, S_tilde, n_pairs, S_in, entry, n_seq, H, stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
