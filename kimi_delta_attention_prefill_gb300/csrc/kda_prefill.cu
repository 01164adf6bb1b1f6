// kda_prefill.cu -- chunkwise KDA prefill on tcgen05 tensor cores (sm_103a).
//
// Chunk-level math ("Kimi K3 ... 服務性能", SemiAnalysis translation, section 6, the
// FlashKDA algorithm), per chunk of C = 64 tokens with entry state S (d_k x d_v):
//     G         = inclusive cumsum of g over the chunk (per channel);  a = exp(G)
//     K_decay   = a * K,   Q_decay = a * Q,   K_restore = exp(G_last - G) * K
//     L         = StrictTril(Diag(beta) K_decay K_inv^T),   M_qk = Tril(Q_decay K_inv^T)
//     INV       = (I + L)^-1
//     U         = INV Diag(beta) (V - K_decay S)
//     O         = Q_decay S + M_qk U
//     S        <- Diag(a_last) S + K_restore^T U
//
// Decay range.  K_inv = K / a is not representable over 64 tokens (with g >= -5 the
// cumulative log-decay reaches -320).  The pages bound the log-decay of a 16-token tile
// by -80 ("Kimi K3.1 Pro 架构完全拆解" 3.2), so the products for L and M_qk are formed
// per 16-token row block tb with reference token b = 16 tb:
//     row side    QA[t] = Q[t] exp(G[t] - G[b_tb(t)])              (<= 1)
//     column side B_tb[s] = K[s] exp(G[b_tb] - G[s]),  s < 16 (tb + 1)
//                 = K[s] exp(G[b_sb(s)] - G[s]) * exp(G[b_tb] - G[b_sb(s)])
//                   (first factor in [1, e^75], second <= 1)
// and row block tb reads its entries from the MMA with B_tb.  Every tile, diagonal ones
// included, is the same dense bf16 GEMM; nothing overflows.
//
// Precision.  L / M_qk use bf16 operands (the rebased factors need bf16's exponent
// range).  Every other product uses fp16 operands (11-bit significand, all values
// bounded by the normalised keys) with fp32 accumulation in TMEM; INV is formed in fp32
// on the CUDA cores.  The state lives in TMEM in fp32 for the whole sequence.
//
// One CTA (256 threads) runs one (sequence, head) chain serially over its chunks.
// Thread 0 issues TMA copies and tcgen05 MMAs; completion is tracked with mbarriers,
// every wait is bounded and a timeout ends the CTA with KDA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cstring>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

// TMEM columns.  S uses the 128-lane layout (lane = d_k row); P/U and O are M = 64
// accumulators (row t at lane 32 (t / 16) + t % 16).  The four L/M_qk accumulators
// overlap O: they are consumed before O is first written in a chunk.
constexpr uint32_t kTS = 0, kTP = 128, kTO = 256, kTLM = 256;
__host__ __device__ constexpr uint32_t lm_col(int tb) { return tb == 0 ? 0u : tb == 1 ? 16u : tb == 2 ? 48u : 96u; }

// Shared-memory map (bytes from a 1024-aligned base).
constexpr uint32_t SM_Q = 0;             // q tile (bf16, 2 K-panels)  -> Q_decay (fp16)
constexpr uint32_t SM_K = 16384;         // k tile                    -> K_decay (fp16)
constexpr uint32_t SM_G = 32768;         // g tile (fp32 [64][128])   -> [QA; KA] (bf16, 2 K-panels x 128 rows)
constexpr uint32_t SM_V = 65536;         // v tiles, two stages of 16 KiB
constexpr uint32_t SM_B = 98304;         // B_tb (bf16), 40 KiB      -> W, Ptmp, M_qk, INVbeta
constexpr uint32_t SM_KR = 139264;       // K_restore (fp16, [t][i], 2 M-panels)
constexpr uint32_t SM_XU = 155648;       // X then U (fp16, [t][j], 2 N-panels)
constexpr uint32_t SM_S = 172032;        // S (fp16, [i][j], 2 N-panels x 128 rows)
constexpr uint32_t SM_MISC = 204800;
// inside SM_B after the L/M_qk products are consumed
constexpr uint32_t SM_WL = SM_B;                 // fp32 [64][68]: L (strictly lower, row-scaled by beta)
constexpr uint32_t SM_WI = SM_B + 17408;         // fp32 [64][68]: INV, built block by block
constexpr uint32_t SM_PT = SM_B + 34816;         // fp32 4 x [16][16] block scratch (ends at SM_B + 38912)
constexpr uint32_t SM_INVB = SM_B;               // fp16 [64][64] K-major INV Diag(beta) (over L, once dead)
constexpr uint32_t SM_MQK = SM_MISC;             // fp16 [64][64] K-major M_qk (over the cumsum scratch)
__host__ __device__ constexpr uint32_t btb_off(int tb) { return tb == 0 ? 0u : tb == 1 ? 4096u : tb == 2 ? 12288u : 24576u; }
// misc
constexpr uint32_t SM_TOT = SM_MISC;             // fp32 [16][128] token-quad sums
constexpr uint32_t SM_GB = SM_TOT + 8192;        // fp32 [4][128] G at block starts
constexpr uint32_t SM_GL = SM_GB + 2048;         // fp32 [128]    G at the last token
constexpr uint32_t SM_AT = SM_GL + 512;          // fp32 [4][128] exp(G[b_tb])
constexpr uint32_t SM_RT = SM_AT + 2048;         // fp32 [4][128] exp(G_last - G[b_tb])
constexpr uint32_t SM_F = SM_RT + 2048;          // fp32 [6][128] exp(G[b_tb] - G[b_sb])
constexpr uint32_t SM_AL = SM_F + 3072;          // fp32 [128]    a_last
constexpr uint32_t SM_BETA = SM_AL + 512;        // fp32 [64]
constexpr uint32_t SM_BAR = SM_BETA + 256;       // mbarriers
constexpr uint32_t SM_CTRL = SM_BAR + 64;        // tmem slot, flags
constexpr uint32_t kSmemBytes = SM_CTRL + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
static_assert(kSmemAlloc <= 232448, "shared memory budget");

enum { BAR_IN = 0, BAR_V0 = 1, BAR_V1 = 2, BAR_LM = 3, BAR_P = 4, BAR_U = 5, BAR_S = 6, kNumBars = 7 };

struct Work {
  int seq, h;
  int64_t bos;       // first packed row of the sequence
  int len;           // tokens in the sequence
  int c0, c1;        // chunk range [c0, c1) of this CTA
  const float* entry;  // entry state [128][128] or nullptr (zeros)
  float* s_out;        // final state destination or nullptr
  int ck_begin, ck_end;  // checkpoint slots this CTA may write
};

struct KParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_g;
  const float* beta;
  const float* S_in;
  const int32_t* cu;
  const int32_t* ckpt_off;
  const int32_t* ckpt_pos;
  __nv_bfloat16* o;
  float* S_out;
  float* ckpts;
  int* status;
  int n_seq, H;
  int64_t total_tokens;
  int64_t n_ckpt;
  const int4* items;      // work items (split path) or nullptr: item x = whole sequence x
  const int* item_count;  // device count of valid items
  float* slots;           // split-path state slots [slot][H][3][128][128]
};

__device__ __forceinline__ float4 ld4(const uint8_t* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}

// Validate this sequence's slice of cu_seqlens / checkpoints (device-side argument
// contents).  Returns true when usable.
__device__ bool check_sequence(const KParams& p, int seq, int64_t& bos, int& len, int& cb, int& ce) {
  const int64_t a = p.cu[seq], b = p.cu[seq + 1];
  if (a < 0 || b < a || b > p.total_tokens) return false;
  if (seq == 0 && a != 0) return false;
  if (seq == p.n_seq - 1 && b != p.total_tokens) return false;
  bos = a;
  len = static_cast<int>(b - a);
  cb = ce = 0;
  if (p.ckpt_off) {
    cb = p.ckpt_off[seq];
    ce = p.ckpt_off[seq + 1];
    if (cb < 0 || ce < cb || ce > p.n_ckpt) return false;
    if (seq == 0 && cb != 0) return false;
    if (seq == p.n_seq - 1 && ce != p.n_ckpt) return false;
    int prev = 0;
    for (int j = cb; j < ce; ++j) {
      const int pos = p.ckpt_pos[j];
      if (pos <= prev || pos > len) return false;
      if ((pos % kChunk) != 0 && pos != len) return false;
      prev = pos;
    }
  }
  return true;
}

// ------------------------------------------------------------- INV = (I + L)^-1
// L is 64 x 64 strictly lower triangular, fp32 in shared memory with row stride kLdw.
// Block forward substitution over 16 x 16 blocks (D_i = (I + L_ii)^-1):
//     INV_ii = D_i,   INV_ij = -D_i (L_ij D_j + sum_{j<k<i} L_ik INV_kj)   (i > j)
// evaluated in dependency stages, one warp per 16 x 16 block product.  The result is
// scaled by beta along columns and stored as the fp16 K-major operand INV Diag(beta).
constexpr int kLdw = 68;  // padded row stride (floats): conflict-free float4 row reads

// acc += A * B for 16 x 16 blocks; lane owns row lane / 2, columns 8 (lane % 2) .. +7.
__device__ __forceinline__ void blk_mac(const float* A, int lda, const float* B, int ldb, float (&acc)[8], int lane) {
  const int r = lane >> 1, c0 = (lane & 1) * 8;
  float a[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = *reinterpret_cast<const float4*>(A + r * lda + 4 * q);
    a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float4 b0 = *reinterpret_cast<const float4*>(B + k * ldb + c0);
    const float4 b1 = *reinterpret_cast<const float4*>(B + k * ldb + c0 + 4);
    acc[0] += a[k] * b0.x; acc[1] += a[k] * b0.y; acc[2] += a[k] * b0.z; acc[3] += a[k] * b0.w;
    acc[4] += a[k] * b1.x; acc[5] += a[k] * b1.y; acc[6] += a[k] * b1.z; acc[7] += a[k] * b1.w;
  }
}
__device__ __forceinline__ void blk_load(const float* C, int ldc, float (&acc)[8], int lane) {
  const int r = lane >> 1, c0 = (lane & 1) * 8;
  const float4 x = *reinterpret_cast<const float4*>(C + r * ldc + c0);
  const float4 y = *reinterpret_cast<const float4*>(C + r * ldc + c0 + 4);
  acc[0] = x.x; acc[1] = x.y; acc[2] = x.z; acc[3] = x.w; acc[4] = y.x; acc[5] = y.y; acc[6] = y.z; acc[7] = y.w;
}
__device__ __forceinline__ void blk_store(float* C, int ldc, const float (&acc)[8], int lane, float sign) {
  const int r = lane >> 1, c0 = (lane & 1) * 8;
  *reinterpret_cast<float4*>(C + r * ldc + c0) = make_float4(sign * acc[0], sign * acc[1], sign * acc[2], sign * acc[3]);
  *reinterpret_cast<float4*>(C + r * ldc + c0 + 4) = make_float4(sign * acc[4], sign * acc[5], sign * acc[6], sign * acc[7]);
}
__device__ __forceinline__ void blk_copy(const float* S, int lds, float* D, int ldd, int lane) {
  float acc[8];
  blk_load(S, lds, acc, lane);
  blk_store(D, ldd, acc, lane, 1.f);
}

// All 256 threads call this (it synchronises the CTA).
__device__ void invert_unit_lower(const float* WL, float* WI, float* PT, const float* beta, uint8_t* invb, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  auto L = [&](int i, int j) { return WL + 16 * i * kLdw + 16 * j; };
  auto I = [&](int i, int j) { return WI + 16 * i * kLdw + 16 * j; };
  auto P = [&](int k) { return PT + 256 * k; };

  // diagonal blocks: thread (b, c) solves column c of (I + L_bb) x = e_c
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15;
    const float* Lb = L(b, b);
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m) s += Lb[r * kLdw + m] * x[m];
      x[r] = (r == c) ? 1.f : (r < c ? 0.f : -s);
    }
    float* Db = I(b, b);
#pragma unroll
    for (int r = 0; r < 16; ++r) Db[r * kLdw + c] = x[r];
  }
  __syncthreads();
  // T_ij = L_ij D_j (stored where INV_ij will go)
  if (warp < 6) {
    const int i = warp < 1 ? 1 : warp < 3 ? 2 : 3;
    const int j = warp < 1 ? 0 : warp < 3 ? warp - 1 : warp - 3;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    blk_mac(L(i, j), kLdw, I(j, j), kLdw, acc, lane);
    blk_store(I(i, j), kLdw, acc, lane, 1.f);
  }
  __syncthreads();
  // INV_{i,i-1} = -D_i T_{i,i-1} -> P(i-1)
  if (warp < 3) {
    const int i = warp + 1;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    blk_mac(I(i, i), kLdw, I(i, i - 1), kLdw, acc, lane);
    blk_store(P(i - 1), 16, acc, lane, -1.f);
  }
  __syncthreads();
  // R_20 = T_20 + L_21 INV_10, R_31 = T_31 + L_32 INV_21 (in place); first sub-diagonal into place
  if (warp < 2) {
    const int i = warp + 2, j = warp;
    float acc[8];
    blk_load(I(i, j), kLdw, acc, lane);
    blk_mac(L(i, i - 1), kLdw, P(j), 16, acc, lane);
    blk_store(I(i, j), kLdw, acc, lane, 1.f);
  } else if (warp < 5) {
    const int k = warp - 2;
    blk_copy(P(k), 16, I(k + 1, k), kLdw, lane);
  }
  __syncthreads();
  // INV_20 = -D_2 R_20 -> P(0), INV_31 = -D_3 R_31 -> P(1)
  if (warp < 2) {
    const int i = warp + 2, j = warp;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    blk_mac(I(i, i), kLdw, I(i, j), kLdw, acc, lane);
    blk_store(P(j), 16, acc, lane, -1.f);
  }
  __syncthreads();
  // R_30 = T_30 + L_31 INV_10 + L_32 INV_20 (in place); second sub-diagonal into place
  if (warp == 0) {
    float acc[8];
    blk_load(I(3, 0), kLdw, acc, lane);
    blk_mac(L(3, 1), kLdw, I(1, 0), kLdw, acc, lane);
    blk_mac(L(3, 2), kLdw, P(0), 16, acc, lane);
    blk_store(I(3, 0), kLdw, acc, lane, 1.f);
  } else if (warp == 1) {
    blk_copy(P(0), 16, I(2, 0), kLdw, lane);
  } else if (warp == 2) {
    blk_copy(P(1), 16, I(3, 1), kLdw, lane);
  }
  __syncthreads();
  // INV_30 = -D_3 R_30 (warp 0, registers); every block -> INV Diag(beta), fp16, K-major [t][s].
  // The fp16 operand overwrites L, which is no longer read.
  auto put8 = [&](int t, int g, const float (&v)[8]) {
    const int s0 = 8 * g;
    st4(invb + sw128(t, 2 * s0), pack_half2(v[0] * beta[s0], v[1] * beta[s0 + 1]),
        pack_half2(v[2] * beta[s0 + 2], v[3] * beta[s0 + 3]), pack_half2(v[4] * beta[s0 + 4], v[5] * beta[s0 + 5]),
        pack_half2(v[6] * beta[s0 + 6], v[7] * beta[s0 + 7]));
  };
  if (warp == 0) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    blk_mac(I(3, 3), kLdw, I(3, 0), kLdw, acc, lane);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = -acc[e];
    put8(48 + (lane >> 1), lane & 1, acc);
  } else {
    for (int task = tid - 32; task < 512; task += kThreads - 32) {
      const int t = task >> 3, g = task & 7;
      if (t >= 48 && g < 2) continue;  // block (3, 0): warp 0
      float v[8];
      if ((g >> 1) > (t >> 4)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
      } else {
        const float4 x = *reinterpret_cast<const float4*>(WI + t * kLdw + 8 * g);
        const float4 y = *reinterpret_cast<const float4*>(WI + t * kLdw + 8 * g + 4);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
      }
      put8(t, g, v);
    }
  }
}

__device__ __forceinline__ void issue_tile_loads(const KParams& p, uint8_t* sm, uint64_t* bars, int which, int h,
                                                 int64_t row0, int vstage) {
  // which: bit0 q, bit1 k, bit2 g, bit3 v
  const int r = static_cast<int>(row0);
  if (which & 1) {
    tma_load_3d(sm + SM_Q, &p.tm_q, &bars[BAR_IN], 0, h, r);
    tma_load_3d(sm + SM_Q + 8192, &p.tm_q, &bars[BAR_IN], 64, h, r);
  }
  if (which & 2) {
    tma_load_3d(sm + SM_K, &p.tm_k, &bars[BAR_IN], 0, h, r);
    tma_load_3d(sm + SM_K + 8192, &p.tm_k, &bars[BAR_IN], 64, h, r);
  }
  if (which & 4) tma_load_3d(sm + SM_G, &p.tm_g, &bars[BAR_IN], 0, h, r);
  if (which & 8) {
    uint8_t* dst = sm + SM_V + vstage * 16384;
    tma_load_3d(dst, &p.tm_v, &bars[BAR_V0 + vstage], 0, h, r);
    tma_load_3d(dst + 8192, &p.tm_v, &bars[BAR_V0 + vstage], 64, h, r);
  }
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM_BAR);
  volatile int* ctrl = reinterpret_cast<volatile int*>(sm + SM_CTRL);  // [0] tmem base, [1] abort, [2] valid
  float* s_beta = reinterpret_cast<float*>(sm + SM_BETA);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, hcol = warp >> 2;

  // ---- work item: (sequence, head, chunk range, mode)
  int4 it;
  if (p.items) {
    if (static_cast<int>(blockIdx.x) >= *p.item_count) return;
    it = p.items[blockIdx.x];
  } else {
    it = make_int4(static_cast<int>(blockIdx.x), 0, -1, kModeFull);
  }
  const int mode = it.w & 7, slot = it.w >> 3;
  Work w;
  w.seq = it.x;
  w.h = blockIdx.y;
  if (tid == 0) {
    int64_t bos; int len, cb, ce;
    const bool ok = check_sequence(p, w.seq, bos, len, cb, ce);
    ctrl[2] = ok ? 1 : 0;
    if (!ok) report_status(p.status, 7 /* KDA_ERR_DEVICE_CHECK */);
  }
  __syncthreads();
  if (!ctrl[2]) return;
  const bool do_o = mode == kModeFull || mode == kModeFirst || mode == kModeTail;
  const bool v_zero = mode == kModeTrans, entry_identity = mode == kModeTrans;
  {
    const int64_t a = p.cu[w.seq], b = p.cu[w.seq + 1];
    const int64_t unit = static_cast<int64_t>(w.seq) * p.H + w.h;
    auto slot_buf = [&](int buf) { return p.slots + ((static_cast<int64_t>(slot) * p.H + w.h) * 3 + buf) * (kHeadDim * kHeadDim); };
    w.bos = a;
    w.len = static_cast<int>(b - a);
    const int nch = (w.len + kChunk - 1) / kChunk;
    w.c0 = it.y;
    w.c1 = it.z < 0 ? nch : it.z;
    float* s_out = p.S_out ? p.S_out + unit * (kHeadDim * kHeadDim) : nullptr;
    const float* s_in = p.S_in ? p.S_in + unit * (kHeadDim * kHeadDim) : nullptr;
    switch (mode) {
      case kModeFirst: w.entry = s_in; w.s_out = slot_buf(0); break;
      case kModeZero: w.entry = nullptr; w.s_out = slot_buf(0); break;
      case kModeTrans: w.entry = nullptr; w.s_out = slot_buf(1); break;
      case kModeTail: w.entry = slot_buf(2); w.s_out = (w.c1 == nch) ? s_out : nullptr; break;
      default: w.entry = s_in; w.s_out = s_out; break;
    }
    w.ck_begin = w.ck_end = 0;
    if (do_o && p.ckpt_off) {
      w.ck_end = p.ckpt_off[w.seq + 1];
      int j = p.ckpt_off[w.seq];
      while (j < w.ck_end && p.ckpt_pos[j] <= w.c0 * kChunk) ++j;
      w.ck_begin = j;
    }
  }

  // ---- empty sequence: the final state is the entry state
  if (w.c1 <= w.c0) {
    if (w.s_out)
      for (int e = tid; e < kHeadDim * kHeadDim; e += kThreads) w.s_out[e] = w.entry ? w.entry[e] : 0.f;
    return;
  }

  // ---- setup: barriers, TMEM, tensor-map prefetch, first loads
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q); tma_prefetch_desc(&p.tm_k); tma_prefetch_desc(&p.tm_v); tma_prefetch_desc(&p.tm_g);
    ctrl[1] = 0;
  }
  if (warp == 0) { tmem_alloc(reinterpret_cast<uint32_t*>(sm + SM_CTRL), kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(ctrl[0]);
  const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;  // this warp's lane base

  if (tid == 0) {
    const int64_t row0 = w.bos + static_cast<int64_t>(w.c0) * kChunk;
    mbar_arrive_expect_tx(&bars[BAR_IN], 65536);
    issue_tile_loads(p, sm, bars, 1 | 2 | 4, w.h, row0, 0);
    mbar_arrive_expect_tx(&bars[BAR_V0], 16384);
    issue_tile_loads(p, sm, bars, 8, w.h, row0, 0);
  }

  // ---- entry state -> TMEM (fp32) and the fp16 operand copy
  {
    const int i = quarter * 32 + lane;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float r[16];
      const int c = hcol * 64 + m * 16;
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        float4 v4 = w.entry ? *reinterpret_cast<const float4*>(w.entry + i * kHeadDim + c + e) : make_float4(0, 0, 0, 0);
        if (entry_identity)
          v4 = make_float4(i == c + e ? 1.f : 0.f, i == c + e + 1 ? 1.f : 0.f, i == c + e + 2 ? 1.f : 0.f,
                           i == c + e + 3 ? 1.f : 0.f);
        r[e] = v4.x; r[e + 1] = v4.y; r[e + 2] = v4.z; r[e + 3] = v4.w;
      }
      tmem_st16(tmem + tl + kTS + c, r);
      uint8_t* dst = sm + SM_S + hcol * 16384;
      st4(dst + sw128(i, 32 * m), pack_half2(r[0], r[1]), pack_half2(r[2], r[3]), pack_half2(r[4], r[5]),
          pack_half2(r[6], r[7]));
      st4(dst + sw128(i, 32 * m + 16), pack_half2(r[8], r[9]), pack_half2(r[10], r[11]), pack_half2(r[12], r[13]),
          pack_half2(r[14], r[15]));
    }
    tmem_wait_st();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // Descriptor bases; per-k-step offsets are added in 16-byte units.
  const uint64_t dG = smem_desc(smem_u32(sm + SM_G), 16, 1024, kSwizzle128B);     // [QA; KA], K-panel 16384 B
  const uint64_t dK = smem_desc(smem_u32(sm + SM_K), 16, 1024, kSwizzle128B);     // K_decay, K-panel 8192 B
  const uint64_t dQ = smem_desc(smem_u32(sm + SM_Q), 16, 1024, kSwizzle128B);     // Q_decay
  const uint64_t dS = smem_desc(smem_u32(sm + SM_S), 16384, 1024, kSwizzle128B);  // S, MN-major, k-step 2048 B
  const uint64_t dInv = smem_desc(smem_u32(sm + SM_INVB), 16, 1024, kSwizzle128B);
  const uint64_t dXU = smem_desc(smem_u32(sm + SM_XU), 8192, 1024, kSwizzle128B);  // MN-major, k-step 2048 B
  const uint64_t dKR = smem_desc(smem_u32(sm + SM_KR), 8192, 1024, kSwizzle128B);  // MN-major A, k-step 2048 B
  const uint64_t dMq = smem_desc(smem_u32(sm + SM_MQK), 16, 1024, kSwizzle128B);
  const uint64_t dB0 = smem_desc(smem_u32(sm + SM_B), 16, 1024, kSwizzle128B);

  int ck = w.ck_begin;
  bool aborted = false;
  const int n_chunks = w.c1 - w.c0;
  float beta_next = 0.f;
  if (tid < kChunk) {
    const int64_t r = w.bos + static_cast<int64_t>(w.c0) * kChunk + tid;
    beta_next = (tid < min(kChunk, w.len - w.c0 * kChunk)) ? p.beta[r * p.H + w.h] : 0.f;
  }
  for (int n = 0; n < n_chunks && !aborted; ++n) {
    const int cidx = w.c0 + n;
    const int64_t row0 = w.bos + static_cast<int64_t>(cidx) * kChunk;
    const int valid = min(kChunk, w.len - cidx * kChunk);
    const int vstage = n & 1;
    const bool has_next = (n + 1) < n_chunks;
    const int64_t row_next = row0 + kChunk;

    // ---- 1. inputs of this chunk
    if (tid < kChunk) {
      s_beta[tid] = beta_next;
      const int vn = has_next ? min(kChunk, w.len - (cidx + 1) * kChunk) : 0;
      beta_next = tid < vn ? p.beta[(row_next + tid) * p.H + w.h] : 0.f;
    }
    bool ok = mbar_wait(&bars[BAR_IN], n & 1) && mbar_wait(&bars[BAR_V0 + vstage], (n >> 1) & 1);
    if (!ok) { if (tid == 0) ctrl[1] = 1; }
    if (tid == 0 && ok && has_next) {
      mbar_arrive_expect_tx(&bars[BAR_V0 + (vstage ^ 1)], 16384);
      issue_tile_loads(p, sm, bars, 8, w.h, row_next, vstage ^ 1);
    }

    // ---- 2. decay prep: cumsum, per-block factors, operands
    const int tq = tid >> 4, cg = tid & 15, tb = tq >> 2;
    float G[4][8];
    {
      const uint8_t* gt = sm + SM_G;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = tq * 4 + u;
        float4 a = ld4(gt + t * 512 + cg * 32), b = ld4(gt + t * 512 + cg * 32 + 16);
        const bool m = t < valid;
        G[u][0] = m ? a.x : 0.f; G[u][1] = m ? a.y : 0.f; G[u][2] = m ? a.z : 0.f; G[u][3] = m ? a.w : 0.f;
        G[u][4] = m ? b.x : 0.f; G[u][5] = m ? b.y : 0.f; G[u][6] = m ? b.z : 0.f; G[u][7] = m ? b.w : 0.f;
      }
#pragma unroll
      for (int u = 1; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) G[u][e] += G[u - 1][e];
      float* tot = reinterpret_cast<float*>(sm + SM_TOT);
      *reinterpret_cast<float4*>(tot + tq * 128 + cg * 8) = make_float4(G[3][0], G[3][1], G[3][2], G[3][3]);
      *reinterpret_cast<float4*>(tot + tq * 128 + cg * 8 + 4) = make_float4(G[3][4], G[3][5], G[3][6], G[3][7]);
    }
    __syncthreads();
    if (ctrl[1]) { aborted = true; break; }
    {
      const float* tot = reinterpret_cast<const float*>(sm + SM_TOT);
      float off[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int j = 0; j < tq; ++j) {
        const float4 a = *reinterpret_cast<const float4*>(tot + j * 128 + cg * 8);
        const float4 b = *reinterpret_cast<const float4*>(tot + j * 128 + cg * 8 + 4);
        off[0] += a.x; off[1] += a.y; off[2] += a.z; off[3] += a.w;
        off[4] += b.x; off[5] += b.y; off[6] += b.z; off[7] += b.w;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) G[u][e] += off[e];
      if ((tq & 3) == 0) {
        float* gb = reinterpret_cast<float*>(sm + SM_GB) + (tq >> 2) * 128 + cg * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) gb[e] = G[0][e];
      }
      if (tq == 15) {
        float* gl = reinterpret_cast<float*>(sm + SM_GL) + cg * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) gl[e] = G[3][e];
      }
    }
    __syncthreads();
    {
      const int i = tid & 127;
      const float* gb = reinterpret_cast<const float*>(sm + SM_GB);
      const float gl = reinterpret_cast<const float*>(sm + SM_GL)[i];
      if (tid < 128) {
        float* at = reinterpret_cast<float*>(sm + SM_AT);
        float* rt = reinterpret_cast<float*>(sm + SM_RT);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          at[b * 128 + i] = __expf(gb[b * 128 + i]);
          rt[b * 128 + i] = __expf(gl - gb[b * 128 + i]);
        }
        reinterpret_cast<float*>(sm + SM_AL)[i] = __expf(gl);
      } else {
        float* f = reinterpret_cast<float*>(sm + SM_F);
        int idx = 0;
#pragma unroll
        for (int b = 1; b < 4; ++b)
#pragma unroll
          for (int s = 0; s < b; ++s, ++idx) f[idx * 128 + i] = __expf(gb[b * 128 + i] - gb[s * 128 + i]);
      }
    }
    __syncthreads();
    {
      const float* gb = reinterpret_cast<const float*>(sm + SM_GB) + tb * 128 + cg * 8;
      const float* at = reinterpret_cast<const float*>(sm + SM_AT) + tb * 128 + cg * 8;
      const float* rt = reinterpret_cast<const float*>(sm + SM_RT) + tb * 128 + cg * 8;
      const float* fp = reinterpret_cast<const float*>(sm + SM_F);
      const int kpanel = cg >> 3, kchunk = cg & 7;
      float gbr[8], atr[8], rtr[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) { gbr[e] = gb[e]; atr[e] = at[e]; rtr[e] = rt[e]; }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = tq * 4 + u;
        const bool m = t < valid;
        const uint32_t so = sw128(t, 16 * kchunk);
        uint8_t* qp = sm + SM_Q + kpanel * 8192 + so;
        uint8_t* kp = sm + SM_K + kpanel * 8192 + so;
        float qf[8], kf[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(qp), qf);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(kp), kf);
        float qd[8], kd[8], qa[8], ka[8], kb[8], kr[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float kk = m ? kf[e] : 0.f;
          const float x = G[u][e] - gbr[e];   // <= 0, >= -75
          const float E = __expf(x);
          const float Ei = __expf(-x);
          qa[e] = qf[e] * E;
          ka[e] = kk * E;
          qd[e] = qa[e] * atr[e];
          kd[e] = ka[e] * atr[e];
          kb[e] = kk * Ei;
          kr[e] = kb[e] * rtr[e];
        }
        st4(qp, pack_half2(qd[0], qd[1]), pack_half2(qd[2], qd[3]), pack_half2(qd[4], qd[5]), pack_half2(qd[6], qd[7]));
        st4(kp, pack_half2(kd[0], kd[1]), pack_half2(kd[2], kd[3]), pack_half2(kd[4], kd[5]), pack_half2(kd[6], kd[7]));
        uint8_t* qa_p = sm + SM_G + kpanel * 16384;
        st4(qa_p + so, pack_bf162(qa[0], qa[1]), pack_bf162(qa[2], qa[3]), pack_bf162(qa[4], qa[5]),
            pack_bf162(qa[6], qa[7]));
        st4(qa_p + sw128(64 + t, 16 * kchunk), pack_bf162(ka[0], ka[1]), pack_bf162(ka[2], ka[3]),
            pack_bf162(ka[4], ka[5]), pack_bf162(ka[6], ka[7]));
        st4(sm + SM_KR + kpanel * 8192 + so, pack_half2(kr[0], kr[1]), pack_half2(kr[2], kr[3]),
            pack_half2(kr[4], kr[5]), pack_half2(kr[6], kr[7]));
#pragma unroll
        for (int tb2 = 0; tb2 < 4; ++tb2) {
          if (tb2 < tb) continue;
          float sc[8];
          if (tb2 == tb) {
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[e] = kb[e];
          } else {
            const float* f = fp + ((tb2 * (tb2 - 1)) / 2 + tb) * 128 + cg * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[e] = kb[e] * f[e];
          }
          const uint32_t rows = 16u * (tb2 + 1);
          st4(sm + SM_B + btb_off(tb2) + kpanel * rows * 128 + so, pack_bf162(sc[0], sc[1]), pack_bf162(sc[2], sc[3]),
              pack_bf162(sc[4], sc[5]), pack_bf162(sc[6], sc[7]));
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- 3. L / M_qk products (bf16) and K_decay S (fp16)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t rows = 16u * (b + 1);
        const uint32_t idesc = idesc_f16(128, rows, true, false, false);
        const uint64_t db = dB0 + (btb_off(b) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = dG + (((kk >> 2) * 16384 + 32 * (kk & 3)) >> 4);
          const uint64_t bd = db + (((kk >> 2) * rows * 128 + 32 * (kk & 3)) >> 4);
          mma_f16(tmem + kTLM + lm_col(b), ad, bd, idesc, kk > 0);
        }
      }
      mma_commit(&bars[BAR_LM]);
      const uint32_t idesc = idesc_f16(64, 128, false, false, true);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_f16(tmem + kTP, dK + (((kk >> 2) * 8192 + 32 * (kk & 3)) >> 4), dS + ((kk * 2048) >> 4), idesc, kk > 0);
      mma_commit(&bars[BAR_P]);
    }

    // ---- 4. S <- Diag(a_last) S in TMEM (the previous chunk's update has completed)
    {
      const int i = quarter * 32 + lane;
      const float al = reinterpret_cast<const float*>(sm + SM_AL)[i];
      float r[4][16];
#pragma unroll
      for (int m = 0; m < 4; ++m) tmem_ld16(tmem + tl + kTS + hcol * 64 + m * 16, r[m]);
      tmem_wait_ld();
#pragma unroll
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int e = 0; e < 16; ++e) r[m][e] *= al;
        tmem_st16(tmem + tl + kTS + hcol * 64 + m * 16, r[m]);
      }
      tmem_wait_st();
    }

    // ---- 5. read L and M_qk (row block tb reads the accumulator built with B_tb)
    ok = mbar_wait(&bars[BAR_LM], n & 1);
    if (!ok && tid == 0) ctrl[1] = 1;
    tc_fence_after();
    if (hcol == 0) {
      // quarter 0/1: M_qk rows 0..63 ; quarter 2/3: L rows 0..63
      const bool is_l = quarter >= 2;
      const int t = (quarter & 1) * 32 + lane;
      const int tbl = t >> 4;
      const int g0 = (quarter & 1) ? 3 : 0, ng = (quarter & 1) ? 7 : 3;  // 16-column groups of this warp
      const int lo = static_cast<int>(lm_col(tbl)), hi = lo + 16 * (tbl + 1);
      const float bt = s_beta[t];
      float r[7][16];
#pragma unroll
      for (int gi = 0; gi < 7; ++gi)
        if (gi < ng) tmem_ld16(tmem + tl + kTLM + (g0 + gi) * 16, r[gi]);
      tmem_wait_ld();
#pragma unroll
      for (int gi = 0; gi < 7; ++gi) {
        const int col = (g0 + gi) * 16;
        if (gi >= ng || col < lo || col >= hi) continue;
        const int s0 = col - lo;  // s block start
        if (is_l) {
          float* wr = reinterpret_cast<float*>(sm + SM_WL) + t * kLdw + s0;
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(wr + e) =
                make_float4((s0 + e < t) ? bt * r[gi][e] : 0.f, (s0 + e + 1 < t) ? bt * r[gi][e + 1] : 0.f,
                            (s0 + e + 2 < t) ? bt * r[gi][e + 2] : 0.f, (s0 + e + 3 < t) ? bt * r[gi][e + 3] : 0.f);
        } else {
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = (s0 + e <= t) ? r[gi][e] : 0.f;
          uint8_t* mp = sm + SM_MQK;
          st4(mp + sw128(t, 2 * s0), pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]),
              pack_half2(v[6], v[7]));
          st4(mp + sw128(t, 2 * s0 + 16), pack_half2(v[8], v[9]), pack_half2(v[10], v[11]), pack_half2(v[12], v[13]),
              pack_half2(v[14], v[15]));
        }
      }
      // zero the s blocks past this row's block
      for (int sb = tbl + 1; sb < 4; ++sb) {
        if (is_l) {
          float* wr = reinterpret_cast<float*>(sm + SM_WL) + t * kLdw + sb * 16;
#pragma unroll
          for (int e = 0; e < 16; e += 4) *reinterpret_cast<float4*>(wr + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          uint8_t* mp = sm + SM_MQK;
          st4(mp + sw128(t, 32 * sb), 0, 0, 0, 0);
          st4(mp + sw128(t, 32 * sb + 16), 0, 0, 0, 0);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctrl[1]) { aborted = true; break; }

    // ---- 6. next chunk's g; O = Q_decay S (fp16)
    if (tid == 0) {
      tc_fence_after();
      if (has_next) {
        mbar_arrive_expect_tx(&bars[BAR_IN], 65536);
        issue_tile_loads(p, sm, bars, 4, w.h, row_next, 0);
      }
      if (do_o) {
        const uint32_t idesc = idesc_f16(64, 128, false, false, true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16(tmem + kTO, dQ + (((kk >> 2) * 8192 + 32 * (kk & 3)) >> 4), dS + ((kk * 2048) >> 4), idesc, kk > 0);
      }
    }

    // ---- 7. INV = (I + L)^-1 in fp32 by 16 x 16 blocks, then INV Diag(beta) as fp16
    invert_unit_lower(reinterpret_cast<float*>(sm + SM_WL), reinterpret_cast<float*>(sm + SM_WI),
                      reinterpret_cast<float*>(sm + SM_PT), s_beta, sm + SM_INVB, tid);

    // ---- 8. X = V - K_decay S  (rows past the sequence end are zero)
    ok = mbar_wait(&bars[BAR_P], n & 1);
    if (!ok && tid == 0) ctrl[1] = 1;
    tc_fence_after();
    {
      const int t = quarter * 16 + (lane & 15);
      const uint8_t* vt = sm + SM_V + vstage * 16384 + hcol * 8192;
      uint8_t* xp = sm + SM_XU + hcol * 8192;
      float r[4][16];
#pragma unroll
      for (int m = 0; m < 4; ++m) tmem_ld16(tmem + tl + kTP + hcol * 64 + m * 16, r[m]);
      tmem_wait_ld();
      if (lane < 16) {
        const bool mk = t < valid;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float v0[8], v1[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(vt + sw128(t, 32 * m)), v0);
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(vt + sw128(t, 32 * m + 16)), v1);
          float x[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = mk ? (v_zero ? 0.f : v0[e]) - r[m][e] : 0.f;
            x[8 + e] = mk ? (v_zero ? 0.f : v1[e]) - r[m][8 + e] : 0.f;
          }
          st4(xp + sw128(t, 32 * m), pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
              pack_half2(x[6], x[7]));
          st4(xp + sw128(t, 32 * m + 16), pack_half2(x[8], x[9]), pack_half2(x[10], x[11]), pack_half2(x[12], x[13]),
              pack_half2(x[14], x[15]));
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctrl[1]) { aborted = true; break; }

    // ---- 9. next chunk's k; U = INV Diag(beta) X
    if (tid == 0) {
      tc_fence_after();
      if (has_next) issue_tile_loads(p, sm, bars, 2, w.h, row_next, 0);
      const uint32_t idesc = idesc_f16(64, 128, false, false, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_f16(tmem + kTP, dInv + ((32 * kk) >> 4), dXU + ((kk * 2048) >> 4), idesc, kk > 0);
      mma_commit(&bars[BAR_U]);
    }

    // ---- 10. U -> fp16 operand
    ok = mbar_wait(&bars[BAR_U], n & 1);
    if (!ok && tid == 0) ctrl[1] = 1;
    tc_fence_after();
    {
      const int t = quarter * 16 + (lane & 15);
      uint8_t* up = sm + SM_XU + hcol * 8192;
      float r[4][16];
#pragma unroll
      for (int m = 0; m < 4; ++m) tmem_ld16(tmem + tl + kTP + hcol * 64 + m * 16, r[m]);
      tmem_wait_ld();
      if (lane < 16) {
        const bool mk = t < valid;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[m][e] = mk ? r[m][e] : 0.f;
          st4(up + sw128(t, 32 * m), pack_half2(r[m][0], r[m][1]), pack_half2(r[m][2], r[m][3]),
              pack_half2(r[m][4], r[m][5]), pack_half2(r[m][6], r[m][7]));
          st4(up + sw128(t, 32 * m + 16), pack_half2(r[m][8], r[m][9]), pack_half2(r[m][10], r[m][11]),
              pack_half2(r[m][12], r[m][13]), pack_half2(r[m][14], r[m][15]));
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctrl[1]) { aborted = true; break; }

    // ---- 11. next chunk's q; S += K_restore^T U; O += M_qk U
    if (tid == 0) {
      tc_fence_after();
      if (has_next) issue_tile_loads(p, sm, bars, 1, w.h, row_next, 0);
      const uint32_t id_s = idesc_f16(128, 128, false, true, true);
      const uint32_t id_o = idesc_f16(64, 128, false, false, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ud = dXU + ((kk * 2048) >> 4);
        mma_f16(tmem + kTS, dKR + ((kk * 2048) >> 4), ud, id_s, 1);
        if (do_o) mma_f16(tmem + kTO, dMq + ((32 * kk) >> 4), ud, id_o, 1);
      }
      mma_commit(&bars[BAR_S]);
    }

    // ---- 12. outputs, next S operand, checkpoint / final state
    ok = mbar_wait(&bars[BAR_S], n & 1);
    if (!ok && tid == 0) ctrl[1] = 1;
    tc_fence_after();
    {
      const int t = quarter * 16 + (lane & 15);
      const bool wr = do_o && lane < 16 && t < valid;
      __nv_bfloat16* orow = p.o + ((row0 + t) * p.H + w.h) * kHeadDim + hcol * 64;
      float r[4][16];
      if (do_o) {
#pragma unroll
        for (int m = 0; m < 4; ++m) tmem_ld16(tmem + tl + kTO + hcol * 64 + m * 16, r[m]);
        tmem_wait_ld();
      }
      if (wr) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4* dst = reinterpret_cast<uint4*>(orow + m * 16);
          dst[0] = make_uint4(pack_bf162(r[m][0], r[m][1]), pack_bf162(r[m][2], r[m][3]), pack_bf162(r[m][4], r[m][5]),
                              pack_bf162(r[m][6], r[m][7]));
          dst[1] = make_uint4(pack_bf162(r[m][8], r[m][9]), pack_bf162(r[m][10], r[m][11]),
                              pack_bf162(r[m][12], r[m][13]), pack_bf162(r[m][14], r[m][15]));
        }
      }
    }
    {
      const int pos = min((cidx + 1) * kChunk, w.len);
      float* ckdst = nullptr;
      if (ck < w.ck_end && p.ckpt_pos[ck] == pos) {
        ckdst = p.ckpts + (static_cast<int64_t>(ck) * p.H + w.h) * (kHeadDim * kHeadDim);
        ++ck;
      }
      float* fin = (n + 1 == n_chunks) ? w.s_out : nullptr;
      const int i = quarter * 32 + lane;
      uint8_t* dst = sm + SM_S + hcol * 16384;
      float r[4][16];
#pragma unroll
      for (int m = 0; m < 4; ++m) tmem_ld16(tmem + tl + kTS + hcol * 64 + m * 16, r[m]);
      tmem_wait_ld();
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int c = hcol * 64 + m * 16;
        st4(dst + sw128(i, 32 * m), pack_half2(r[m][0], r[m][1]), pack_half2(r[m][2], r[m][3]),
            pack_half2(r[m][4], r[m][5]), pack_half2(r[m][6], r[m][7]));
        st4(dst + sw128(i, 32 * m + 16), pack_half2(r[m][8], r[m][9]), pack_half2(r[m][10], r[m][11]),
            pack_half2(r[m][12], r[m][13]), pack_half2(r[m][14], r[m][15]));
        if (ckdst) {
          float4* d4 = reinterpret_cast<float4*>(ckdst + i * kHeadDim + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_float4(r[m][4 * e], r[m][4 * e + 1], r[m][4 * e + 2], r[m][4 * e + 3]);
        }
        if (fin) {
          float4* d4 = reinterpret_cast<float4*>(fin + i * kHeadDim + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_float4(r[m][4 * e], r[m][4 * e + 1], r[m][4 * e + 2], r[m][4 * e + 3]);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctrl[1]) { aborted = true; break; }
  }

  if (aborted) {
    // Let copies and MMAs still in flight land before TMEM is released (bounded).
    if (tid == 0) {
      report_status(p.status, 6 /* KDA_ERR_TIMEOUT */);
      for (int b = 0; b < kNumBars; ++b) { mbar_wait(&bars[b], 0, 1u << 20); mbar_wait(&bars[b], 1, 1u << 20); }
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, bool is_f32, int H, int64_t T) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = is_f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {kHeadDim * esz, static_cast<cuuint64_t>(H) * kHeadDim * esz};
  cuuint32_t box[3] = {is_f32 ? 128u : 64u, 1u, 64u};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, is_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  is_f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int n_seq, int H, int64_t total_tokens, int n_segments, int num_sms) {
  return split_layout(n_seq, H, total_tokens, n_segments, num_sms).bytes;
}

cudaError_t launch_prefill(const PrefillArgs& a, int num_sms) {
  KParams p;
  memset(&p, 0, sizeof(p));
  const int64_t T = a.total_tokens;
  if (T > 0) {
    if (!make_map(&p.tm_q, a.q, false, a.H, T) || !make_map(&p.tm_k, a.k, false, a.H, T) ||
        !make_map(&p.tm_v, a.v, false, a.H, T) || !make_map(&p.tm_g, a.g, true, a.H, T))
      return cudaErrorInvalidValue;
  }
  p.beta = a.beta; p.S_in = a.S_in; p.cu = a.cu_seqlens; p.ckpt_off = a.ckpt_off; p.ckpt_pos = a.ckpt_pos;
  p.o = static_cast<__nv_bfloat16*>(a.o); p.S_out = a.S_out; p.ckpts = a.ckpts; p.status = a.status;
  p.n_seq = a.n_seq; p.H = a.H; p.total_tokens = T; p.n_ckpt = a.n_ckpt;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const SplitLayout L = split_layout(a.n_seq, a.H, T, a.n_segments, num_sms);
  if (L.extra == 0) {
    // one CTA per (sequence, head), whole sequence
    prefill_kernel<<<dim3(static_cast<unsigned>(a.n_seq), static_cast<unsigned>(a.H)), kThreads, kSmemAlloc,
                     a.stream>>>(p);
    return cudaGetLastError();
  }
  // sequence split: plan, pass 1 (first segments + (S~, M) of middle segments), scan, pass 3
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  cudaError_t e = launch_split_plan(a, L, num_sms);
  if (e != cudaSuccess) return e;
  p.slots = reinterpret_cast<float*>(ws + L.off_slots);
  p.items = reinterpret_cast<const int4*>(ws + L.off_items1);
  p.item_count = reinterpret_cast<const int*>(ws);
  prefill_kernel<<<dim3(static_cast<unsigned>(L.max1), static_cast<unsigned>(a.H)), kThreads, kSmemAlloc,
                   a.stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_split_scan(a, L)) != cudaSuccess) return e;
  p.items = reinterpret_cast<const int4*>(ws + L.off_items3);
  p.item_count = reinterpret_cast<const int*>(ws) + 1;
  prefill_kernel<<<dim3(static_cast<unsigned>(L.max3), static_cast<unsigned>(a.H)), kThreads, kSmemAlloc,
                   a.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
