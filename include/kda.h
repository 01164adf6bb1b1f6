/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * The operation (per head; "Kimi K3.1 Pro 架构完全拆解", section 3.1):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t,          alpha_t = exp(g_t) per d_k channel
 *
 * with S_t a d_k x d_v matrix (row = d_k channel, column = d_v channel) and g the
 * natural-log decay, bounded below by g_min = -5 (section 3.2 of the same page).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - d_k = d_v = d = 128 (KDA_HEAD_DIM); any other d returns KDA_ERR_UNSUPPORTED.
 *  - Every pointer argument is a DEVICE pointer on the current CUDA device, owned by
 *    the caller.  The library allocates no device memory and keeps no state between
 *    calls, with two exceptions described at those calls: kda_prefill_noalloc's fixed
 *    scratch array, and the streams and events kda_prefill_host keeps per device.  Tensor
 *    pointers must be 16-byte aligned (KDA_ERR_ALIGNMENT otherwise).
 *  - Calls are asynchronous on `stream`: they validate what the host can see, enqueue
 *    kernels and return.  A non-KDA_OK return means nothing was enqueued (except
 *    KDA_ERR_CUDA, returned when a launch itself failed).
 *  - `dev_status` (optional, device int): kernels that find a problem only visible on
 *    the device (inconsistent cu_seqlens / checkpoint contents, an n_commit out of
 *    range, a bounded wait that ran out) write a kda_status code there, first error
 *    wins; the work unit concerned is skipped.  The library never clears it: zero it
 *    before the call and read it after synchronising.  NULL disables the report.
 *  - Element types: kda_bf16 is the IEEE bfloat16 bit pattern; float is IEEE fp32.
 *  - Input ranges the tensor-core path relies on: q and k L2-normalised per (token,
 *    head) (the model normalises them before the recurrence), |v| well below 6e4, and
 *    g in [-5, 0].  Outside them results may overflow to inf/NaN.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent sizes */
  KDA_ERR_UNSUPPORTED = 2,   /* d != 128, n_tok outside [1, 4], no sm_103a device */
  KDA_ERR_ALIGNMENT = 3,     /* a tensor pointer not 16-byte aligned */
  KDA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
  KDA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  KDA_ERR_TIMEOUT = 6,       /* device-side: a bounded wait ran out (written to dev_status) */
  KDA_ERR_DEVICE_CHECK = 7   /* device-side: argument contents inconsistent (dev_status) */
} kda_status;

#define KDA_HEAD_DIM 128
#define KDA_CHUNK 64
#define KDA_MAX_DECODE_TOKENS 4

/* Human-readable name of a status code (static string, never NULL). */
const char* kda_status_string(int status);

/* ABI version of this library (major * 100 + minor). */
int kda_version(void);

/*
 * kda_decode -- one decode step, or a verify step of up to 4 tokens, per (sequence, head).
 *
 * Source: "Kimi K3 ... 服務性能" (SemiAnalysis translation) section 6: the decode kernel
 * follows the delta-rule form
 *     X = Diag(alpha_t) S;  u_t = beta_t (v_t - X^T k_t);  S = X + k_t u_t^T;  o_t = S^T q_t.
 * Verify ("Kimi K3.1 Pro 架构完全拆解" 3.4; "部署 Kimi K3 ..." section 4): the n_tok
 * cached projected inputs are replayed on-chip and only the state after the accepted
 * prefix is written back.
 *
 *   q, k, v    [B, n_tok, H, d]  bf16       g  [B, n_tok, H, d] fp32    beta [B, n_tok, H] fp32
 *   S_state    [B, H, d, d]      fp32, read, then overwritten in place with the state
 *                                after n_commit[b] tokens (left untouched when 0)
 *   n_commit   [B] int32 in [0, n_tok], or NULL for n_tok; an entry out of range leaves
 *              that sequence's state untouched and reports KDA_ERR_DEVICE_CHECK
 *   o          [B, n_tok, H, d]  fp32: outputs of all n_tok tokens
 *   1 <= n_tok <= 4.  B or H == 0 is a no-op.
 */
kda_status kda_decode(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g, const float* beta,
                      float* S_state, const int32_t* n_commit, float* o, int B, int n_tok, int H, int d,
                      int* dev_status, cudaStream_t stream);

/*
 * kda_prefill_workspace_size -- bytes of device workspace kda_prefill needs for the
 * same (n_seq, H, d, total_tokens, n_segments).  0 means no workspace is needed.
 */
size_t kda_prefill_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int n_segments);

/*
 * kda_prefill -- chunkwise prefill over packed variable-length sequences.
 *
 * Sources: the chunk-level matrix form of "Kimi K3 ... 服務性能" section 6 (FlashKDA
 * algorithm: prep a = exp(cumsum g), K_decay, Q_decay, K_inv, K_restore, L, INV, M_qk;
 * recurrence U = INV Diag(beta)(V - K_decay S), O = Q_decay S + M_qk U,
 * S <- Diag(a_last) S + K_restore^T U) with chunk length C = 64; the sequence split of
 * "部署 Kimi K3 ..." sections 1.2 and 2 (per-segment transition M and zero-start
 * state S~, entry states by an associative prefix scan S = S~ + M S_in); state
 * checkpoints at requested positions (same page, section 3.2).
 *
 *   q, k, v      [total_tokens, H, d]  bf16
 *   g            [total_tokens, H, d]  fp32      beta [total_tokens, H] fp32
 *   S_in         [n_seq, H, d, d] fp32 initial states (read only), or NULL for zeros
 *   cu_seqlens   [n_seq + 1] int32: sequence i owns packed rows [cu[i], cu[i+1]);
 *                cu[0] = 0, non-decreasing, cu[n_seq] = total_tokens (checked on device)
 *   ckpt_off     [n_seq + 1] int32 CSR offsets into ckpt_pos (or NULL: no checkpoints)
 *   ckpt_pos     [n_ckpt] int32: for sequence i, positions ckpt_pos[ckpt_off[i] ..
 *                ckpt_off[i+1]) strictly increasing in (0, len_i], each a multiple of
 *                64 or equal to len_i.  A position p means "the state after the
 *                sequence's p-th token of this call".  Violations: KDA_ERR_DEVICE_CHECK.
 *   o            [total_tokens, H, d] bf16 (round to nearest even from fp32)
 *   S_out        [n_seq, H, d, d] fp32 final states, or NULL
 *   ckpts        [n_ckpt, H, d, d] fp32, slot j = checkpoint ckpt_pos[j] (write only)
 *   n_segments   0: the library splits long sequences by its own rule (a function of the
 *                sequence's own length, H and the SM count only, so a sequence gives the
 *                same bits packed or alone): the count with the least chain time when the
 *                two passes run in waves of one CTA per SM, never two segments (they only
 *                run one after the other); k >= 1: split every sequence into
 *                min(k, its chunk count) segments.
 *   workspace    device buffer of kda_prefill_workspace_size(...) bytes (may be NULL
 *                when that is 0), 256-byte aligned.
 * Output rows of other sequences, and padding, are never written.
 */
kda_status kda_prefill(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g, const float* beta,
                       const float* S_in, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                       const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt, kda_bf16* o,
                       float* S_out, float* ckpts, int H, int d, int n_segments, void* workspace,
                       size_t workspace_bytes, int* dev_status, cudaStream_t stream);


/*
 * kda_prefill_gated -- kda_prefill with the layer's output stage fused into the output
 * write: instead of o, it writes
 *
 *     y[t, h, :] = sigmoid(gate[t, h, :]) * norm_weight * o~ / sqrt(mean_c(o~[c]^2) + eps)
 *
 * where o~ = S_t^T q_t is the recurrent output kda_prefill would write (kept in fp32, not
 * rounded, before the normalisation).  Source: "Kimi K3.1 Pro 架构完全拆解" section 3.3
 * (full-rank output gate): y_t = W_o [Sigmoid(W_g x_t) * RMSNorm(o~_t)]; this computes the
 * bracket, with the gate logits W_g x_t supplied by the caller.  The page names RMSNorm
 * without its weight or epsilon: norm_weight is a per-channel weight shared by all heads
 * and eps is added to the mean square.
 *
 *   gate         [total_tokens, H, d] bf16 gate logits (read only)
 *   norm_weight  [d] fp32, or NULL for ones
 *   eps          >= 0 and finite (else KDA_ERR_INVALID_ARG)
 *   y            [total_tokens, H, d] bf16 (round to nearest even), in place of o
 * Every other argument, the state outputs and the errors are those of kda_prefill.
 */
kda_status kda_prefill_gated(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const kda_bf16* gate, const float* norm_weight, float eps,
                             const float* S_in, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                             const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt, kda_bf16* y,
                             float* S_out, float* ckpts, int H, int d, int n_segments, void* workspace,
                             size_t workspace_bytes, int* dev_status, cudaStream_t stream);

/*
 * Paged state.  "部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景" section 3: the
 * prefix cache keeps each head's state as one 64 KiB block, snapshots it at hash-aligned
 * positions, and a hit resumes from the cached snapshot, which other requests may share;
 * "Kimi K3.1 Pro 架构完全拆解" section 8: the states live in one unified pool.  The paged
 * entry points address every state through such a pool:
 *
 *   state_pool   [n_pages, d, d] fp32, 16-byte aligned: page p holds one head's state
 *                (row = d_k), n_pages <= 2^31 - 1
 *   page tables  device int32; an entry is a page index in [0, n_pages) or -1 = none (a
 *                zero entry state, or nothing written).  Another value is a device error
 *                (KDA_ERR_DEVICE_CHECK).
 *
 * Copy on hit: a call writes each page at most once and never writes a page that it reads,
 * except that a unit (one sequence and head) may write its final or committed state back
 * to its own entry page (in place).  Before the work runs, the library checks this over
 * the tables on the device, with an owner table in the caller's workspace (4 bytes per
 * page): on a violation it reports KDA_ERR_DEVICE_CHECK and the call writes nothing (no
 * outputs, no states).  A shared snapshot therefore stays bit-unchanged: a continuation
 * names it as its entry page and a fresh page for its result.
 */

/*
 * kda_prefill_paged -- kda_prefill / kda_prefill_gated with the states in a page pool.
 *
 *   s_in_page    [n_seq * H] (entry seq * H + h): page of the entry state, -1 = zeros;
 *                NULL = all zeros
 *   s_out_page   [n_seq * H]: page receiving the final state, -1 = not written; NULL = none
 *   ckpt_page    [n_ckpt * H] (entry j * H + h, j in ckpt_pos order): page receiving
 *                checkpoint j of head h, -1 = not written; required when n_ckpt > 0
 *   gate         NULL: write o as kda_prefill does; otherwise gate / norm_weight / eps and
 *                the output y are those of kda_prefill_gated
 *   workspace    kda_prefill_paged_workspace_size(...) bytes, 256-byte aligned (never 0:
 *                the page check always runs)
 * Every other argument, the checkpoint positions and the errors are those of kda_prefill.
 */
size_t kda_prefill_paged_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int n_segments,
                                        int64_t n_pages);
kda_status kda_prefill_paged(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const kda_bf16* gate, const float* norm_weight, float eps,
                             float* state_pool, int64_t n_pages, const int32_t* s_in_page,
                             const int32_t* s_out_page, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens,
                             const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt,
                             const int32_t* ckpt_page, kda_bf16* o, int H, int d, int n_segments, void* workspace,
                             size_t workspace_bytes, int* dev_status, cudaStream_t stream);

/*
 * kda_decode_paged -- kda_decode with the states in a page pool.
 *
 *   s_in_page    [B * H] (entry b * H + h): page the state is read from, -1 = zeros
 *   s_out_page   [B * H]: page receiving the state after n_commit[b] tokens, -1 = not
 *                written; NULL = in place (s_in_page).  A destination other than the
 *                source always receives it, the entry state itself when n_commit[b] = 0
 *                (speculative decode from a shared snapshot: the snapshot stays unchanged).
 *   workspace    kda_decode_paged_workspace_size(n_pages) bytes, 256-byte aligned
 * Every other argument and the errors are those of kda_decode.
 */
size_t kda_decode_paged_workspace_size(int64_t n_pages);
kda_status kda_decode_paged(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                            const float* beta, float* state_pool, int64_t n_pages, const int32_t* s_in_page,
                            const int32_t* s_out_page, const int32_t* n_commit, float* o, int B, int n_tok, int H,
                            int d, void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream);

/*
 * kda_decode_fused -- a decode / verify step from the layer's projected inputs, with its
 * front end (and optionally its output stage) in the same kernel.
 *
 * "Kimi K3.1 Pro 架构完全拆解" section 3.4: for speculative decoding only the projected
 * inputs are cached, and one fused kernel replays the accepted tokens (short convolution,
 * input normalisation, gating, the recurrence, output normalisation) and writes the state
 * back.  The steps ("Kimi K3 ... 服務性能" section 7; K3.1 page section 3.2), per (sequence b,
 * token i, head h), channel c:
 *     x~_i = sum_{j < W} conv_w[s, h, c, j] x_{i-j}     (x = qp, kp, vp for s = 0, 1, 2; inputs
 *                                                        before token 0 come from conv_cache)
 *     optionally x~ <- x~ Sigmoid(x~) (SiLU, conv_act = 1)
 *     q = q~ / ||q~||,  k = k~ / ||k~||  (over the head's d channels; a zero vector stays 0)
 *     alpha = exp(g_min Sigmoid(exp(a_log[h]) z)),  beta = Sigmoid(b)
 *     then the recurrence, outputs and commit of kda_decode, and, with gate != NULL, the
 *     output stage y = Sigmoid(gate) norm_weight o / sqrt(mean(o^2) + eps) in place of o.
 * The pages print neither the convolution width, an activation after it, nor beta's
 * activation: those are the readings above (W and the activation are arguments).
 *
 *   qp, kp, vp   [B, n_tok, H, d] bf16 projected inputs
 *   conv_w       [3, H, d, W] fp32 filters (q, k, v), 1 <= W <= 4
 *   conv_cache   [B, H, 3, W - 1, d] fp32: the W - 1 projected inputs before this step,
 *                oldest first; on return those before token n_commit[b] (unchanged when
 *                n_commit[b] = 0).  May be NULL when W = 1.
 *   conv_act     0: none, 1: SiLU
 *   z            [B, n_tok, H, d] fp32 decay-gate pre-activations;  a_log [H] fp32
 *   g_min        the decay's lower bound, finite and < 0 (-5 on the pages)
 *   b            [B, n_tok, H] fp32 beta logits
 *   gate         [B, n_tok, H, d] bf16 output-gate logits, or NULL (o as kda_decode)
 *   norm_weight  [d] fp32 or NULL (ones);  eps >= 0 and finite
 *   S_state, n_commit, o, B, n_tok, H, d, dev_status, stream: as kda_decode
 */
kda_status kda_decode_fused(const kda_bf16* qp, const kda_bf16* kp, const kda_bf16* vp, const float* conv_w,
                            float* conv_cache, int conv_width, int conv_act, const float* z, const float* a_log,
                            float g_min, const float* b, const kda_bf16* gate, const float* norm_weight, float eps,
                            float* S_state, const int32_t* n_commit, float* o, int B, int n_tok, int H, int d,
                            int* dev_status, cudaStream_t stream);

/*
 * kda_prefill_host -- kda_prefill from HOST buffers, with the transfers overlapped.
 *
 * The inputs and outputs live in host memory (pin them: cudaMemcpyAsync from pageable memory
 * is not asynchronous).  The call cuts the packed token stream into blocks (borders on the
 * chunk grid of the sequence they cut: a multiple of 64 tokens from its start) and pipelines
 * them: block j + 1's rows of q, k, v, g, beta are uploaded while block j is computed on
 * `stream` and block j - 1's rows of o are downloaded; the final states follow the last
 * block.  Each block is an ordinary kda_prefill whose sequences start from the running
 * states, updated in place in the workspace, so a sequence cut into blocks goes through
 * exactly the chunks and fp32 states of one kda_prefill call (same bits whenever neither
 * path splits a sequence into segments).  Not on the pages: an executor for callers whose
 * tensors start on the host ("部署 Kimi K3 ..." section 1.1 motivates overlapping the
 * transfers with the work).
 *
 *   q, k, v, g, beta, S_in (or NULL: zeros), cu_seqlens, o, S_out: as kda_prefill, in HOST
 *                memory; cu_seqlens is read on the host to plan the blocks (a bad packing is
 *                KDA_ERR_INVALID_ARG); no checkpoints
 *   block_tokens 0: the library's choice (total_tokens / 8 rounded to 64, at least 1024);
 *                else a multiple of 64.  At most 64 blocks (KDA_ERR_UNSUPPORTED beyond).
 *   workspace    DEVICE memory of kda_prefill_host_workspace_size(...) bytes, 256-byte
 *                aligned: device copies of the inputs, o and the states
 * The call enqueues the work and returns: `stream` is made to wait for the last transfer, so
 * synchronising it (or an event recorded on it) means o and S_out are in host memory.  The
 * host buffers must stay valid until then.  The transfers run on two streams of the library's
 * own, created with a set of events by the first call on each device and kept for the life
 * of the process (not after cudaDeviceReset: do not call it on a device after a reset).
 * Calls from several host threads are safe; their transfers share those streams and run in
 * call order.
 */
size_t kda_prefill_host_workspace_size(int n_seq, int H, int d, int64_t total_tokens, int64_t block_tokens);
kda_status kda_prefill_host(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                            const float* beta, const float* S_in, const int32_t* cu_seqlens, int n_seq,
                            int64_t total_tokens, kda_bf16* o, float* S_out, int H, int d, int64_t block_tokens,
                            void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream);
/* The block borders kda_prefill_host would use (host only, no CUDA call): writes up to
 * max_borders of the n + 1 borders 0 = b_0 < ... < b_n = total_tokens and returns n (0 for
 * no sequences), or -1 for a bad packing or block size, or more than 64 blocks. */
int kda_prefill_host_blocks(const int32_t* cu_seqlens, int n_seq, int64_t total_tokens, int64_t block_tokens,
                            int64_t* borders, int max_borders);

/*
 * Cross-device sequence split (KCP).  "部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra
 * 全景" section 2: a sequence's tokens are split over ranks in order; each rank summarises
 * its token range by the pair (M, S~) -- the cumulative transition
 * M = prod_t (I - beta_t k_t k_t^T) Diag(alpha_t) and the state S~ the range produces from a
 * zero entry state -- so that its exit state for an entry state S is S~ + M S.  The ranks
 * all-gather their pairs (a fixed 2 x 64 KiB per head, whatever the token count), each
 * folds the pairs of the ranks before it onto the sequence's entry state, and runs its own
 * range from the resulting true entry state with kda_prefill.  These two calls are the
 * device parts; the exchange is the caller's (the Python binding's kcp module does it over
 * torch.distributed).
 *
 * kda_prefill_pairs -- (M, S~) of every (sequence, head) over that sequence's rows.
 *   q, k, v, g, beta, cu_seqlens, n_seq, total_tokens, H, d, dev_status: as kda_prefill
 *   M, S_tilde   [n_seq, H, d, d] fp32 each (write only), row = d_k.  A sequence with no
 *                rows gets M = I and S~ = 0.
 * No workspace.  One chain per (sequence, head) for each of the two, on the prefill kernel.
 */
kda_status kda_prefill_pairs(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                             const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t total_tokens, float* M,
                             float* S_tilde, int H, int d, int* dev_status, cudaStream_t stream);

/*
 * kda_combine_pairs -- the entry state after n_pairs ranges, per (sequence, head):
 *     E = S_in;  for r = 0 .. n_pairs - 1:  E = S~_r + M_r E;  entry = E
 * (same page, section 2: the local sequential combine of the preceding ranks' pairs).
 *   M, S_tilde   [n_pairs, n_seq, H, d, d] fp32 (may be NULL when n_pairs = 0)
 *   S_in         [n_seq, H, d, d] fp32, or NULL for zeros
 *   entry        [n_seq, H, d, d] fp32 (write only; must not overlap the inputs)
 * fp32 arithmetic; n_pairs = 0 copies S_in.
 */
kda_status kda_combine_pairs(const float* M, const float* S_tilde, int n_pairs, const float* S_in, float* entry,
                             int n_seq, int H, int d, cudaStream_t stream);

/*
 * kda_debug_stall_next_prefill -- test hook for the bounded waits (no counterpart on the
 * pages).  The next prefill launch of this process runs a test instance of the kernel
 * whose prep warps withhold their first hand-off of chunk `chunk` (counted within each
 * work item) and whose waits give up after 4096 polls.  The recurrence's wait for that
 * hand-off then runs out: both warp groups leave their loops together, the copies and
 * tensor-core products still in flight land (bounded), the tensor memory is released, and
 * KDA_ERR_TIMEOUT is written to dev_status; that call's outputs are undefined.  Nothing
 * faults or traps and the CUDA context stays usable.  Host side only; one-shot.  (The
 * production instance's waits give up after 2^26 polls.)
 */
void kda_debug_stall_next_prefill(int chunk);

/*
 * kda_prefill_noalloc -- kda_prefill for callers that cannot allocate device memory.
 *
 * This entry point has no counterpart on the pages; it exists for the library's users.
 * Some callers have no way to provide the workspace kda_prefill may ask for: a plugin
 * inside a serving framework that owns all device memory and passes the plugin only its
 * input and output tensors, or a path where cudaMalloc (which can synchronise the device)
 * is not allowed.  This variant takes that scratch from a fixed array inside the library
 * (KDA_NOALLOC_SCRATCH_BYTES = 32 MiB of device memory, held on every GPU where the library
 * is loaded until the process exits) and otherwise behaves exactly like kda_prefill, with
 * the same arguments minus workspace / workspace_bytes.  It allocates nothing.
 *
 *  - A problem whose kda_prefill_workspace_size(...) exceeds KDA_NOALLOC_SCRATCH_BYTES is
 *    rejected with KDA_ERR_WORKSPACE before anything is enqueued (the 1M-token, 8-head
 *    prefill with the library's own split needs about 31.5 MB on a 152-SM GB300, and fits
 *    up to 167 SMs; split counts forced through n_segments can need more).
 *  - Set-up: the first call on each device, made while that device is current and whatever
 *    the problem (an empty one, n_seq = 0, will do), looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it for the rest of the process.  Under the CUDA
 *    runtime's default lazy module loading, that first call is also when the driver loads
 *    the library code holding the array onto the device and reserves its 32 MiB.  Make the
 *    first call during the caller's own set-up: before a framework claims the device's
 *    memory, and before any stream capture on the device.  A failed look-up returns
 *    KDA_ERR_CUDA and leaves no error pending in the runtime.
 *  - The cached address does not survive cudaDeviceReset: after a reset of a device, do not
 *    call kda_prefill_noalloc on it again in the same process.
 *  - Every call shares the one array and it keeps the previous call's contents (no part of
 *    it needs to start at zero: each call writes every entry it reads).  Calls whose work
 *    may overlap on the GPU -- on different streams, or from several host threads without
 *    ordering -- race on it: order them on one stream.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
kda_status kda_prefill_noalloc(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const float* g,
                               const float* beta, const float* S_in, const int32_t* cu_seqlens, int n_seq,
                               int64_t total_tokens, const int32_t* ckpt_off, const int32_t* ckpt_pos, int64_t n_ckpt,
                               kda_bf16* o, float* S_out, float* ckpts, int H, int d, int n_segments,
                               int* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
