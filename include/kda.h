/*
 * kda.h -- C ABI of libkda: Kimi Delta Attention (KDA) on one GB300 GPU.
 *
 * The operation (mhpq.cn/news/56770, section "KDA 到底在算什么"): per head, a
 * dk x dv state S is decayed, corrected and written once per token,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 *
 * alpha_t being a dk-vector (one retention per key channel, i.e. per row of
 * S) and beta_t a scalar.  The retention comes from the lower-bounded gate
 * (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section
 * "下界衰减：一个纯粹为硬件让步的算法改动"):
 *
 *     log alpha = gmin * sigmoid(z),   gmin = -5,
 *
 * with the per-head scale e^A of that section already folded into z by the
 * caller.  q and k are L2-normalised inside the library as
 * x / sqrt(sum x^2 + 1e-6) (mhpq.cn/news/56770, the Q/K preprocessing
 * paragraph; the page gives no epsilon, 1e-6 is this library's choice).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, contiguous, packed over a variable-length batch):
 *     q, k        [T_tot, H, dk]   io dtype (fp32 or bf16)
 *     v, out      [T_tot, H, dv]   io dtype
 *     z           [T_tot, H, dk]   fp32 gate logits
 *     beta        [T_tot, H]       fp32 write strength, used as given
 *     state       [N, H, dk, dv]   fp32, row = key channel
 *     cu_seqlens  [N + 1]          int32 offsets, cu_seqlens[0] = 0,
 *                                  non-decreasing, cu_seqlens[N] = T_tot
 * Pointers marked "device" must point to device memory of the current
 * device; every such buffer is owned by the caller.  The library allocates
 * no memory of its own besides one static device error word, never frees,
 * and never synchronises except in kda_get_device_error().
 *
 * Execution: work is enqueued asynchronously on `stream` (NULL = legacy
 * default stream).  Calls are thread-safe when they use distinct streams
 * and do not share output buffers.
 *
 * Errors: argument problems the host can see (NULL required pointer,
 * unsupported size or dtype, a host copy of cu_seqlens that is not
 * monotone or disagrees with total_tokens) return KDA_ERR_INVALID_ARGUMENT
 * and enqueue nothing.  A failed launch returns KDA_ERR_CUDA.  Problems only
 * the device can see (device cu_seqlens out of range or non-monotone) skip
 * the offending work item and set the device error word, which
 * kda_get_device_error() reports.
 *
 * Supported sizes: dk, dv in {32, 64, 128}; H >= 1; N >= 1; T_tot >= 0.
 * Zero-length sequences are legal: their final state equals their initial
 * state.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream, declared here so that this header
 * does not need the CUDA headers. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARGUMENT = 1, /* rejected on the host, nothing enqueued   */
  KDA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (size/dtype)   */
  KDA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed     */
  KDA_ERR_TIMEOUT = 4,          /* a bounded device-side wait expired       */
  KDA_ERR_DEVICE_CHECK = 5      /* a device-side argument check failed      */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Shapes and options of one call. */
typedef struct {
  int32_t num_seqs;     /* N: sequences (prefill) or live requests (decode) */
  int32_t total_tokens; /* T_tot: packed tokens; equals N for decode        */
  int32_t num_heads;    /* H                                                */
  int32_t dk;           /* key / query channels per head                    */
  int32_t dv;           /* value channels per head                          */
  int32_t io_dtype;     /* kda_dtype_t of q, k, v and out                   */
  /* Optional HOST copy of cu_seqlens ([N + 1] int32), used only to plan
   * the launch (longest-first order, splitting long sequences across SMs).
   * May be NULL; then the plan assumes nothing about lengths.  When given
   * it is checked and must equal the device copy. */
  const int32_t* cu_seqlens_host;
  /* Optional device scratch for splitting long sequences across SMs in
   * kda_chunk_fwd (see kda_chunk_fwd_workspace_size), 256-byte aligned.
   * NULL / 0 disables the split; an area smaller than the size query asks
   * for limits the split to plans that fit in it.  Results are the same
   * (within rounding) either way. */
  void* workspace;
  size_t workspace_bytes;
  /* Optional per-head log-scale A of the gate, DEVICE [H] fp32: the gate is
   * g = -5 sigmoid(e^{A_h} z) (blog.higcp.com "猜想：K3 可能是最适合 TPU 的
   * MoE 架构", section "下界衰减"; A is a learnable per-head log-scale).  NULL
   * means A = 0, i.e. g = -5 sigmoid(z), with any scale already folded into z.
   * Read by every call that takes z. */
  const float* a_log;
  /* Optional state checkpoints of the prefill calls (kda_chunk_fwd,
   * kda_recurrent_fwd, kda_chunk_fwd_noalloc): with checkpoint_every = E > 0
   * (a multiple of 64), checkpoint j of sequence n (j = 1 .. floor(len_n / E))
   * is the state after its first j E tokens, written fp32 [dk][dv] per head to
   * checkpoints[(checkpoint_offsets[n] + j - 1) * H + h].  checkpoint_offsets
   * is a DEVICE [N + 1] int32 exclusive prefix sum of floor(len_n / E); both
   * buffers are the caller's.  E = 0 writes none (the pointers are ignored).
   * The pages place such states at fixed token offsets so that a prefix can
   * be resumed (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
   * "三条容易被忽略的代价" (2): states kept at hash-block ends). */
  float* checkpoints;
  const int32_t* checkpoint_offsets;
  int32_t checkpoint_every;
  /* 0: one gate logit per key channel, z [T_tot, H, dk] (KDA).  1: one per
   * head, z [T_tot, H] (decode: [N, H]), the same retention for every row of
   * S -- the scalar-alpha case, which the pages identify with Gated DeltaNet
   * (mhpq.cn/news/56770, section "KDA 到底在算什么": Gated DeltaNet has one
   * scalar alpha_t per token where KDA has one per key channel).  Every call
   * that takes z honours it. */
  int32_t gate_per_head;
} kda_desc_t;

/*
 * kda_chunk_fwd -- prefill over a packed variable-length batch.
 *
 * Chunkwise evaluation of the recurrence above (mhpq.cn/news/56770, section
 * "KDA 到底在算什么"; the chunked-with-reciprocal-decay form of
 * blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减").
 * For every sequence n and head h, the state starts at initial_state[n, h]
 * (zeros when initial_state is NULL), runs over the tokens
 * cu_seqlens[n] .. cu_seqlens[n+1]-1 writing out[t, h, :] = S_t^T q_t, and
 * is stored to final_state[n, h] when final_state is not NULL.
 *
 *   q, k, v, z, beta   device, read-only, layouts above
 *   initial_state      device, [N, H, dk, dv] fp32, or NULL for zeros
 *   cu_seqlens         device, [N + 1] int32
 *   out                device, [T_tot, H, dv] io dtype, written
 *   final_state        device, [N, H, dk, dv] fp32, written, or NULL;
 *                      may alias initial_state exactly (in-place prefix
 *                      caching): each (n, h) state is read before it is
 *                      written.  out must not alias any input.
 *
 * bf16 inputs run the tensor-core path (dk = dv = 128) or the CUDA-core
 * path (other sizes); fp32 inputs always run the fp32 CUDA-core path.
 *
 * Range limit of the tensor-core path: its dense products take fp16
 * operands (11-bit significand, largest magnitude 65504), made from the
 * state entering each 64-token chunk, the corrections v - S^T k+ and the
 * pseudo-values U.  A bf16 v or an fp32 state can exceed that range.  When
 * any such operand
 * reaches 65504 in magnitude the call's outputs are not valid and the
 * kernel sets KDA_ERR_DEVICE_CHECK in the device error word (read it with
 * kda_get_device_error); the following calls are unaffected.  Data of that
 * magnitude must go through kda_recurrent_fwd (fp32 throughout) or fp32
 * inputs.
 */
kda_status_t kda_chunk_fwd(const kda_desc_t* desc, const void* q, const void* k,
                           const void* v, const float* z, const float* beta,
                           const float* initial_state, const int32_t* cu_seqlens,
                           void* out, float* final_state, kda_stream_t stream);

/* Bytes of device scratch that let kda_chunk_fwd split long sequences
 * across SMs for this descriptor (0 when no split would be planned).
 * Needs desc->cu_seqlens_host.  Returns KDA_ERR_INVALID_ARGUMENT on a bad
 * descriptor. */
kda_status_t kda_chunk_fwd_workspace_size(const kda_desc_t* desc, size_t* bytes);

/*
 * kda_recurrent_fwd -- the same operation and arguments as kda_chunk_fwd,
 * evaluated token by token (the recurrence exactly as written on
 * mhpq.cn/news/56770, section "KDA 到底在算什么") with the fp32 state held in
 * registers.  It is the GPU reference the chunked path is compared with;
 * it is slower on long sequences.  workspace fields are ignored.
 */
kda_status_t kda_recurrent_fwd(const kda_desc_t* desc, const void* q, const void* k,
                               const void* v, const float* z, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens,
                               void* out, float* final_state, kda_stream_t stream);

/*
 * kda_decode_step -- one new token for each of N live requests, updating
 * their states in place (the decode regime: blog.higcp.com
 * "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "三条容易被忽略的代价" (3),
 * where state traffic dominates at large batch).
 *
 *   desc               num_seqs = total_tokens = N (requests)
 *   q, k               device, [N, H, dk] io dtype
 *   v                  device, [N, H, dv] io dtype
 *   z                  device, [N, H, dk] fp32
 *   beta               device, [N, H] fp32
 *   state              device, [N, H, dk, dv] fp32, read and overwritten
 *                      with S_t
 *   out                device, [N, H, dv] io dtype, written with S_t^T q_t
 * desc->cu_seqlens_host and workspace are ignored.
 */
kda_status_t kda_decode_step(const kda_desc_t* desc, const void* q, const void* k,
                             const void* v, const float* z, const float* beta,
                             float* state, void* out, kda_stream_t stream);

/*
 * Speculative decoding without per-position state snapshots.  The pages
 * (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "三条容易被
 * 忽略的代价" (1)) note that the in-place state update cannot be rolled back
 * when verification rejects drafted tokens, that a snapshot per draft
 * position would multiply state traffic, and that K3 instead keeps the
 * window's inputs and replays the accepted tokens to rebuild the state.
 *
 * kda_decode_window -- outputs of W draft tokens per request from the
 * committed states, which are read and NOT changed: token i of request b
 * sees the state after the committed tokens and drafts 0 .. i.
 *
 *   desc               num_seqs = B requests, total_tokens = B * W
 *   window             W >= 1 draft tokens per request
 *   q, k               device, [B * W, H, dk] io dtype (request-major: row
 *                      b * W + i is draft i of request b)
 *   v                  device, [B * W, H, dv] io dtype
 *   z                  device, [B * W, H, dk] fp32
 *   beta               device, [B * W, H] fp32
 *   state              device, [B, H, dk, dv] fp32, read only
 *   out                device, [B * W, H, dv] io dtype, written
 *
 * kda_decode_replay -- after verification: applies the first accept_len[b]
 * drafts of request b (0 .. W; the same cached inputs as the window call) to
 * its state, which is written once (state traffic: one read and one write
 * per step instead of one snapshot per draft position).  accept_len is a
 * DEVICE [B] int32; a value outside 0 .. W leaves that request's state
 * unchanged and sets the device error word (KDA_ERR_DEVICE_CHECK).
 *
 * Both honour desc->a_log; cu_seqlens_host, workspace and the checkpoint
 * fields are ignored.  Host-side argument errors return
 * KDA_ERR_INVALID_ARGUMENT and enqueue nothing.
 */
kda_status_t kda_decode_window(const kda_desc_t* desc, int32_t window, const void* q,
                               const void* k, const void* v, const float* z, const float* beta,
                               const float* state, void* out, kda_stream_t stream);
kda_status_t kda_decode_replay(const kda_desc_t* desc, int32_t window, const void* q,
                               const void* k, const void* v, const float* z, const float* beta,
                               const int32_t* accept_len, float* state, kda_stream_t stream);

/*
 * kda_decode_replay_window -- the two calls above fused into one pass over
 * each request's state, as the pages describe the replay (one recurrent
 * loop): the first accept_len[b] drafts of the previous window (inputs
 * prev_*, [B * prev_window, H, .]) are applied and the state is written,
 * then the outputs of the new window (q .. beta, [B * window, H, .]) are
 * computed from it (the new drafts do not change the stored state).  The
 * state is read once and written once per call.  desc->total_tokens =
 * B * window.  A request whose accept_len is outside 0 .. prev_window keeps
 * its state, gets no outputs and sets the device error word.
 */
kda_status_t kda_decode_replay_window(const kda_desc_t* desc, int32_t prev_window,
                                      const void* prev_q, const void* prev_k, const void* prev_v,
                                      const float* prev_z, const float* prev_beta,
                                      const int32_t* accept_len, int32_t window, const void* q,
                                      const void* k, const void* v, const float* z,
                                      const float* beta, float* state, void* out,
                                      kda_stream_t stream);

/*
 * The decode-side calls with their surrounding per-token steps fused into the
 * same pass.  The pages describe K3's replay kernel as one recurrent loop that
 * fuses the short convolution, the input norm, the gating, the KDA recurrence
 * and the output norm (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
 * section "三条容易被忽略的代价" (1)); the pages define neither the
 * convolution's nor the output norm's form, so this library reads them as:
 *
 *   convolution: the depthwise causal convolution + Swish of kda_short_conv,
 *     applied to the raw q and k of every token before their L2 norm, the
 *     positions before a token reading that request's convolution state (its
 *     last W-1 raw inputs, oldest first);
 *   output norm: a per-head RMS norm of each output row,
 *     out = o / sqrt(mean_j o_j^2 + eps) * out_norm_weight[h].
 *
 * Options (NULL = none of them):
 *   conv_width          W: 0 = no convolution (q, k used as given), 1..4
 *                       (KDA_ERR_UNSUPPORTED above 4)
 *   conv_weight_q/_k    device [H, dk, W] fp32 taps (tap j multiplies
 *                       x[t - (W-1) + j]), required when W > 0
 *   conv_state_q/_k     device [B, H, dk, W-1] fp32, required when W > 1:
 *                       read, and advanced in place by the tokens that are
 *                       committed to the state (not by a window's drafts)
 *   out_norm_weight     device [H, dv] fp32, or NULL for no output norm
 *   out_norm_eps        >= 0
 */
typedef struct {
  int32_t conv_width;
  const float* conv_weight_q;
  const float* conv_weight_k;
  float* conv_state_q;
  float* conv_state_k;
  const float* out_norm_weight;
  float out_norm_eps;
} kda_fusion_t;

/* kda_decode_step with the options of `fusion`: q and k of each request
 * pass through the convolution (its state advances by this token) and the
 * outputs through the output norm.  Other arguments and errors as for
 * kda_decode_step; state must be 16-byte aligned. */
kda_status_t kda_decode_step_fused(const kda_desc_t* desc, const kda_fusion_t* fusion,
                                   const void* q, const void* k, const void* v, const float* z,
                                   const float* beta, float* state, void* out,
                                   kda_stream_t stream);

/* kda_decode_replay_window with the options of `fusion`, in one kernel: the
 * accepted prefix of the previous window (prev_*, raw inputs) is replayed
 * through convolution, norm, gate and recurrence, and the state and the
 * convolution states are written once; then the new window's drafts (raw
 * inputs) run from there, their outputs through the output norm, leaving
 * both states as the replay left them.  prev_window = 0 skips the replay
 * (prev_* and accept_len are not read); window = 0 computes no outputs (q ..
 * beta and out are not read; desc->total_tokens = 0).  Not both 0.
 * desc->total_tokens = B * window.  An accept_len outside 0 .. prev_window
 * leaves that request's states alone, gives it no outputs and sets the
 * device error word. */
kda_status_t kda_decode_replay_window_fused(
    const kda_desc_t* desc, const kda_fusion_t* fusion, int32_t prev_window, const void* prev_q,
    const void* prev_k, const void* prev_v, const float* prev_z, const float* prev_beta,
    const int32_t* accept_len, int32_t window, const void* q, const void* k, const void* v,
    const float* z, const float* beta, float* state, void* out, kda_stream_t stream);

/*
 * kda_chunk_fwd_fused -- kda_chunk_fwd over RAW q and k: the short
 * convolution + Swish of `fusion` (the Q/K preprocessing of mhpq.cn/news/56770,
 * section "KDA 到底在算什么", read as in kda_short_conv) runs inside the prefill
 * kernel on the q and k tiles it has loaded, before their L2 norm, so the
 * convolved q and k are never written to or read back from device memory.
 * Each sequence's convolution states (conv_state_q / _k, [N, H, dk, W-1])
 * are read as the raw inputs before its first token and, once every kernel
 * of the call has read them, overwritten with its last W-1 raw inputs (in
 * place; a sequence shorter than W-1 keeps the tail of its old state).
 *
 *   fusion             NULL or conv_width 0: exactly kda_chunk_fwd.
 *                      conv_width 1..4 needs the tensor-core path (bf16 io,
 *                      dk = dv = 128), else KDA_ERR_UNSUPPORTED; conv_state_*
 *                      are required when W > 1 and must not alias any other
 *                      buffer of the call.  out_norm_weight must be NULL
 *                      (KDA_ERR_UNSUPPORTED): the output norm belongs to the
 *                      decode-side calls.
 * Other arguments, options (workspace split, checkpoints, a_log,
 * gate_per_head) and errors as for kda_chunk_fwd.  The convolved q and k
 * stay in fp16 inside the kernel (finer than the bf16 that kda_short_conv
 * writes); a convolved value of magnitude 65504 or more sets
 * KDA_ERR_DEVICE_CHECK, like the tensor-core path's other fp16 operands.
 */
kda_status_t kda_chunk_fwd_fused(const kda_desc_t* desc, const kda_fusion_t* fusion,
                                 const void* q, const void* k, const void* v, const float* z,
                                 const float* beta, const float* initial_state,
                                 const int32_t* cu_seqlens, void* out, float* final_state,
                                 kda_stream_t stream);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd for callers that cannot allocate
 * device memory.  The pages describe no counterpart of this entry point.
 *
 * kda_chunk_fwd splits a few long sequences across SMs only when the caller
 * passes scratch in desc->workspace.  Callers whose device memory is owned
 * by a host framework that reserved all of HBM up front, plugins that are
 * not allowed to allocate, and latency-critical loops that cannot afford
 * cudaMalloc's implicit synchronisation may have no way to provide it.
 * This variant takes the same arguments (inputs and outputs still come from
 * the caller; desc->workspace is ignored) and uses instead a scratch array
 * of KDA_NOALLOC_SCRATCH_BYTES that is part of the library: every GPU that
 * loads libkda holds it until the process exits.  It calls no cudaMalloc,
 * no cudaFree and no allocating library routine.
 *
 *   - Every call that may split looks up the array's device address on the
 *     current device (cudaGetSymbolAddress); the first such call on a device
 *     also loads the library's module there, so make it before any stream
 *     capture on that device.
 *   - The split is the best plan whose segment summaries fit in
 *     KDA_NOALLOC_SCRATCH_BYTES; when none fits (see
 *     kda_chunk_fwd_workspace_size for what the best plan would need), the
 *     sequences run unsplit, which needs no scratch at all.
 *   - All calls share the one array and it keeps the last call's contents;
 *     every byte a call reads is written earlier in that same call, so
 *     nothing needs clearing.  Calls whose work overlaps on the GPU (for
 *     example on two streams) race on the array: serialise them.
 * Results are those of kda_chunk_fwd with a sufficient workspace.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
kda_status_t kda_chunk_fwd_noalloc(const kda_desc_t* desc, const void* q, const void* k,
                                   const void* v, const float* z, const float* beta,
                                   const float* initial_state, const int32_t* cu_seqlens,
                                   void* out, float* final_state, kda_stream_t stream);

/*
 * kda_testing_inject_wait_timeout -- testing aid for the failure path (the
 * device-side waits are bounded; this makes one of them run out).  The next
 * `launches` tensor-core prefill launches issued from the calling host thread
 * arm their first input barrier with 16 bytes that no copy delivers and cut
 * the wait budget to ~10 ms: the wait expires, the kernel records
 * KDA_ERR_TIMEOUT in the device error word, cancels the phantom bytes, lets
 * its real copies land, frees its Tensor Memory and returns.  Outputs of
 * such a launch are undefined.  0 disarms.
 */
void kda_testing_inject_wait_timeout(int launches);

/* Static, human-readable name of a status. */
/*
 * kda_chunk_fwd_host -- kda_chunk_fwd over inputs and outputs in HOST memory
 * (page-locked for the copies to overlap), for callers whose batch is not yet
 * on the device.  The batch is cut into `groups` groups of whole sequences of
 * about equal token count; the copies of one group into the device overlap
 * the kernel of the previous one and the copies of the one before back out.
 * Results equal those of kda_chunk_fwd on the same data except that the long-
 * sequence split across SMs is not used.
 *
 *   desc               as for kda_chunk_fwd; workspace / workspace_bytes:
 *                      DEVICE staging area of at least
 *                      kda_chunk_fwd_host_workspace_size() bytes, 256-byte
 *                      aligned, owned by the caller (one call at a time per
 *                      area); checkpoint_every must be 0 (else
 *                      KDA_ERR_UNSUPPORTED); a_log stays a DEVICE pointer
 *   groups             >= 1 (8 is a good default)
 *   q, k, v, z, beta, initial_state (or NULL), out, final_state (or NULL)
 *                      HOST, layouts as for kda_chunk_fwd
 *   cu_seqlens         HOST [N + 1] int32 (desc->cu_seqlens_host may be NULL
 *                      or this same pointer)
 * The call returns once the work is enqueued; work later enqueued on
 * `stream` runs after out and final_state are written to host memory, so a
 * cudaStreamSynchronize(stream) makes them readable.  The host buffers must
 * stay valid (and the inputs unchanged) until then.
 */
kda_status_t kda_chunk_fwd_host(const kda_desc_t* desc, int32_t groups, const void* q,
                                const void* k, const void* v, const float* z, const float* beta,
                                const float* initial_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, kda_stream_t stream);

/* Bytes of device staging area kda_chunk_fwd_host needs for this descriptor
 * (all inputs and outputs of the batch, both state arrays reserved). */
kda_status_t kda_chunk_fwd_host_workspace_size(const kda_desc_t* desc, size_t* bytes);

/*
 * kda_recurrent_bwd -- reverse mode of kda_chunk_fwd / kda_recurrent_fwd:
 * the gradients of a loss L with respect to every input, given dL/d out and
 * dL/d final_state.  The pages give the forward only (mhpq.cn/news/56770,
 * section "KDA 到底在算什么"; the gate of blog.higcp.com "猜想：K3 可能是最
 * 适合 TPU 的 MoE 架构", section "下界衰减"); the gradients are the chain rule
 * through those definitions, L2-normalisation and gate included, evaluated
 * token by token in fp32 in reverse order.  The states S_{t-1} it needs are
 * rebuilt forward from states the call itself keeps every 8 tokens in the
 * workspace.
 *
 *   desc               as for kda_chunk_fwd; any supported dk, dv (below 128
 *                      the inputs are zero-padded to 128 channels inside the
 *                      workspace, which changes no gradient of the real
 *                      channels and costs the work of dk = dv = 128);
 *                      gate_per_head = 1 takes z [T_tot, H] and gives dz
 *                      [T_tot, H] (the per-channel terms summed);
 *                      cu_seqlens_host is REQUIRED; workspace /
 *                      workspace_bytes must hold
 *                      kda_recurrent_bwd_workspace_size() bytes (16-byte
 *                      aligned); a_log is honoured; checkpoint fields are
 *                      ignored.
 *   q, k, v, z, beta, initial_state, cu_seqlens
 *                      the forward call's inputs (initial_state may be NULL)
 *   d_out              device, [T_tot, H, dv] io dtype: dL/d out
 *   d_final_state      device, [N, H, dk, dv] fp32, or NULL for zeros
 *   dq, dk, dz         device, [T_tot, H, dk] fp32 (dz [T_tot, H] with one
 *                      gate per head), written (dz is the gradient w.r.t. the
 *                      gate logits z as passed)
 *   dv                 device, [T_tot, H, dv] fp32, written
 *   dbeta              device, [T_tot, H] fp32, written
 *   d_initial_state    device, [N, H, dk, dv] fp32, written, or NULL
 * Every pointer to per-token or state data must be 16-byte aligned, and no
 * output may alias an input.  Errors as for kda_chunk_fwd; a device copy of
 * cu_seqlens whose lengths exceed those of the host copy skips the
 * offending sequences and sets the device error word.
 */
kda_status_t kda_recurrent_bwd(const kda_desc_t* desc, const void* q, const void* k,
                               const void* v, const float* z, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens,
                               const void* d_out, const float* d_final_state, float* dq,
                               float* dk, float* dv, float* dz, float* dbeta,
                               float* d_initial_state, kda_stream_t stream);

/* Bytes of device workspace kda_recurrent_bwd needs for this descriptor
 * (needs desc->cu_seqlens_host): for every resident CTA (at most one per
 * SM) 64 KiB per 8 tokens of the longest sequence, plus 512 KiB; below
 * dk = dv = 128 also the zero-padded copies of the inputs and gradients. */
kda_status_t kda_recurrent_bwd_workspace_size(const kda_desc_t* desc, size_t* bytes);

/*
 * kda_chunk_bwd -- the same gradients as kda_recurrent_bwd from the chunked
 * (WY / UT) form of the recurrence (mhpq.cn/news/56770, section "KDA 到底在算
 * 什么", evaluated chunkwise; the chunked forward with a custom reverse mode
 * is the training kernel of blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架
 * 构", section "第二层").  Per 16-token chunk the state products (dO S^T,
 * dR S^T, U dS'^T, K~ dS', Q+^T dO - K+^T dR, ...) and the chunk's own 16 x 16
 * products run on the tensor cores (bf16 MMAs, fp32 accumulation); states
 * and their gradients stay fp32.  A forward sweep keeps the state entering
 * every chunk, and the chunk's R = V - K+ S, U, A and T, in the workspace.
 * Arguments, layouts, dtypes, alignment and errors exactly as for
 * kda_recurrent_bwd (any supported dk, dv; per-channel or per-head gate;
 * a_log honoured; cu_seqlens_host REQUIRED); the workspace must hold
 * kda_chunk_bwd_workspace_size() bytes.  Accuracy: every tensor-core operand
 * is split into a high and a low bf16 part (16 significant bits, three
 * multiplies per product, fp32 accumulation), and the gradient of the
 * log-decay is summed without cancelling terms, so the gradients agree with
 * an fp64 evaluation to about 1e-5 relative L2, like kda_recurrent_bwd.
 */
kda_status_t kda_chunk_bwd(const kda_desc_t* desc, const void* q, const void* k, const void* v,
                           const float* z, const float* beta, const float* initial_state,
                           const int32_t* cu_seqlens, const void* d_out,
                           const float* d_final_state, float* dq, float* dk, float* dv,
                           float* dz, float* dbeta, float* d_initial_state, kda_stream_t stream);

/* Bytes of device workspace kda_chunk_bwd needs (needs desc->cu_seqlens_host):
 * for every resident CTA (at most one per SM) 84 KiB per 16 tokens of the
 * longest sequence (the state entering each chunk and 20 KiB of the chunk's
 * own products); below dk = dv = 128 also the zero-padded copies of the inputs
 * and gradients. */
kda_status_t kda_chunk_bwd_workspace_size(const kda_desc_t* desc, size_t* bytes);

/*
 * kda_short_conv -- the Q/K preprocessing before the recurrence
 * (mhpq.cn/news/56770, section "KDA 到底在算什么", the Q/K preprocessing
 * paragraph: a short causal convolution over the most recent few positions,
 * then a Swish activation, then the L2 normalisation that kda_chunk_fwd and
 * kda_decode_step apply themselves).  The page gives neither width nor form;
 * this call is a depthwise causal convolution of width W (1..4) without bias:
 *
 *     y[t, h, d] = swish( sum_{j<W} weight[h, d, j] x[t - (W-1) + j, h, d] ),
 *     swish(u) = u / (1 + e^{-u}),
 *
 * where the positions before a sequence's first token read its convolution
 * state.  Apply it to q and to k (one call each, with their own weights).
 *
 *   desc             num_seqs, total_tokens, num_heads, io_dtype as for
 *                    kda_chunk_fwd; the channel count is desc->dk (32, 64
 *                    or 128); other fields are ignored.  For a decode step
 *                    pass cu_seqlens = 0, 1, .., N.
 *   width            W, 1..4 (KDA_ERR_UNSUPPORTED above 4)
 *   x                device, [T_tot, H, dk] io dtype, read
 *   weight           device, [H, dk, W] fp32 (tap j multiplies x[t-(W-1)+j])
 *   conv_state_in    device, [N, H, dk, W-1] fp32: each sequence's W-1 inputs
 *                    before its first token, oldest first; NULL for zeros
 *   cu_seqlens       device, [N + 1] int32
 *   y                device, [T_tot, H, dk] io dtype, written; must not
 *                    alias x, weight or conv_state_in
 *   conv_state_out   device, [N, H, dk, W-1] fp32, written with each
 *                    sequence's last W-1 inputs (continued from
 *                    conv_state_in when shorter), or NULL; may alias
 *                    conv_state_in exactly (it is written after every read)
 * x and y must be 16-byte aligned.  A device cu_seqlens that does not start
 * at 0, end at T_tot and rise monotonically sets the device error word.
 */
kda_status_t kda_short_conv(const kda_desc_t* desc, int32_t width, const void* x,
                            const float* weight, const float* conv_state_in,
                            const int32_t* cu_seqlens, void* y, float* conv_state_out,
                            kda_stream_t stream);

/*
 * Context parallelism: one long sequence cut along its tokens across
 * devices.  The state update is affine in the state (mhpq.cn/news/56770,
 * section "KDA 到底在算什么"), so a piece of a sequence maps the state entering
 * it to S_out = M S_in + S~.  The pages' context-parallel KDA (blog.higcp.com
 * "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "第二层") has each device
 * summarise its piece by (M, S~), exchange the summaries in one all-gather,
 * rebuild the state entering its piece by a prefix scan, and then run its
 * piece from that state (kda_chunk_fwd with initial_state = that state).
 *
 * kda_chunk_fwd_summary -- the affine summary of every sequence of a packed
 * batch (each rank's pieces):
 *
 *   desc               as for kda_chunk_fwd; bf16 io and dk = dv = 128 only
 *                      (else KDA_ERR_UNSUPPORTED); cu_seqlens_host is
 *                      REQUIRED; a_log and gate_per_head are honoured;
 *                      workspace / workspace_bytes: optional device scratch
 *                      (256-byte aligned) that lets long sequences be cut
 *                      into segments summarised side by side and composed
 *                      (kda_chunk_fwd_summary_workspace_size gives what the
 *                      best plan needs; a smaller area limits the plan);
 *                      checkpoint fields are ignored.
 *   q, k, v, z, beta, cu_seqlens   device, as for kda_chunk_fwd (q, k, v, z
 *                      16-byte aligned)
 *   transition         device, [N, H, dk, dk] fp32, written: M, the product
 *                      of the sequence's per-token transitions
 *                      (I - beta k k^T) Diag(alpha), row = output key channel
 *   offset_state       device, [N, H, dk, dv] fp32, written: S~, the state
 *                      the sequence reaches from zeros
 * An empty sequence gives M = I and S~ = 0.  Neither output may alias an
 * input or the other.  In fp32, M's entries underflow to zero when the
 * piece decays them below about e^-87; M S_in + S~ stays accurate.
 */
kda_status_t kda_chunk_fwd_summary(const kda_desc_t* desc, const void* q, const void* k,
                                   const void* v, const float* z, const float* beta,
                                   const int32_t* cu_seqlens, float* transition,
                                   float* offset_state, kda_stream_t stream);

/* Bytes of device scratch that let kda_chunk_fwd_summary split long
 * sequences across SMs (0 when no split would be planned).  Needs
 * desc->cu_seqlens_host. */
kda_status_t kda_chunk_fwd_summary_workspace_size(const kda_desc_t* desc, size_t* bytes);

/*
 * kda_state_scan -- the prefix scan of the scheme above: starting from
 * initial_state (zeros when NULL), applies S <- M_i S + S~_i for
 * i = 0 .. count-1, in fp32, to every (sequence, head).  Rank r of a
 * context-parallel run calls it with count = r on the gathered summaries
 * of ranks 0 .. R-1 to get the state entering its pieces.
 *
 *   desc               num_seqs (N), num_heads (H), dk, dv (32, 64 or 128);
 *                      other fields are ignored
 *   count              >= 0; 0 copies initial_state (or writes zeros)
 *   transitions        device, [count, N, H, dk, dk] fp32 (rank-major, as an
 *                      all-gather of kda_chunk_fwd_summary's transition
 *                      lays them out); may be NULL when count = 0
 *   offsets            device, [count, N, H, dk, dv] fp32, likewise
 *   initial_state      device, [N, H, dk, dv] fp32, or NULL for zeros
 *   entry_state        device, [N, H, dk, dv] fp32, written; may alias
 *                      initial_state exactly, not transitions or offsets
 */
kda_status_t kda_state_scan(const kda_desc_t* desc, int32_t count, const float* transitions,
                            const float* offsets, const float* initial_state,
                            float* entry_state, kda_stream_t stream);

const char* kda_status_string(kda_status_t status);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device: KDA_OK, KDA_ERR_DEVICE_CHECK or KDA_ERR_TIMEOUT.  Returns
 * KDA_ERR_CUDA if the synchronisation itself fails. */
kda_status_t kda_get_device_error(kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
