/*
 * kda.h — C ABI of libkda.so: Kimi Delta Attention (KDA) on one GB300 (sm_103a).
 *
 * KDA is the gated delta-rule linear attention of the Kimi K3 model.  Per head
 * it carries a state S of dv x dk values.  For each token, with q, k, v after
 * ShortConv(kernel 4) + SiLU and q, k L2-normalised, alpha = exp(g) a
 * per-key-channel decay (g >= -5) and beta a scalar in [0, 1]:
 *
 *     S~  = S Diag(alpha)                 (decay, one factor per key channel)
 *     S   = S~ + beta (v - S~ k) k^T      (delta-rule correction)
 *     o   = scale * S q
 *
 * Sources: "Kimi-K3 深度解析: 2.8T 开源 MoE 模型的架构创新与设计哲学", section 三,
 * subsection "KDA 的关键改进" (the two update equations); "Kimi K3 架构全景",
 * section 02, KDA column (96 heads x 128, ShortConv kernel 4, gate lower bound
 * -5.0, operators chunk_kda / fused_recurrent_kda, recurrent state instead of a
 * KV cache); "深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA (short
 * convolution with SiLU on q, k, v; L2 norm of q and k inside the kernel;
 * per-channel decay bounded below by -5; full-rank output gate).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer (and the prefill's workspace) is CALLER-OWNED DEVICE
 *    memory on the current CUDA device.  The library allocates no device memory,
 *    frees nothing and keeps no state between calls apart from one device error
 *    word (see kda_device_error) and, per device, two CUDA streams that
 *    kda_chunk_fwd creates on its first overlapped call (see kda_chunk_fwd; make
 *    that first call outside a stream capture).
 *  - Calls are asynchronous: they check their arguments on the host, enqueue
 *    kernels on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *    return.  An argument error returns before anything is enqueued.  A launch
 *    failure returns KDA_ERR_CUDA.  kda_last_error() gives a message.
 *  - Layouts are row-major, innermost index last:
 *      q, k, g            [T_total, H, dk]
 *      v, o               [T_total, H, dv]
 *      beta               [T_total, H]
 *      states             [N, H, dv, dk]   fp32 (S is dv x dk)
 *      raw front-end rows [T_total, x_row_stride], the first H*d used
 *      conv_w             [3*H*d, 4] bf16: rows are q channels, then k, then v;
 *                          taps oldest .. current token
 *      conv_state         [N, 3, 3*H*d] bf16: the last three raw inputs of each
 *                          sequence, oldest row first, same channel order
 *      cu_seqlens         [N + 1] int32 on the device, non-decreasing, first 0,
 *                          last T_total (NULL = one sequence of T_total tokens)
 *  - Every device pointer must be 16-byte aligned.  Only d = dk = dv = 128 is
 *    supported (KDA_ERR_UNSUPPORTED otherwise); chunk_size must be 64.
 *  - Preconditions the kernels rely on: g in [-5, 0], beta in [0, 1], finite
 *    inputs.  They are not clamped.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* a null, misaligned or inconsistent argument          */
    KDA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d != 128)            */
    KDA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed                 */
    KDA_ERR_DEVICE = 4       /* a kernel reported a fault through the error word     */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/* Bits of the device error word (see kda_device_error). */
#define KDA_DEVICE_ERR_WAIT_TIMEOUT 1u
#define KDA_DEVICE_ERR_GATE_RANGE 2u
#define KDA_DEVICE_ERR_BETA_RANGE 4u

/*
 * Front end of a prefill: ShortConv(kernel 4) + SiLU on each of q, k, v, then
 * L2 normalisation of q and k over each head's d channels ("深入 Kimi-K3: Hugging
 * Face 仓库分析", paragraph on KDA; kernel size from "Kimi K3 架构全景", section 02).
 *
 * For part p in {q, k, v}, channel c, token t of sequence n:
 *   y = sum_{i=0..3} conv_w[p*H*d + c][i] * x_p[t - 3 + i][c]
 *   a = y / (1 + exp(-y))
 *   q_out, k_out = a / sqrt(sum over the head's channels of a^2 + eps); v_out = a
 * Positions before a sequence's first token read conv_state_in[n] (row 3 - j
 * for j positions back), or zero when conv_state_in is NULL.  The convolution
 * has no bias and restarts at every cu_seqlens boundary.
 *
 *  xq, xk, xv      raw bf16 rows [T_total, x_row_stride] (x_row_stride >= H*d,
 *                  a multiple of 8 elements)
 *  conv_w          bf16 [3*H*d, 4]
 *  cu_seqlens, N   see conventions
 *  conv_state_in   bf16 [N, 3, 3*H*d] or NULL
 *  conv_state_out  bf16 [N, 3, 3*H*d] or NULL: receives the last three raw
 *                  inputs of each sequence (reading conv_state_in for sequences
 *                  shorter than 3).  May be the same buffer as conv_state_in.
 *  out_dtype       storage type of q_out, k_out, v_out ([T_total, H, d])
 */
KDA_API kda_status kda_shortconv_l2norm(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                                const void* conv_w, const int32_t* cu_seqlens, int N, int64_t T_total,
                                int H, int d, const void* conv_state_in, void* conv_state_out, float eps,
                                kda_dtype out_dtype, void* q_out, void* k_out, void* v_out, void* stream);

/*
 * Chunkwise prefill (the chunk_kda operator of "Kimi K3 架构全景", section 02):
 * runs the recurrence above over every sequence of a packed batch and returns
 * every token's output and each sequence's final state.  The result equals the
 * token-by-token recurrence; the chunk form only reorders the arithmetic.
 *
 *  q, k            [T_total, H, dk], storage `dtype`; L2-normalised by the caller
 *  v               [T_total, H, dv], storage `dtype`
 *  g               fp32 [T_total, H, dk], log-decay in [-5, 0]
 *  beta            fp32 [T_total, H], in [0, 1]
 *  init_state      fp32 [N, H, dv, dk] or NULL (= zeros)
 *  cu_seqlens, N   see conventions; sequences may be empty (final = initial)
 *  scale           multiplies every output
 *  chunk_size      64
 *  dtype           KDA_DTYPE_F32: fp32 inputs and output, computed in fp32 with
 *                  explicit position-pair decays (no use of the -5 bound).
 *                  KDA_DTYPE_BF16: bf16 inputs and output, intra-chunk products
 *                  on bf16 tensor cores with fp32 accumulation, fp32 state.
 *  out_gate        bf16 [T_total, H*dv] or NULL: if given, o *= sigmoid(out_gate)
 *                  (the full-rank output gate, "深入 Kimi-K3: Hugging Face 仓库分析")
 *  o               [T_total, H, dv], storage `dtype`
 *  final_state     fp32 [N, H, dv, dk] or NULL.  May be the same buffer as
 *                  init_state (each sequence's state is read before it is written).
 *  workspace       device scratch of workspace_bytes bytes, 16-byte aligned, used
 *                  only during the call (stream-ordered).  KDA_DTYPE_BF16 needs at
 *                  least the `min_bytes` of kda_chunk_fwd_workspace_size and runs
 *                  fastest with `full_bytes`; with less, the chunks are processed in
 *                  several ranges.  KDA_DTYPE_F32 ignores it (may be NULL, 0).
 *
 * Overlapped ranges: when the call has at least 256 chunk rows (a chunk row is 64 tokens of
 * every sequence's chunk numbering, all heads) and the workspace holds at least 256 of them,
 * consecutive ranges of max(128, rows / 8) chunk rows overlap (at most half of what the workspace
 * holds).  The call then forks two internal streams from `stream` with events (the operand kernel
 * on a low-priority one, the state pass on a high-priority one) and makes `stream` wait for both
 * before it returns; nothing else changes for the caller, and the results are the same bits as
 * one range.  The two internal streams are per device and shared by every call: overlapped calls
 * on one device are serialised through them even when the callers use independent streams.
 * Otherwise every range runs on `stream`, one after the other.
 *
 * Device resets: the library carries its own (statically linked) CUDA runtime, whose loaded kernels and
 * device variables belong to the device context of the process's first call, and it keeps the
 * addresses of its device error word and static scratch and its two streams per device.  None of
 * that survives a reset of the device (cudaDeviceReset by the caller's runtime destroys the context):
 * do not call the library in a process after resetting a device it has been used on.
 *
 * The bf16 path runs two kernels per range of chunks: the first computes, for every
 * (chunk, head) at once, everything that does not depend on the carried state (the
 * in-chunk decays, the A_kk / A_qk blocks, T = (I + A_kk)^-1, W = T diag(beta) K e^G and
 * T diag(beta) itself) and stores the chunk's operands in the workspace (82,432 bytes per
 * chunk and head); the second walks each sequence's chunks in order with the state, forming
 * U = T diag(beta) V from v itself.
 */
KDA_API kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                         int dk, int dv, float scale, int chunk_size, kda_dtype dtype, const void* out_gate,
                         void* o, float* final_state, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The prefill with its front end fused in: the result of kda_shortconv_l2norm (bf16 outputs)
 * followed by kda_chunk_fwd (bf16), without writing and re-reading q and k (the front end runs on
 * the same arithmetic, so the outputs are the same bits: q and k inside the kernel that builds the
 * chunk operands, v by the stand-alone front end into o, from where the state pass reads it).  This is the
 * pages' normalisation "in the kernel" taken one step further ("深入 Kimi-K3: Hugging Face 仓库
 * 分析", paragraph on KDA).
 *
 *  xq, xk, xv, x_row_stride, conv_w, conv_state_in, conv_state_out, eps
 *                  as kda_shortconv_l2norm (conv_state_out may alias conv_state_in)
 *  g, beta, init_state, cu_seqlens, N, scale, chunk_size, out_gate, o, final_state, workspace
 *                  as kda_chunk_fwd with dtype KDA_DTYPE_BF16 (o bf16 [T_total, H, d])
 *
 * o holds v during the call (the front end writes v there and the state pass reads each chunk's
 * tile of it before writing that chunk's outputs over it), so o must not overlap xq, xk, xv,
 * out_gate, g or beta: KDA_ERR_INVALID_ARG otherwise.
 */
KDA_API kda_status kda_chunk_fwd_frontend(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                                  const void* conv_w, const void* conv_state_in, void* conv_state_out,
                                  float eps, const float* g, const float* beta, const float* init_state,
                                  const int32_t* cu_seqlens, int N, int64_t T_total, int H, int d,
                                  float scale, int chunk_size, const void* out_gate, void* o,
                                  float* final_state, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_chunk_fwd without a caller workspace (no counterpart in the sources; an interface
 * convenience for callers that cannot allocate device memory, e.g. code running inside an
 * allocator-free runtime or under a memory pool it does not own).  The bf16 path uses a
 * 64 MiB scratch array that is part of the library's device image (every GPU that loads the
 * library holds it until exit), so neither the caller nor the library allocates anything: no
 * cudaMalloc, no internal streams, no events.  Its chunk ranges (as many chunk rows per range
 * as fit in 64 MiB; 6 rows at H = 96) run one after the other on `stream`.
 * The first call on a device looks up the array's device address (with that device current)
 * and keeps it; make that first call before any stream capture.
 * Returns KDA_ERR_UNSUPPORTED, before enqueueing anything, when even one chunk row of all
 * heads does not fit (the `min_bytes` of kda_chunk_fwd_workspace_size exceeds 64 MiB: H above
 * about 290).  Calls share the scratch, which keeps the last call's contents: calls that
 * overlap on one device race and must be ordered (one stream, or streams ordered by events).
 * Arguments and layouts as kda_chunk_fwd.
 */
KDA_API kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* init_state, const int32_t* cu_seqlens, int N,
                                 int64_t T_total, int H, int dk, int dv, float scale, int chunk_size,
                                 kda_dtype dtype, const void* out_gate, void* o, float* final_state,
                                 void* stream);

/*
 * Workspace of kda_chunk_fwd for these sizes (no device access): *full_bytes runs every
 * chunk in one range, *min_bytes is the least accepted (one chunk row of all heads).
 * Both are 0 for KDA_DTYPE_F32.  have_cu_seqlens: whether cu_seqlens will be given.
 * Either output pointer may be NULL.
 */
KDA_API kda_status kda_chunk_fwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv, int chunk_size,
                                        kda_dtype dtype, int have_cu_seqlens, size_t* full_bytes,
                                        size_t* min_bytes);

/*
 * Summaries of segments of sequences, for carrying the state across them (a long sequence split
 * into segments, each worked on separately, e.g. one per device).  The update of "Kimi-K3 深度
 * 解析", section 三 ("KDA 的关键改进"), S_t = S_{t-1} Diag(alpha_t)(I - beta_t k_t k_t^T) +
 * beta_t v_t k_t^T, is affine in S_{t-1}, so each (sequence, head) segment maps its entering state S
 * to  S M + E  with
 *   E = its final state from a zero start (what kda_chunk_fwd returns without init_state), and
 *   M = X_1 X_2 ... X_L, X_t = Diag(exp g_t)(I - beta_t k_t k_t^T)  (its transition operator).
 * M is the final state of the same recurrence with v = 0 from S = I, and is computed that way on
 * the chunk path (bf16 products, fp32 state).
 *
 *  q               bf16 [T_total, H, 128] or NULL: M and E do not depend on it (k stands in)
 *  k, g, beta, cu_seqlens, N, T_total, H, dk, dv, chunk_size
 *                  as kda_chunk_fwd with dtype KDA_DTYPE_BF16 (dk = dv = 128, chunk_size 64)
 *  v               bf16 [T_total, H, 128]; may be NULL when end_state is NULL
 *  end_state       fp32 [N, H, 128, 128] out (E), or NULL
 *  transition      fp32 [N, H, 128, 128] out (M), or NULL; not both NULL
 *  workspace       as kda_chunk_fwd; with the `full_bytes` of kda_chunk_fwd_workspace_size the
 *                  chunk operands are computed once for both outputs, with less twice
 *
 * Writes nothing else.  Errors as kda_chunk_fwd.
 */
KDA_API kda_status kda_chunk_segment_summary(const void* q, const void* k, const void* v, const float* g,
                                             const float* beta, const int32_t* cu_seqlens, int N, int64_t T_total,
                                             int H, int dk, int dv, int chunk_size, float* end_state,
                                             float* transition, void* workspace, size_t workspace_bytes,
                                             void* stream);

/*
 * Backward of kda_chunk_fwd (the chunk_kda operator is what trains the model, "月之暗面发布Kimi K3
 * 开源大模型技术报告", 架构): given dL/do for every token and dL/dS_final for every sequence, the
 * gradients of L with respect to q, k, v, g, beta and the initial state.  The result equals reverse
 * mode through the token-by-token recurrence; the kernels take the chain rule through the chunk form
 * (a forward pass that keeps the state entering every chunk, a reverse pass over the chunks for the
 * gradient of the state, then every (chunk, head) at once).  fp32 inputs: fp32 arithmetic on the CUDA
 * cores with explicit position-pair decays (no use of the -5 bound).  bf16 inputs: every product on the
 * tensor cores with fp32 accumulation, each fp32 operand split into bf16 pieces to keep fp32-level
 * accuracy (hi + lo, three bf16 products; three pieces and six products in the position-pair sums), the
 * decays factorised around 16-token blocks as in kda_chunk_fwd (so g must respect the -5 bound there);
 * with bf16 inputs the g and beta range checks of kda_chunk_fwd run too (the bits of kda_device_error).
 *
 *  q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, chunk_size
 *                  as kda_chunk_fwd (q, k, v and d_o in storage `dtype`, F32 or BF16)
 *  d_o             dL/do [T_total, H, dv], storage `dtype`
 *  d_final_state   fp32 dL/dS_final [N, H, dv, dk] or NULL (= zeros)
 *  dq, dk_out      fp32 [T_total, H, dk] out
 *  dv_out          fp32 [T_total, H, dv] out
 *  dg              fp32 [T_total, H, dk] out
 *  dbeta           fp32 [T_total, H] out
 *  d_init_state    fp32 dL/dS0 [N, H, dv, dk] out, or NULL
 *  workspace       device scratch of at least kda_chunk_bwd_workspace_size bytes, 16-byte aligned,
 *                  used only during the call (stream-ordered)
 *
 * Outputs must not alias inputs or each other.  Errors as kda_chunk_fwd.
 */
KDA_API kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                                 int dk, int dv, float scale, int chunk_size, kda_dtype dtype, const void* d_o,
                                 const float* d_final_state, float* dq, float* dk_out, float* dv_out, float* dg,
                                 float* dbeta, float* d_init_state, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * Bytes of workspace kda_chunk_bwd needs for these sizes (into *bytes): the state entering each chunk
 * and the gradient leaving it (64 KB each per chunk and head), six fp32 values per token, head and
 * channel, two per token and head, and per chunk and head three 64 x 128 and four 64 x 64 fp32 tiles,
 * two vectors of 128, and 131,840 bytes of bf16 tiles for the tensor-core passes (bf16 inputs).
 */
KDA_API kda_status kda_chunk_bwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv, int chunk_size,
                                                size_t* bytes);

/*
 * The decay gate and the full-rank output gate from the layer input ("深入 Kimi-K3: Hugging Face 仓库
 * 分析", paragraph on KDA: the decay is per channel, driven by a low-rank projection plus a per-head
 * parameter, with a lower bound of -5; the output gate is full rank; "Kimi K3 架构全景", section 02:
 * gate lower_bound -5.0).  The pages give no formula; read here as
 *   gate = x W_gate^T,   z = x W_a^T (rank `rank`),   g = max(-5, -softplus(z W_b^T + a_h))
 * with a_h one parameter per head (the same for the head's d channels); -softplus keeps every
 * decay factor exp(g) at most 1 and the floor keeps it at least e^-5.  x W_gate^T and x W_a^T run as
 * one tcgen05 GEMM over the stacked weights, z W_b^T as a second one with the gate in its epilogue;
 * fp32 accumulation, z rounded to bf16 between the two.
 *
 *  x            bf16 [T, hidden] (row-major)
 *  w_gate_a     bf16 [H*d + rank, hidden]: rows [0, H*d) W_gate, rows [H*d, H*d + rank) W_a
 *  w_b          bf16 [H*d, rank]
 *  a_head       fp32 [H]
 *  gate         bf16 [T, H*d] out (the `out_gate` of kda_chunk_fwd)
 *  g            fp32 [T, H, d] out (the `g` of kda_chunk_fwd), in [-5, 0]
 *  z_workspace  bf16 [T, rank] scratch
 *  T in [0, 2^31), hidden a positive multiple of 8, d = 128, rank a multiple of 32 in [32, 4096].
 *  All pointers 16-byte aligned device memory (with T = 0, x, gate, g and z_workspace may be NULL).
 */
KDA_API kda_status kda_gate_generator(const void* x, int64_t T, int hidden, const void* w_gate_a, const void* w_b,
                                      const float* a_head, int H, int d, int rank, void* gate, float* g,
                                      void* z_workspace, void* stream);

/*
 * The map of a segment applied to a state:  S_out[i] = S_in[i] M[i] + E[i]  for i < count, each a
 * fp32 128 x 128 row-major matrix (S_in NULL: S_out = E).  Folding the segments of a sequence in
 * order with it gives each segment's entering state (see kda_chunk_segment_summary).  Products in
 * fp32, k summed in order.  S_out may alias any input.  All pointers 16-byte aligned device
 * memory; count >= 0.
 */
KDA_API kda_status kda_state_combine(const float* S_in, const float* M, const float* E, float* S_out, int64_t count,
                                     void* stream);

/*
 * One decode step (the fused_recurrent_kda operator of "Kimi K3 架构全景",
 * section 02) for N sequences of one new token each, fused end to end: the
 * ShortConv(4) + SiLU + L2 norm front end on the token's raw q, k, v (shifting
 * conv_state in place), then the recurrence on the fp32 state (in place), and
 * the output.
 *
 *  xq, xk, xv      raw bf16 rows [N, x_row_stride] (x_row_stride >= H*d, a
 *                  multiple of 8 elements)
 *  conv_w          bf16 [3*H*d, 4]
 *  g               fp32 [N, H, dk] log-decay in [-5, 0];  beta fp32 [N, H]
 *  state           fp32 [N, H, dv, dk], read and overwritten
 *  conv_state      bf16 [N, 3, 3*H*d], read and overwritten (rows shift up by
 *                  one, the raw token enters as row 2)
 *  o               bf16 [N, H, dv]
 */
KDA_API kda_status kda_recurrent_step(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                              const void* conv_w, const float* g, const float* beta, float* state,
                              void* conv_state, int N, int H, int dk, int dv, float scale, float eps, void* o,
                              void* stream);

/* Static description of a status code. */
KDA_API const char* kda_status_string(kda_status s);

/* Message of the last failing call on this host thread ("" if none). */
KDA_API const char* kda_last_error(void);

/*
 * Reads and clears the device error word of the current device (synchronous:
 * waits for all work on the device).  0 = no fault; otherwise the OR of the
 * KDA_DEVICE_ERR_* bits (defined after kda_dtype) raised since the last read:
 *   KDA_DEVICE_ERR_WAIT_TIMEOUT  one of a kernel's bounded waits ran out (the kernel
 *                                stopped instead of hanging; its outputs are incomplete)
 *   KDA_DEVICE_ERR_GATE_RANGE    a log-decay g outside [-5, 0], or not finite (the bf16
 *                                chunk path relies on the bound, "Kimi K3 架构全景",
 *                                section 02, gate lower bound -5.0; "月之暗面发布Kimi K3
 *                                开源大模型技术报告", 架构)
 *   KDA_DEVICE_ERR_BETA_RANGE    a beta outside [0, 1], or not finite
 * The range bits are raised by kda_chunk_fwd, kda_chunk_fwd_frontend,
 * kda_chunk_fwd_noalloc, kda_chunk_segment_summary and kda_chunk_bwd with bf16 inputs
 * (every g and beta of every token is checked as it is read) and by kda_recurrent_step; the
 * call still completes (nothing traps) and its results are then unspecified.
 * Returns KDA_ERR_CUDA if the read itself fails.
 */
KDA_API kda_status kda_device_error(unsigned int* code);

/*
 * Diagnostic (no counterpart in the sources): launches one CTA whose thread waits on an
 * mbarrier that nothing ever arrives at, polling at most `poll_limit` times (1 .. 2^24),
 * exactly as the library's kernels wait on their tensor-core and copy barriers.  The
 * wait runs out, the kernel records KDA_DEVICE_ERR_WAIT_TIMEOUT in the device error word
 * and returns; kda_device_error() then reports it.  It exercises the path a kernel takes
 * instead of hanging, without faulting the GPU.  Asynchronous on `stream`.
 */

KDA_API kda_status kda_selftest_bounded_wait(unsigned int poll_limit, void* stream);

/* Library version, e.g. "0.1.0". */
KDA_API const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
