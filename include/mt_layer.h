/*
 * mt_layer.h -- C ABI of a GB300 (sm_103a) forward pass of one GPT/Llama Transformer layer,
 * as one tensor-parallel (TP) rank computes it.
 *
 * What is computed (page titles and sections of the Megatron pages this follows):
 *   "快速入门 / Pai-Megatron-Patch 项目深度学习总结文档" §3.1, layer tree and layer spec:
 *       input_layernorm -> SelfAttention(linear_qkv, core_attention [causal], linear_proj)
 *       -> bias-dropout-add -> pre_mlp_layernorm -> MLP(linear_fc1, linear_fc2) -> bias-dropout-add.
 *   "Megatron-LM 深度学习与源码分析文档" Part 2 §2 (Tensor Parallel):
 *       Y = XW; column-parallel W=[W_1..W_p], Y_i = X W_i; row-parallel W=[W_1;..;W_p],
 *       Y_i = X_i W_i, Y = sum_i Y_i; QKV is column-parallel with heads/TP heads per rank;
 *       MLP Z = phi(X W_1), Y = Z W_2 with fc1 column- and fc2 row-parallel (SwiGLU widens fc1).
 *   "ai阅读megatron", TransformerConfig (num_query_groups => GQA) and the Llama flag sets
 *       (--swiglu, --normalization RMSNorm, rotary position embeddings).
 *   Dropout is the identity (rate 0.0 in the launch flags of "快速入门" §6.1); the softmax
 *   scale is 1/sqrt(head_dim) (query-key layer scaling disabled, same flags).
 *
 * Notation: T = seq*batch tokens, H = hidden, d = head_dim, nh_r = heads/tp, ng_r = groups/tp,
 * q_w = nh_r*d, kv_w = ng_r*d, f_r = ffn/tp, f1_r = 2*f_r (SwiGLU) or f_r (GeLU).
 *
 * Layouts.  All tensors are bfloat16, row-major.  Activations use the [seq, batch, hidden]
 * order, i.e. a [T, H] matrix whose row t = s*batch + b.  Weights are [out, in] (rows are
 * output features, the F.linear convention):
 *   w_qkv [q_w + 2*kv_w, H] rows = [this rank's q heads | its k groups | its v groups],
 *         each head d consecutive rows;  w_o [H, q_w];  w_fc1 [f1_r, H] rows = [gate | up]
 *         for SwiGLU;  w_fc2 [H, f_r];  norm gains/shifts [H];  biases [out].
 *   RoPE: rotate-half pairs (i, i+d/2), angle = s * rope_base^(-2i/d), on q and k after the bias.
 *   GQA: q head h (within the rank) reads kv group h / (nh_r/ng_r).
 *
 * Ownership.  The caller owns x, the weights, every output and the workspace (all device
 * memory unless stated).  The library owns the handle, a 4-byte device error word and 16 MiB
 * of device memory for the fp32 partial sums of the GEMMs' K-split tail tiles (with 4 KiB of
 * arrival counters), allocated in mt_layer_create and freed in mt_layer_destroy.  Calls that take a
 * stream are asynchronous on it; a handle must not be used from two host threads at once, and its
 * calls must not overlap on the GPU (on two streams without an ordering event between them): they
 * share the workspace, the partial sums and the counters.
 *
 * Errors.  Every call returns an mt_status; on failure no kernel is launched and
 * mt_last_error() describes the problem (thread-local string, valid until the next call on the
 * same thread).  A kernel that stops waiting (bounded waits on barriers; it never hangs)
 * records MT_ERR_DEVICE_TIMEOUT in the error word; mt_layer_status reports and clears it.
 */
#ifndef MT_LAYER_H
#define MT_LAYER_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mt_layer mt_layer; /* opaque, library-owned */

enum { MT_NORM_RMS = 0, MT_NORM_LAYER = 1 };
enum { MT_ACT_SWIGLU = 0, MT_ACT_GELU_TANH = 1 };

typedef enum {
  MT_OK = 0,
  MT_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, non-positive size, bad enum        */
  MT_ERR_UNSUPPORTED = 2,     /* well-formed but outside the supported shapes (see create)   */
  MT_ERR_NO_WORKSPACE = 3,    /* no workspace set, or smaller than mt_layer_workspace_bytes  */
  MT_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (message has the detail)  */
  MT_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up on a barrier wait; its outputs are invalid */
  MT_ERR_UNIMPLEMENTED = 6
} mt_status;

/* One rank's weights.  Device pointers to bf16, 16-byte aligned.  Norm shifts are ignored
 * for RMSNorm and required for LayerNorm.  A NULL bias means "no bias".  Row-parallel biases
 * (b_o, b_fc2) are added once, after the partial sums (bias-dropout-add). */
typedef struct {
  const void *norm1_w, *norm1_b; /* [H]                 */
  const void *w_qkv, *b_qkv;     /* [q_w + 2 kv_w, H]   */
  const void *w_o, *b_o;         /* [H, q_w], [H]       */
  const void *norm2_w, *norm2_b; /* [H]                 */
  const void *w_fc1, *b_fc1;     /* [f1_r, H]           */
  const void *w_fc2, *b_fc2;     /* [H, f_r], [H]       */
} mt_weights;

/* Create a handle for one rank (tp_rank of tp_size) of a layer with the given full-model
 * shape ("ai阅读megatron", TransformerConfig fields hidden_size, num_attention_heads,
 * num_query_groups, kv_channels, ffn_hidden_size).  rope_base == 0 disables RoPE.
 * Supported: head_dim in {64, 128}; heads % query_groups == 0; heads, query_groups and ffn
 * divisible by tp_size; hidden % 8 == 0, hidden <= 8192; (ffn/tp_size) % 8 == 0.
 * Needs the current CUDA device to be sm_103 (GB300).  Host call; allocates about 16 MiB of
 * device memory (the error word, the RoPE frequencies and the K-split partial sums).  Returns
 * MT_ERR_UNSUPPORTED / MT_ERR_INVALID_ARG otherwise. */
int mt_layer_create(int hidden, int heads, int query_groups, int head_dim, int ffn, int norm, int act,
                    float rope_base, int tp_size, int tp_rank, mt_layer** out);

/* Norm epsilon (inside the square root); default 1e-5. */
int mt_layer_set_eps(mt_layer* L, float eps);

/* Device workspace needed for a call with this seq and batch (intermediates: normed input,
 * q/k/v in attention layout, attention output, h, normed h, MLP hidden, RoPE table, and
 * host-path staging for x and y). */
int mt_layer_workspace_bytes(const mt_layer* L, int seq, int batch, size_t* bytes);

/* Lend the library a device buffer of `bytes` (256-byte aligned) for the calls that follow.
 * The caller keeps ownership and must keep it alive while calls using it are in flight. */
int mt_layer_set_workspace(mt_layer* L, void* dev_ptr, size_t bytes);

/* Whole layer.  x [T, H] -> y_partial [T, H], in the order of the layer spec of "快速入门 /
 * Pai-Megatron-Patch 项目深度学习总结文档" §3.1 (input_layernorm, linear_qkv, core_attention with the
 * causal mask, linear_proj, bias-dropout-add, pre_mlp_layernorm, linear_fc1, linear_fc2,
 * bias-dropout-add), with the column/row splits of "Megatron-LM 深度学习与源码分析文档" Part 2 §2:
 *   tp_size == 1: y = h + fc2(act(fc1(norm2(h)))) + b_fc2, with h = x + o_proj(attn(norm1(x))) + b_o.
 *   tp_size  > 1: the all-reduce between the two blocks is replaced by the identity,
 *                 h = x + Y_attn,i + b_o, and y_partial = Y_mlp,i(h) is this rank's
 *                 pre-reduce row-parallel partial (no bias, no residual).
 * 7 kernel launches on `cuda_stream` (a cudaStream_t; NULL = legacy default stream): norm1 (which
 * also writes the RoPE table), QKV GEMM, attention, output projection, norm2, fc1, fc2. */
int mt_layer_forward(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* y_partial,
                     void* cuda_stream);

/* Attention block only: attn_out [T, H] = Y_attn,i, this rank's pre-reduce partial of the
 * output projection (no bias, no residual).  The caller sums the partials over ranks and
 * forms h = x + sum_i Y_attn,i + b_o ("Megatron-LM 深度学习与源码分析文档" Part 2 §2, Row Parallel). */
int mt_layer_forward_attn(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* attn_out,
                          void* cuda_stream);

/* MLP block only: y_partial [T, H] = Y_mlp,i(h), this rank's pre-reduce fc2 partial
 * (no bias, no residual); the caller forms y = h + sum_i Y_mlp,i + b_fc2. */
int mt_layer_forward_mlp(mt_layer* L, const void* h, int seq, int batch, const mt_weights* w, void* y_partial,
                         void* cuda_stream);

/* Packed variable-length samples ("快速入门 / Pai-Megatron-Patch 项目深度学习总结文档" §4.1 and §8,
 * sequence packing: several samples concatenated into one sequence, with cu_seqlens the cumulative
 * sample lengths [0, len1, len1+len2, ...] and attention kept inside each sample as FlashAttention's
 * variable-length form does).  x, y_partial: [total_tokens, H] (batch 1, samples back to back).
 * cu_seqlens: DEVICE array of num_seqs + 1 ints, cu[0] = 0, non-decreasing, cu[num_seqs] =
 * total_tokens; max_seqlen (host) bounds every sample's length (empty samples are allowed).
 * Sample i is tokens [cu[i], cu[i+1]): its queries see only its own earlier keys, and RoPE positions
 * restart at 0 in every sample, so each sample computes what it would alone.  Otherwise as
 * mt_layer_forward (TP semantics included).  Workspace: mt_layer_workspace_bytes_packed.
 * cu_seqlens that turn out inconsistent on the device are reported by mt_layer_status as
 * MT_ERR_INVALID_ARG (every access stays in bounds; the outputs are then invalid). */
int mt_layer_workspace_bytes_packed(const mt_layer* L, int total_tokens, int num_seqs, int max_seqlen, size_t* bytes);
int mt_layer_forward_packed(mt_layer* L, const void* x, int total_tokens, const int* cu_seqlens, int num_seqs,
                            int max_seqlen, const mt_weights* w, void* y_partial, void* cuda_stream);

/* ---- FP8 (E4M3) forward path -----------------------------------------------------------
 * The FP8 recipe of "ai阅读megatron" (--fp8-hybrid: E4M3 in the forward pass) and "快速入门"
 * §8.2 (dynamic scaling that tracks each tensor's amax over a history, amax_compute_algo max):
 * the four GEMMs take E4M3 operands.  A tensor with scale s is stored as codes of x * s (round to
 * nearest even, saturating to +-448) and the fp32 accumulator is multiplied by the two operands'
 * 1/s.  Weights use current scaling (s = 448 / amax, mt_quantize_e4m3).  The four activations that
 * feed the GEMMs -- normed x, the attention output, normed h, the MLP hidden -- use delayed
 * scaling: a forward quantises with the scales in the handle, records each activation's amax in
 * an amax history, and sets the next scales to 448 / max(history).  q/k/v, the attention, h and
 * y stay bf16. */
typedef struct {
  const void *w_qkv, *w_o, *w_fc1, *w_fc2;           /* E4M3 codes, shapes as in mt_weights       */
  const float *deq_qkv, *deq_o, *deq_fc1, *deq_fc2;  /* device: each weight's 1/scale             */
} mt_fp8_weights;

/* Allocate the handle's delayed-scaling state (host call): activation scales 1, an amax history
 * of amax_history_len entries per activation (1..65536; the pages' recipe uses 1024), zeroed. */
int mt_layer_fp8_enable(mt_layer* L, int amax_history_len);

/* Set the four activation scales (host array: normed x, attention output, normed h, MLP hidden;
 * positive, finite) and clear the history.  Synchronises the device. */
int mt_layer_fp8_set_scales(mt_layer* L, const float* scales);

/* Read the current activation scales and the amax each activation recorded in the last FP8
 * forward (host arrays of 4).  Synchronises the device. */
int mt_layer_fp8_state(mt_layer* L, float* scales, float* last_amax);

/* Whole layer with the four GEMMs on E4M3 (needs mt_layer_fp8_enable; hidden and ffn/tp_size
 * multiples of 16).  w supplies the bf16 norm weights and biases (its projection pointers are not
 * used); w8 the E4M3 projections.  Semantics, layouts and workspace as mt_layer_forward; 9 kernel
 * launches (the last updates the amax history). */
int mt_layer_forward_fp8(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w,
                         const mt_fp8_weights* w8, void* y_partial, void* cuda_stream);

/* Current per-tensor scaling of n bf16 values (n a multiple of 8): amax_deq[0] <- max |x| (as
 * float), amax_deq[1] <- 1/s with s = 448 / amax (s = 1 for an all-zero tensor), dst <- E4M3
 * codes of x * s.  src, dst, amax_deq: device (16/16/8-byte aligned).  Two launches. */
int mt_quantize_e4m3(const void* src, size_t n, void* dst, float* amax_deq, void* cuda_stream);

/* C[M, N] = (A[M, K] * B[N, K]^T) * (*deq_a) * (*deq_b) with E4M3 A and B, fp32 accumulation,
 * bf16 C (the FP8 layer's GEMM).  Device pointers; K % 16 == 0, N % 8 == 0. */
int mt_gemm_e4m3(const void* A, const void* B, void* C, int M, int N, int K, const float* deq_a, const float* deq_b,
                 void* cuda_stream);

/* mt_layer_forward with x and y in HOST memory: copies x into the workspace, runs the layer and
 * copies y back; `cuda_stream` reaches the end of the call once y is in host memory, and the host
 * buffers must stay valid until then.  With both buffers pinned and at least 512 tokens the copies
 * are overlapped with the layer on a copy stream owned by the handle: x arrives in row chunks (two,
 * up to four from 8192 tokens; norm1 and the QKV GEMM of a chunk run as soon as it is in) and the
 * fc2 GEMM runs per chunk (each chunk of y is copied back while the next is computed).  Pageable
 * buffers are copied before and after the layer. */
int mt_layer_forward_host(mt_layer* L, const void* x_host, int seq, int batch, const mt_weights* w,
                          void* y_host, void* cuda_stream);

/* ---- backward pass (tp_size == 1) ---------------------------------------------------------
 * Gradients of a scalar loss through the layer, given dL/dy (the pages' purpose is training:
 * the forward-backward step of "ai阅读megatron"'s training loop).  The forward intermediates are
 * recomputed first (full activation recompute, "快速入门" §8), then the chain rule runs through
 * the same readings as the forward.  All gradients are bf16 with fp32 accumulation inside. */
typedef struct { /* device pointers, shapes as in mt_weights; NULL = gradient not wanted */
  void *norm1_w, *norm1_b, *w_qkv, *b_qkv, *w_o, *b_o, *norm2_w, *norm2_b, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
} mt_grads;

/* Workspace the backward pass needs (a superset of the forward's: the forward intermediates, the
 * pre-activation fc1 output, gradient scratch in bf16, fp32 dq in head-major order and up to four
 * partial copies of fp32 dk/dv, the per-row softmax statistics, a head-major copy of dO and a bf16
 * V).  No [seq, seq] matrix is stored: the attention backward rebuilds the probabilities tile by
 * tile. */
int mt_layer_backward_workspace_bytes(const mt_layer* L, int seq, int batch, size_t* bytes);

/* dx [T, H] = dL/dx and the requested weight gradients, given x and dy = dL/dy [T, H].  Needs
 * tp_size == 1, seq % 8 == 0, hidden <= 8192 and a workspace of mt_layer_backward_workspace_bytes.  Asynchronous
 * on cuda_stream: the forward recomputed, then the GEMMs, elementwise kernels and the two
 * flash-attention backward kernels (dQ; dK and dV); the handle orders two streams of its own after
 * cuda_stream (the dQ kernel, and the weight gradients beside the chain of dx) and joins them back
 * into it before the call's work ends. */
int mt_layer_backward(mt_layer* L, const void* x, const void* dy, int seq, int batch, const mt_weights* w, void* dx,
                      const mt_grads* g, void* cuda_stream);

/* Training without the recompute (the level below activation checkpointing in the memory-saving
 * ladder of "快速入门" §10.3, which stores the activations instead of recomputing them):
 * mt_layer_forward_train computes y [T, H] exactly as mt_layer_forward (same kernels, the
 * same bits) and leaves the intermediates the gradients need in the workspace (of
 * mt_layer_backward_workspace_bytes); mt_layer_backward_saved then computes what mt_layer_backward
 * computes from them, without recomputing the forward.  Between the two calls the workspace must
 * not be used by another call of the handle, and x, seq, batch and the weights must be the same.
 * Same requirements and errors as mt_layer_backward. */
int mt_layer_forward_train(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* y,
                           void* cuda_stream);
int mt_layer_backward_saved(mt_layer* L, const void* x, const void* dy, int seq, int batch, const mt_weights* w,
                            void* dx, const mt_grads* g, void* cuda_stream);

/* Where an intermediate lives inside the workspace (for inspection in tests).  `which`:
 * 0 norm1 out [T,H]; 1 q [batch, nh_r, seq, d] after RoPE; 2 k [batch, ng_r, seq, d] after RoPE;
 * 3 v [batch, ng_r, seq, d] in fp16 (the attention's P V product runs on fp16 P and V, so |v|
 *   must stay below 65504);
 * 4 attention out [T, q_w]; 5 h [T,H]; 6 norm2 out [T,H]; 7 MLP hidden [T, f_r];
 * 8 RoPE table [seq, d/2] float2 (cos, sin). */
int mt_layer_workspace_region(const mt_layer* L, int seq, int batch, int which, size_t* offset, size_t* bytes);

/* Wait for the work this handle queued (the stream of its last call and its own copy stream;
 * other streams of the process are not waited for) and report a device-side failure recorded
 * since the last call (MT_ERR_DEVICE_TIMEOUT, or MT_ERR_INVALID_ARG for inconsistent packed
 * cu_seqlens), clearing it (and, after a failure, the K-split arrival counters, which a launch
 * that gave up may have left counted).  The error word is read through the handle's copy stream,
 * so no device-wide synchronisation happens.  Calls captured into a CUDA graph are not waited for:
 * synchronise the stream that launches the graph first.  Host call. */
int mt_layer_status(mt_layer* L);

/* Thread-local description of the last failure on this thread ("" after success). */
const char* mt_last_error(void);

void mt_layer_destroy(mt_layer* L);

/* Per-kernel timing.  Kernel slots: 0 the attention backward (its dQ and dK/dV kernels, which run
 * side by side on two streams, as one interval from before the first to after both; a launch
 * count of 1 per backward), 1 norm1 (with the RoPE table), 2 QKV GEMM, 3 attention,
 * 4 output-projection GEMM, 5 norm2, 6 fc1 GEMM, 7 fc2 GEMM (MT_PROFILE_SLOTS).  slot_mask selects
 * the slots whose launches this handle brackets with a pair of CUDA events on their stream (bit s
 * for slot s; MT_PROFILE_ALL for every slot, 0 to stop); values outside 0..MT_PROFILE_ALL return
 * MT_ERR_INVALID_ARG.  Each event pair costs a little time, so a caller timing whole steps
 * selects only the slots it needs.  Up to 8192 launches are kept.  mt_layer_profile_read waits for
 * the recorded events, writes per slot the number of launches and their summed milliseconds into
 * the caller's arrays (MT_PROFILE_SLOTS entries each) and clears the record. */
#define MT_PROFILE_SLOTS 8
#define MT_PROFILE_ALL ((1 << MT_PROFILE_SLOTS) - 1)
int mt_layer_profile_enable(mt_layer* L, int slot_mask);
int mt_layer_profile_read(mt_layer* L, int* launches, double* total_ms);

/* Number of kernels this handle has launched since it was created (every forward, backward and
 * staged call, profiled or not), written to *count.  MT_ERR_INVALID_ARG on NULL arguments. */
int mt_layer_launch_count(const mt_layer* L, unsigned long long* count);

/* ---- utility entry points (kernel-level; used by the parity tests) -------------------- */

/* C[M, N] = A[M, K] * B[N, K]^T in bf16 with fp32 accumulation, on the layer's tcgen05 GEMM
 * ("Megatron-LM 深度学习与源码分析文档" Part 2 §2, Y = XW with W stored [out, in]).
 * Device pointers, 16-byte aligned; K % 8 == 0 and N % 8 == 0. */
int mt_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, void* cuda_stream);

/* C[M, N] = A B^T as mt_gemm_bf16 with either operand stored transposed: a_layout 0 = A is [M, K]
 * row-major, 1 = A is [K, M] row-major (M contiguous); b_layout 0 = B is [N, K], 1 = B is [K, N].
 * The tcgen05 MMA reads a transposed operand directly (MN-major shared-memory tiles), the form the
 * backward pass uses for dW = dY^T X and dX = dY W.  Device pointers, 16-byte aligned; the contiguous
 * dimension of each operand and N must be multiples of 8 (MT_ERR_UNSUPPORTED otherwise);
 * MT_ERR_INVALID_ARG for NULL pointers, non-positive sizes or layouts other than 0 and 1. */
int mt_gemm_bf16_t(const void* A, int a_layout, const void* B, int b_layout, void* C, int M, int N, int K,
                   void* cuda_stream);

/* GEMM kernel choice for every later launch in the process (all handles): 0 automatic (the
 * default: pairs of CTAs sharing one M = 256 tcgen05.mma per 256 x 256 tile when M > 128, else one
 * CTA per 128 x 256 tile), 1 one CTA per tile always, 2 CTA pairs wherever M > 128 (the same as
 * 0 now; kept for the tests that force each kernel).  Both kernels compute the same fp32 sums in the same K
 * order.  A tuning and testing control; returns MT_ERR_INVALID_ARG for other values. */
int mt_gemm_set_pairing(int mode);

/* Attention kernel form for every later launch in the process (all handles): 0 automatic (the
 * default: one CTA takes two query heads of one kv group when the group serves an even number of
 * heads and those two-head CTAs number at least twice the SMs, or, at head_dim 64 with an odd
 * number of heads per group, two heads of two groups; otherwise one head per CTA), 1 one head per
 * CTA always, 2 two heads per CTA wherever a form allows it.  One or two heads of one group per
 * CTA give bit-identical outputs (each head's products and softmax are the same instructions in
 * the same order).  A tuning and testing control; returns MT_ERR_INVALID_ARG for other values. */
int mt_attn_set_heads_per_cta(int mode);

/* How the CTA-pair GEMM cuts the tiles of its last, partial wave, for every later launch in the
 * process: 0 automatic (the default): the GEMMs of a layer handle cut each tail tile into 2 to 4
 * ranges of K when the tail still fits in one wave of SM pairs and each range drops at least 16 K
 * blocks; the range holding the first K blocks waits (bounded) for the others' fp32 partial sums,
 * adds them in K order and runs the epilogue; elsewhere (and for the handle-less mt_gemm_* calls)
 * the tail tiles are cut into 2 or 4 pieces along N.  1: along N only.  The K ranges change the
 * fp32 summation order of the tail tiles (the results stay deterministic).  A tuning and testing
 * control; returns MT_ERR_INVALID_ARG for other values. */
int mt_gemm_set_tail_split(int mode);

/* How a GEMM launch of this library is planned, computed on the host without any CUDA call (a
 * testing and tuning aid): C[M, N] with the given epilogue (0 store, 1 residual add, 2 QKV with
 * RoPE and scatter (head_dim 64 or 128), 3 SwiGLU (N = the gate width), 4 GeLU), E4M3 operands
 * when fp8 != 0, as a layer handle's GEMMs (with_handle != 0: K ranges allowed for the tail) or
 * as the handle-less mt_gemm_* calls, on a device with `sms` SMs of which `pair_slots` CTA pairs
 * can be resident (152 and 76 on GB300), under the current mt_gemm_set_pairing and
 * mt_gemm_set_tail_split modes.  Writes plan[0..7] = {pair (1: CTA-pair kernel, 256-row tiles),
 * tiles_m, tiles_n, split (N pieces per tail tile), ksplit (K ranges per tail tile), full_units
 * (whole tiles before the tail), num_units, epi_split (epilogue warps per TMEM lane quadrant that
 * store a tile)}.  MT_ERR_INVALID_ARG for a NULL plan, non-positive sizes, another epilogue or
 * head_dim, or sms < 2, pair_slots outside 1 .. sms / 2. */
int mt_gemm_plan(int M, int N, int K, int epilogue, int head_dim, int fp8, int with_handle, int sms, int pair_slots,
                 int* plan);

/* Sequence-parallel epilogue of a row-parallel linear, for one rank's sequence slice
 * ("Megatron-LM 深度学习与源码分析文档" Part 2 §4 Sequence Parallel: after a RowParallel linear the
 * output is reduce-scattered back to sequence-sharded activations, and LayerNorm/dropout/residual
 * run on S/TP rows per rank; its kernel list names "RowParallel reduce-scatter fused add/norm").
 * On one GPU the ranks' partials are all local, so the reduce-scatter becomes a sum over them:
 * for the rows [row0, row0 + rows) of the [tokens, hidden] activations (rank r of p holds
 * row0 = r * tokens / p, rows = tokens / p: the [s, b, h] layout makes a sequence slice contiguous)
 *     h  = resid + sum_i partials[i] + bias      (fp32 sum; stored as bf16)
 *     hn = Norm(h)                                (statistics over the stored bf16 h)
 * partials: host array of num_partials (1..16) device pointers, each a full [tokens, hidden] bf16
 * pre-reduce partial (e.g. mt_layer_forward_attn outputs).  resid, h_out and hn_out are the slice
 * ([rows, hidden] bf16, device); bias [hidden] may be NULL; norm_w/norm_b as in mt_weights.
 * One kernel launch on cuda_stream; hidden % 8 == 0, hidden <= 8192. */
int mt_sp_reduce_add_norm(const void* const* partials, int num_partials, const void* resid, const void* bias,
                          const void* norm_w, const void* norm_b, int norm, float eps, int tokens, int hidden, int row0,
                          int rows, void* h_out, void* hn_out, void* cuda_stream);

/* Fault-detection self test: launches one CTA that waits on a barrier nothing will complete,
 * giving up after `limit_us` microseconds (1..1000000).  Returns MT_ERR_DEVICE_TIMEOUT when the
 * bounded wait fired and reported itself (the expected outcome), MT_OK if it did not fire. */
int mt_selftest_bounded_wait(int limit_us);

/* ---- allocation-free variant ------------------------------------------------------------ */

/* The whole-layer forward of mt_layer_create + mt_layer_forward in one call that allocates no
 * device memory.  The Megatron pages have no counterpart to this call: it is here for callers
 * that cannot call cudaMalloc -- code that runs inside a host framework whose allocator owns all
 * device memory, and real-time or embedded callers that forbid device allocation (and the device
 * synchronisation cudaMalloc/cudaFree can imply) once they have started.
 *
 * Same arguments, layouts and results as mt_layer_create(...) followed by mt_layer_set_eps(eps)
 * and mt_layer_forward(x, seq, batch, w, y_partial, cuda_stream).  The caller passes x, the
 * weights and y_partial as usual.  The scratch (the layer workspace, the RoPE frequency table and
 * the device error word) lives in one fixed area of MT_STATIC_AREA_BYTES (32 MiB) compiled into
 * the library: every GPU on which the library is used holds it until the process exits.  A call
 * whose workspace would not fit in it (mt_layer_workspace_bytes > MT_STATIC_AREA_BYTES - 1024,
 * e.g. more than about 370 tokens of the Llama-3-8B-shaped layer) returns MT_ERR_UNSUPPORTED and does
 * nothing.  No cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the area's device address (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  The address is kept per
 * device and CUDA context: after cudaDeviceReset (a new context) the next call looks it up again,
 * so that call too should come before any stream capture.  Every call first launches a one-CTA
 * set-up kernel on cuda_stream that clears the error word and writes the RoPE frequencies (passed
 * as kernel arguments), then the layer's kernels.  All calls share the one area, which keeps the
 * last call's contents: calls whose work overlaps on the GPU (other streams, other host threads)
 * race and corrupt each other's results.  Device-side timeouts are recorded in the area's error
 * word (cleared at the start of each call), which mt_layer_forward_static_status reads. */
#define MT_STATIC_AREA_BYTES (32u << 20)
int mt_layer_forward_static(int hidden, int heads, int query_groups, int head_dim, int ffn, int norm, int act,
                            float rope_base, int tp_size, int tp_rank, float eps, const void* x, int seq, int batch,
                            const mt_weights* w, void* y_partial, void* cuda_stream);

/* Outcome of the last mt_layer_forward_static call on this device: waits for the work queued on
 * cuda_stream (the stream that call used), then reads the static area's error word with one
 * device-to-host copy into host stack memory (no allocation).  MT_ERR_DEVICE_TIMEOUT when a kernel
 * of that call gave up on a bounded barrier wait (its outputs are invalid), MT_OK otherwise.  The
 * word is cleared by the next static call, not by this one. */
int mt_layer_forward_static_status(void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* MT_LAYER_H */
