// Host-side declarations shared by the translation units of the layer library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mt {

using bf16 = __nv_bfloat16;

// Epilogue of the tcgen05 GEMM (what happens to each fp32 accumulator row before it is stored).
enum GemmEpilogue : int {
  kEpiStore = 0,   // out = acc (+ bias)
  kEpiResid = 1,   // out = acc (+ bias) + resid            (row-parallel output + bias-dropout-add)
  kEpiQkv = 2,     // bias, RoPE on q/k heads, scatter q/k to [b, head, s, d] and v (fp16) to [b, group, s, d]
  kEpiSwiglu = 3,  // out = silu(gate + b_gate) * (up + b_up); the tile holds 128 gate and 128 up columns
  kEpiGelu = 4,    // out = gelu_tanh(acc + bias)
};

struct GemmParams {
  int M, N, K;        // output rows, output columns (SwiGLU: gate width), reduction length
  int tiles_m, tiles_n, num_tiles;
  int b_row_step;     // SwiGLU: row offset of the up half of W (the gate width); unused otherwise
  // Tile order (rasterisation): tiles come in bands of `band` m-tiles (band_m = 1, m fastest
  // inside a band) or `band` n-tiles (band_m = 0, n fastest), so a band's operand stays in L2.
  int band, band_m;
  // Work units: [0, full_units) are whole tiles; the tiles after them (the last, partial wave)
  // are cut into `split` pieces along N, or (CTA pairs with a K-split workspace) into `ksplit`
  // ranges of K, so that the tail wave is shorter.  num_units in total.
  int full_units, split, num_units;
  // K-split tail (pair kernel): the unit holding K range 0 of a tail tile stores the tile; the
  // others write fp32 partial sums to kws and count them on kflags, which that unit waits for,
  // adds in K order and resets to zero.  kws: [tail tile][ksplit - 1][CTA 2][quadrant 4]
  // [32-column chunk 8][8][lane 32] float4; kflags: [tail tile][CTA 2][quadrant 4][epilogue part 2].
  int ksplit;
  float4* kws;
  int* kflags;
  // CTA pairs (pair = 1): tiles are 256 x 256 and computed by a cluster of two CTAs sharing one
  // M = 256 MMA (tiles_m counts 256-row tiles); otherwise one CTA per 128 x 256 tile.
  int pair;
  // epilogue warps per TMEM lane quadrant that store a tile (1 or 2): 2 where the epilogue would
  // otherwise pace the GEMM (a short main loop per tile, or a single wave of tiles)
  int epi_split;
  // Operand layouts (bf16 only): a_mn = 1 when A is stored [K, M] (M contiguous) instead of [M, K];
  // b_mn = 1 when B is stored [K, N] instead of [N, K].  The tensor maps then hold 64 x 64 boxes
  // (64 M or N elements by 64 K rows) and the MMA reads the tiles MN-major.  Plain stores only.
  int a_mn, b_mn;
  bf16* out;
  int ldo;
  const bf16* bias;   // [N] (SwiGLU: [2N]) or null
  const bf16* resid;  // [M, ldr] or null
  int ldr;
  // kEpiQkv only
  bf16 *q, *k;
  __half* v;           // fp16: the P V product of the attention takes fp16 P
  const float2* rope;  // [positions, d/2] (cos, sin) or null
  int seq, batch, head_dim, q_w, kv_w, nh, ng;
  // packed samples (batch 1): per-token RoPE position; null for dense batches
  const int* pos;
  int row0;            // token row of the launch's first A row (a launch over a chunk of the rows)
  // E4M3 operands: the fp32 accumulator is multiplied by (*deq_a) * (*deq_b); null for bf16
  const float* deq_a;
  const float* deq_b;
  // E4M3 output of the SwiGLU / GeLU epilogue: codes of out * (*q_scale) go to out8 (pitch ldo
  // bytes) instead of `out`, and max |out| is folded into *amax (float bits)
  uint8_t* out8;
  const float* q_scale;
  unsigned* amax;
  // kEpiStore only: fp32 output to out32 (pitch ldo) instead of bf16; acc32 = 1 adds to it
  float* out32;
  int acc32;
  // SwiGLU / GeLU epilogue with bf16 output: when non-null, the pre-activation values (bias added,
  // rounded to bf16) also go to pre (pitch ldp): SwiGLU as [gate N | up N], GeLU as N columns
  bf16* pre;
  int ldp;
  // bf16 output of the store / residual / GeLU / SwiGLU epilogues through the output tensor map
  // (boxes of 32 rows x 32 columns staged in shared memory and written by TMA) instead of per-thread
  // stores
  int tma_out;
  // kEpiStore with bf16 output only: the tile is stored transposed, C[m][n] at out[n * ldo + m]
  // (computing X^T = B A^T lets the MMA read both operands in their faster layouts)
  int c_trans;
  // B is a weight that no kernel of the stream writes: the pair kernel issues the first stages' B
  // loads before it waits for the previous kernel (programmatic dependent launch)
  int b_static;
  int* err;
};

struct AttnParams {
  int seq, batch, nh, ng;  // this rank's query heads and kv groups
  int num_qb;              // ceil(seq / 128); packed samples: ceil(max_seqlen / 128)
  // Packed samples (batch 1, seq = all tokens): sample i is tokens [cu[i], cu[i+1]), rows
  // [cu[i], cu[i+1]) of q, k and v.  null for dense batches.
  const int* cu;
  int num_seqs;
  float scale_log2;        // log2(e) / sqrt(head_dim)
  bf16* o;                 // [seq*batch, ldo], head h at columns h*head_dim
  int ldo;
  // E4M3 output instead of o: codes of o * (*q_scale), pitch ldo bytes; max |o| into *amax
  uint8_t* o8;
  const float* q_scale;
  unsigned* amax;
  // when set (dense batches): log2 of each query row's softmax denominator in the base-2 units of
  // the kernel, lse[(b * nh + h) * seq + s] = m + log2(l), so P = 2^(S * scale_log2 - lse)
  float* lse;
  int* err;
};

// Attention backward (dense batches): from the forward's lse and D = rowsum(dO o O) (both
// [b * nh + h][seq] fp32), fp32 dq [b * nh + h][seq][d] and dk, dv [b * ng + g][seq][d].
struct AttnBwdParams {
  int seq, batch, nh, ng;
  int num_qb;                // ceil(seq / 128)
  float scale, scale_log2;   // 1 / sqrt(d) and log2(e) / sqrt(d)
  const float* lse;
  const float* dsum;
  float *dq, *dk, *dv;
  int* err;
  // dK/dV: the (head, query block) steps of every (key block, kv group) are cut into kv_parts
  // (1..kMaxKvParts) equal runs on separate CTAs; run r writes its partial sums to dk and dv +
  // r * part_stride floats, which the caller adds
  int kv_parts;
  size_t part_stride;
};
constexpr int kMaxKvParts = 4;

// Sequence-parallel epilogue (see mt_sp_reduce_add_norm).
constexpr int kMaxSpParts = 16;
struct SpParams {
  const bf16* parts[kMaxSpParts];  // full [T, H] row-parallel partials
  int nparts;
  size_t row0;                     // first row of the slice inside the partials
  int rows, H;
  const bf16* resid;               // [rows, H]
  const bf16* bias;                // [H] or null
  const bf16 *gamma, *beta;        // [H]; beta only for LayerNorm
  float eps;
  bf16 *h, *hn;                    // [rows, H]
};

// Launch with programmatic stream serialization (the kernel may start while the previous kernel of
// the stream finishes; the kernels of this library wait for it with griddepcontrol.wait before
// touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Number of SMs of the current device (cached).
int num_sms();
// Clusters of two GEMM CTAs that can be resident at once on the current device (cached; at most
// num_sms() / 2): the persistent grid of the CTA-pair GEMM.
int gemm_pair_slots();

// Kernel launchers; return a cudaError_t from the launch.
// fp8 = true: A and B are E4M3 (tensor maps of bytes, boxes 128 wide).
// Attention backward: maps = {Q, dO, K, V as 128-row boxes; Q, dO as 64-row boxes} (bf16,
// 64-element inner boxes, head-major [z][seq][d] tensors).  The dK/dV kernel goes on `st`, then the
// dQ kernel on `st_dq`; the two read the same inputs and write disjoint outputs, so on two streams
// the dQ blocks fill the SMs that the causally uneven dK/dV blocks leave idle.  The caller orders
// `st_dq` after the inputs' producers and joins it back (st_dq may be st).
cudaError_t launch_attention_bwd(int head_dim, const CUtensorMap* maps, const AttnBwdParams& p, cudaStream_t st,
                                 cudaStream_t st_dq);
// Batched copy of R x C bf16 slices z = 0..Z-1 at src + (z / zdiv) sb + (z % zdiv) sh (row pitch sp)
// into dst + z R dp (row pitch dp).
cudaError_t launch_head_slices(const bf16* src, size_t sp, size_t sb, size_t sh, int zdiv, int Z, bf16* dst, size_t dp,
                               int R, int C, cudaStream_t st);
// Dsum[(b nh + h) S + s] = dO[s b, h] . O[s b, h] over the head's d columns.
cudaError_t launch_row_dot(const bf16* dO, const bf16* O, float* Dsum, int S, int B, int nh, int d, cudaStream_t st);

// tmO: the bf16 output [M, N] (pitch ldo) in 32 x 32 boxes with the 64-byte swizzle, read only when p.tma_out;
// tmR: the residual [M, N] (pitch ldr) in the same boxes, read only when p.tma_out in the residual mode.
cudaError_t launch_gemm(int mode, bool fp8, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB64,
                        const CUtensorMap& tmO, const CUtensorMap& tmR, const GemmParams& p, cudaStream_t stream);
size_t gemm_smem_bytes();

cudaError_t launch_attention(int head_dim, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, cudaStream_t stream);
// mt_attn_set_heads_per_cta's mode for every later launch_attention (0, 1 or 2; checked by the caller).
void set_attention_heads_mode(int mode);

// RoPE table rows written by a norm launch: the CTA of row r writes table row row0 + r when it is
// below `rows` ((cos, sin) of s * theta_i, i < half).  The caller's norm launches must cover rows
// [0, rows) before the table is read.
struct RopeRows {
  float2* tab;
  const double* theta;
  int rows, half, row0;
};

// y8 != null: E4M3 output y * (*q_scale) into y8, max |y| folded into *amax.  rope != null: the
// launch also writes RoPE table rows (see RopeRows).
cudaError_t launch_norm(bool layer_norm, const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int hidden,
                        float eps, cudaStream_t stream, uint8_t* y8 = nullptr, const float* q_scale = nullptr,
                        unsigned* amax = nullptr, const RopeRows* rope = nullptr);

// Current per-tensor scaling of n (multiple of 8) bf16 values: slot[0] <- amax (float bits),
// slot[1] <- 1/scale, q <- E4M3 codes of x * 448 / amax.
cudaError_t launch_quantize_e4m3(const bf16* x, size_t n, uint8_t* q, float* slot, cudaStream_t stream);

// ---- backward pass (backward_kernels.cu)
cudaError_t launch_act_bwd(const bf16* u, const bf16* da, bf16* du, size_t T, int f, bool swiglu, cudaStream_t st);
// dx of a norm (plus `add`), and per-CTA partial rows of d gamma (rows [0, norm_bwd_blocks(T)) of
// `partial`, pitch H) and, for LayerNorm, of d beta (the next norm_bwd_blocks(T) rows).
int norm_bwd_blocks(int T);
cudaError_t launch_norm_bwd(const bf16* dy, const bf16* x, const bf16* gamma, const bf16* add, bf16* out,
                            float* partial, int T, int H, float eps, bool layer_norm, cudaStream_t st);
cudaError_t launch_colsum(const void* src, bool f32, size_t ld, int T, int N, float* acc, bf16* out, cudaStream_t st);
// dst[i] = bf16(src[i]) for n elements, n a multiple of 8, 16-byte aligned pointers.
cudaError_t launch_f16_to_bf16(const __half* src, bf16* dst, size_t n, cudaStream_t st);
// dst [C, R] (pitch dp) = src [R, C] (pitch sp)^T, bf16; R, C and the pitches multiples of 8, 16-byte
// aligned pointers (cudaErrorInvalidValue otherwise).
cudaError_t launch_transpose_bf16(const bf16* src, size_t sp, bf16* dst, size_t dp, int R, int C, cudaStream_t st);
// dqkv [T, (nh + 2 ng) d] bf16 from head-major fp32 dq, dk, dv (dk and dv the sums of `parts`
// partial buffers part_stride floats apart), with RoPE's rotation undone on the q and k heads.
cudaError_t launch_rope_bwd_pack(const float* dq, const float* dk, const float* dv, int parts, size_t part_stride,
                                 const float2* rope, bf16* dqkv, int S, int B, int nh, int ng, int d, cudaStream_t st);

// Delayed-scaling update after an FP8 forward (state layout: see fp8_history_kernel).
cudaError_t launch_fp8_history(float* state, int len, int pos, cudaStream_t stream);


cudaError_t launch_sp_add_norm(bool layer_norm, const SpParams& p, cudaStream_t stream);

// Per-token RoPE position of packed samples; invalid cu_seqlens record MT_ERR_INVALID_ARG in *err
// and give in-range positions.
cudaError_t launch_packed_index(const int* cu, int num_seqs, int tokens, int max_seqlen, int* pos, int* err,
                                cudaStream_t stream);

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace mt
