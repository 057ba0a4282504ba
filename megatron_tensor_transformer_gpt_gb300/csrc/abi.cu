// C ABI of the layer library: handle, argument checks, workspace layout, TMA descriptors and
// the kernel sequence of one layer forward on the caller's stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mt_layer.h"
#include "internal.h"

using mt::bf16;

// K-split tails of the CTA-pair GEMM: at most kKsTiles tail tiles and kKsSlots partial sums of
// 256 x 256 fp32 per launch (a tail of r tiles cut into s K ranges stores r (s - 1) of them).  One
// set: only the GEMMs of the caller's stream cut K (the backward's weight-gradient GEMMs, on a stream
// of their own, cut their tails along N), so no two launches share it at once.  The range holding a
// tail tile's first K blocks waits for the other ranges; their CTAs may start late while a
// weight-gradient GEMM holds SMs, but that GEMM waits on nothing outside its own CTAs, so they start.
constexpr int kKsSlots = 64, kKsTiles = 64;

struct mt_layer {
  int hidden, heads, groups, head_dim, ffn, norm, act, tp, rank;
  float rope_base, eps;
  int nh_r, ng_r, f_r, f1_r, q_w, kv_w;
  int device;
  int* d_err;       // device error word (mt_status code of the first device-side failure)
  double* d_theta;  // [head_dim/2] RoPE frequencies base^(-2i/d), or null
  void* ws;
  size_t ws_bytes;
  // FP8 delayed scaling (mt_layer_fp8_*): device state scale[4] | deq[4] | amax bits[4] | pad[4] |
  // history[4][f8_len] for the activations (normed x, attention output, normed h, MLP hidden)
  float* d_f8;
  int f8_len, f8_pos;
  // per-kernel timing (mt_layer_profile_*)
  int profile_mask;  // bit s: bracket the launches of kernel slot s with events
  unsigned long long launch_count;  // kernels launched by this handle (mt_layer_launch_count)
  struct Rec {
    int slot;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  // host-buffer forward: a copy stream and its events (created on first use); the backward also
  // runs its dQ kernel there, between a fork and a join event
  cudaStream_t copy_stream;
  cudaEvent_t copy_ev[9];
  cudaEvent_t fork_ev, join_ev;
  // the backward's weight-gradient GEMMs: a stream of their own (created on first use), forked from
  // the caller's stream where each one's operands are ready and joined back at the end
  cudaStream_t dw_stream;
  cudaEvent_t dw_fork, dw_join;
  // K-split tails of the CTA-pair GEMM: partial sums (kKsSlots slots of 256 x 256 fp32) and
  // arrival counters (kept at zero between launches)
  float4* d_kws;
  int* d_kflags;
  // recorded on the caller's stream at the end of every call that queues work (mt_layer_status
  // waits for it instead of the whole device)
  cudaEvent_t done_ev;
  bool done_pending;
};

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return MT_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MT_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Successful end of a call that queued work on `st`: marks the point mt_layer_status waits for.
// A call captured into a CUDA graph marks nothing (its work runs when the graph is launched).
int done(mt_layer* L, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();  // the legacy stream cannot be queried while another stream captures
    return ok();
  }
  if (cap != cudaStreamCaptureStatusNone) return ok();
  cudaError_t e = cudaEventRecord(L->done_ev, st);
  if (e != cudaSuccess) return cuda_fail(e, "recording the end of the call");
  L->done_pending = true;
  return ok();
}

enum Slot { kSlotAttnBwd = 0, kSlotNorm1, kSlotQkv, kSlotAttn, kSlotO, kSlotNorm2, kSlotFc1, kSlotFc2 };
constexpr size_t kMaxRecords = 8192;

cudaEvent_t pool_event(mt_layer* L) {
  if (!L->pool.empty()) {
    cudaEvent_t e = L->pool.back();
    L->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Counts one kernel launch of the handle and brackets it with events when its slot is profiled.
struct Timed {
  mt_layer* L;
  cudaStream_t st;
  bool on;
  cudaEvent_t a = nullptr;
  int slot;
  Timed(mt_layer* l, int s, cudaStream_t stream)
      : L(l), st(stream), on(l != nullptr && s >= 0 && s < MT_PROFILE_SLOTS && ((l->profile_mask >> s) & 1) && l->recs.size() < kMaxRecords), slot(s) {
    if (l != nullptr) ++l->launch_count;
    if (on) {
      a = pool_event(L);
      cudaEventRecord(a, st);
    }
  }
  ~Timed() {
    if (on) {
      cudaEvent_t b = pool_event(L);
      cudaEventRecord(b, st);
      L->recs.push_back({slot, a, b});
    }
  }
};

// Counts a kernel launch that no profiling slot covers.
void count_launch(mt_layer* L) {
  if (L != nullptr) ++L->launch_count;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Page-locked host memory (copies from and to it run asynchronously, overlapped with kernels).
bool pinned(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error of an unknown pointer
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// The handle's copy stream and its events, created on first use.
int ensure_copy_stream(mt_layer* L) {
  if (L->copy_stream != nullptr) return MT_OK;
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "creating the copy stream");
  auto make = [&](cudaEvent_t& ev) {
    if (ev == nullptr && e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  };
  for (auto& ev : L->copy_ev) make(ev);
  make(L->fork_ev);
  make(L->join_ev);
  if (e != cudaSuccess) {
    cudaStreamDestroy(s);
    return cuda_fail(e, "creating the copy events");
  }
  L->copy_stream = s;
  return MT_OK;
}

// The stream of the backward's weight-gradient GEMMs and its two events, created on first use.
int ensure_dw_stream(mt_layer* L) {
  if (L->dw_stream != nullptr) return MT_OK;
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess && L->dw_fork == nullptr) e = cudaEventCreateWithFlags(&L->dw_fork, cudaEventDisableTiming);
  if (e == cudaSuccess && L->dw_join == nullptr) e = cudaEventCreateWithFlags(&L->dw_join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    if (s != nullptr) cudaStreamDestroy(s);
    return cuda_fail(e, "creating the weight-gradient stream");
  }
  L->dw_stream = s;
  return MT_OK;
}

// ------------------------------------------------------------------ workspace layout
enum Region { kXn = 0, kQ, kK, kV, kO, kH, kHn, kA, kRope, kXStage, kYStage, kPos, kNumRegions };

struct Layout {
  size_t off[kNumRegions];
  size_t size[kNumRegions];
  size_t total;
};

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace of one call: S x B tokens; a RoPE table of `rope_rows` positions; `index_tokens`
// per-token positions (packed samples only).
Layout make_layout(const mt_layer* L, int S, int B, int rope_rows, int index_tokens) {
  Layout lay{};
  const size_t T = static_cast<size_t>(S) * B;
  const size_t d = L->head_dim;
  lay.size[kXn] = T * L->hidden * 2;
  lay.size[kQ] = static_cast<size_t>(B) * L->nh_r * S * d * 2;
  lay.size[kK] = static_cast<size_t>(B) * L->ng_r * S * d * 2;
  lay.size[kV] = static_cast<size_t>(B) * L->ng_r * S * d * 2;
  lay.size[kO] = T * L->q_w * 2;
  lay.size[kH] = T * L->hidden * 2;
  lay.size[kHn] = T * L->hidden * 2;
  lay.size[kA] = T * L->f_r * 2;
  lay.size[kRope] = L->rope_base > 0.f ? static_cast<size_t>(rope_rows) * (d / 2) * sizeof(float2) : 0;
  lay.size[kXStage] = T * L->hidden * 2;
  lay.size[kYStage] = T * L->hidden * 2;
  lay.size[kPos] = static_cast<size_t>(index_tokens) * sizeof(int);
  // q, k and v back to back (their sizes are multiples of 16 bytes), so that the QKV epilogue can
  // write all three through one [heads][tokens][d] tensor map at batch 1
  size_t o = 0;
  for (int r = 0; r < kNumRegions; ++r) {
    lay.off[r] = o;
    o = (r == kQ || r == kK) ? o + lay.size[r] : round_up(o + lay.size[r], 1024);
  }
  lay.total = o;
  return lay;
}

Layout layout_for(const mt_layer* L, int S, int B) {
  return make_layout(L, S, B, S, 0);
}

// Packed samples: batch 1, T tokens.
Layout layout_packed(const mt_layer* L, int T, int max_seqlen) { return make_layout(L, T, 1, max_seqlen, T); }

// Packed-sample description of a call (null for dense batches).
struct Packed {
  const int* cu;  // device, num_seqs + 1 entries
  int num_seqs, max_seqlen;
};

template <typename T>
T* region(const mt_layer* L, const Layout& lay, Region r) {
  return reinterpret_cast<T*>(static_cast<char*>(L->ws) + lay.off[r]);
}

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major bf16 matrix [rows, cols] with `pitch` elements per row; box = 64 columns x box_rows.
int map_2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t pitch, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled (2d %llu x %llu) failed: %d",
                                     (unsigned long long)rows, (unsigned long long)cols, (int)r);
  return MT_OK;
}

// A GEMM's bf16 output [rows, cols] with `pitch` elements per row, written by TMA stores of 32 x 32 boxes
// staged in shared memory with the 64-byte swizzle.
int map_out(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t pitch) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled (output %llu x %llu) failed: %d",
                                     (unsigned long long)rows, (unsigned long long)cols, (int)r);
  return MT_OK;
}

// q, k and v of a batch-1 call as one bf16 tensor [heads][tokens][d] (the heads of q, then of k,
// then of v: the QKV GEMM's column order), for TMA stores of 32-token x 32-column boxes.
int map_qkv_out(CUtensorMap* m, const void* q, uint64_t d, uint64_t tokens, uint64_t heads) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {d, tokens, heads};
  const cuuint64_t strides[2] = {d * 2, tokens * d * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled (qkv output) failed: %d", (int)r);
  return MT_OK;
}

// Sets up the TMA output of a GEMM whose epilogue writes bf16 `out` (store, residual, GeLU, SwiGLU).
int prepare_out(mt::GemmParams& p, int mode, CUtensorMap* to) {
  p.tma_out = (mode != mt::kEpiQkv && p.out != nullptr && p.out8 == nullptr && p.out32 == nullptr) ? 1 : 0;
  if (!p.tma_out) return MT_OK;
  // a transposed store writes an [N, M] output: rows are the tile's columns
  return p.c_trans ? map_out(to, p.out, p.M, p.N, p.ldo) : map_out(to, p.out, p.N, p.M, p.ldo);
}

// Row-major E4M3 (byte) matrix [rows, cols], pitch in bytes; box = 128 columns x box_rows.
int map_2d_u8(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t pitch, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled (e4m3 %llu x %llu) failed: %d",
                                     (unsigned long long)rows, (unsigned long long)cols, (int)r);
  return MT_OK;
}

// bf16 tensor [d2][d1][d0] with element pitches p1 (between d1 rows) and p2 (between d2 slabs);
// box = 64 x box1 x 1.
int map_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t p1, uint64_t p2,
           uint32_t box1) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {p1 * 2, p2 * 2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled (3d) failed: %d", (int)r);
  return MT_OK;
}

mt::GemmParams gemm_params(int M, int N, int K, bool swiglu, int* err) {
  mt::GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + 127) / 128;
  p.tiles_n = swiglu ? (N + 127) / 128 : (N + 255) / 256;
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.b_row_step = swiglu ? N : 0;
  p.err = err;
  return p;
}

// Which GEMM kernel runs (mt_gemm_set_pairing): 0 automatic, 1 one CTA per tile always,
// 2 CTA pairs wherever M > 128.
std::atomic<int> g_pairing{0};
// How the last partial wave of a CTA-pair GEMM is cut (mt_gemm_set_tail_split): 0 automatic
// (along K where a handle provides the partial-sum space and K is long enough, else along N),
// 1 along N only.
std::atomic<int> g_tail{0};

// Kernel, tile order and tail split of one GEMM (see GemmParams).
//   Kernel: CTA pairs (256 x 256 tiles) when M > 128, also below one wave of them on the SM
//   pairs; one CTA per 128 x 256 tile otherwise.
//   Order: if one operand fits in about 56 MB of the 129 MB L2 it is kept resident (the other is
//   streamed once); otherwise bands of m-tiles (or n-tiles) of about 56 MB, whichever streams
//   fewer bytes from DRAM.
//   Split: the tiles of the last partial wave are cut into pieces that still fit in one wave.  CTA
//   pairs with a handle: into 2 to 4 ranges of K, each at least 16 K blocks shorter than the whole
//   tile (a unit's main loop runs at about the same rate per K block whatever its width, so only
//   shorter K shortens the tail; the partial sums cost one fp32 write and read of the tile per
//   extra range).  Otherwise into 2 or 4 pieces along N (QKV pieces keep whole heads; a CTA stages at
//   least 64 B rows, the smallest TMA box used).
// The planning itself, for a device with `sms` SMs of which `pair_slots` CTA pairs can be resident;
// ksplit_ok: the GEMM has a handle's partial-sum space (no CUDA call here).
void plan_gemm_on(mt::GemmParams& p, int mode, int head_dim, bool ksplit_ok, bool fp8, int sms, int pair_slots) {
  const int tiles_m2 = (p.M + 255) / 256;
  const int mode_pairs = g_pairing.load();
  // CTA pairs for every GEMM with more than 128 rows: measured as fast or faster than the one-CTA
  // kernel on every layer shape, also below one wave of clusters (GPT-345M fc2: 64 pair tiles, 35 us
  // against 39 us)
  p.pair = mode_pairs != 1 && p.M > 128 ? 1 : 0;
  if (p.pair) {
    p.tiles_m = tiles_m2;
    p.num_tiles = p.tiles_m * p.tiles_n;
  }
  const double budget = 56.0 * 1024 * 1024;
  const double a_tile = (p.pair ? 256.0 : 128.0) * p.K * 2, b_tile = 256.0 * p.K * 2;
  const double a_all = a_tile * p.tiles_m, b_all = b_tile * p.tiles_n;
  if (a_all <= budget) {
    p.band_m = 1;
    p.band = p.tiles_m;
  } else if (b_all <= budget) {
    p.band_m = 0;
    p.band = p.tiles_n;
  } else {
    const int gm = std::max(1, static_cast<int>(budget / a_tile));
    const int gn = std::max(1, static_cast<int>(budget / b_tile));
    const double tm = a_all + b_all * ((p.tiles_m + gm - 1) / gm);
    const double tn = b_all + a_all * ((p.tiles_n + gn - 1) / gn);
    p.band_m = tm <= tn ? 1 : 0;
    p.band = tm <= tn ? std::min(gm, p.tiles_m) : std::min(gn, p.tiles_n);
  }
  const int workers = p.pair ? pair_slots : sms;
  const int waves = p.num_tiles / workers;
  const int rest = p.num_tiles - waves * workers;
  // pairs: each CTA stages half of a piece's B rows (SwiGLU: all of its gate or up rows)
  int max_split = p.pair ? 2 : 4;
  if (mode == mt::kEpiSwiglu) max_split = 2;
  if (mode == mt::kEpiQkv) max_split = std::min(max_split, std::max(1, 256 / head_dim));
  p.split = 1;
  p.ksplit = 1;
  p.kws = nullptr;
  p.kflags = nullptr;
  const int num_kb = (p.K + (fp8 ? 127 : 63)) / (fp8 ? 128 : 64);
  if (p.pair && ksplit_ok && g_tail.load() == 0 && rest > 0)
    for (int s = 4; s >= 2; --s)
      if (rest * s <= workers && rest * (s - 1) <= kKsSlots && rest <= kKsTiles && num_kb - num_kb / s >= 16) {
        p.ksplit = s;
        break;
      }
  if (p.ksplit == 1)
    for (int s = max_split; s >= 2; s /= 2)
      if (rest > 0 && rest * s <= workers) {
        p.split = s;
        break;
      }
  const int pieces = p.ksplit > 1 ? p.ksplit : p.split;
  p.full_units = pieces > 1 ? waves * workers : p.num_tiles;
  p.num_units = p.full_units + (pieces > 1 ? rest * pieces : 0);
  // two epilogue warps per quadrant where the epilogue would pace the GEMM: a short main loop per
  // tile (K <= 2048), at most one tile per CTA, or a K-split tail with K <= 4096 (its first range
  // adds the partial sums before the epilogue); one elsewhere (measured faster for long K)
  p.epi_split = (p.K <= 2048 || p.num_units <= workers || (p.ksplit > 1 && p.K <= 4096)) ? 2 : 1;
}

void plan_gemm(mt::GemmParams& p, int mode, int head_dim, const mt_layer* L, bool fp8, bool cut_k = true) {
  const bool ksplit_ok = cut_k && L != nullptr && L->d_kws != nullptr;
  const int sms = mt::num_sms();
  // the resident-pair query only where the pair kernel can be chosen (as the planner decides it)
  const int pair_slots = (g_pairing.load() != 1 && p.M > 128) ? mt::gemm_pair_slots() : std::max(1, sms / 2);
  plan_gemm_on(p, mode, head_dim, ksplit_ok, fp8, sms, pair_slots);
  if (p.ksplit > 1) {
    p.kws = L->d_kws;
    p.kflags = L->d_kflags;
  }
}

// One GEMM: A [M, K] (pitch lda) x W [rows_w, K]^T with the given epilogue.
// fp8: A and W hold E4M3 codes (lda and the W pitch K in bytes).  qkv_out (QKV epilogue at batch 1):
// the tensor map of q, k, v as one [heads][tokens][d] tensor, written by TMA stores.
int run_gemm(mt_layer* L, int slot, int mode, const void* A, int lda, const void* W, int rows_w, int M, int N, int K,
             mt::GemmParams p, cudaStream_t st, bool fp8 = false, const CUtensorMap* qkv_out = nullptr) {
  CUtensorMap ta, tb, tb64;
  auto mk = fp8 ? map_2d_u8 : map_2d;
  int rc = mk(&ta, A, K, M, lda, 128);
  if (rc) return rc;
  rc = mk(&tb, W, K, rows_w, K, 128);
  if (rc) return rc;
  rc = mk(&tb64, W, K, rows_w, K, 64);
  if (rc) return rc;
  plan_gemm(p, mode, mode == mt::kEpiQkv ? p.head_dim : 0, L, fp8);
  CUtensorMap to = ta, tr = ta;
  if ((rc = prepare_out(p, mode, &to))) return rc;
  if (mode == mt::kEpiQkv && qkv_out != nullptr) {
    to = *qkv_out;
    p.tma_out = 1;
  }
  if (p.tma_out && mode == mt::kEpiResid && (rc = map_out(&tr, p.resid, p.N, p.M, p.ldr))) return rc;
  // a layer's GEMMs take the weights as B, which no kernel of the layer writes; the handle-less calls
  // may multiply by the output of the kernel just before them
  p.b_static = L != nullptr ? 1 : 0;
  cudaError_t e;
  {
    Timed t(L, slot, st);
    e = mt::launch_gemm(mode, fp8, ta, tb, tb64, to, tr, p, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
  return MT_OK;
}

int check_weights(const mt_layer* L, const mt_weights* w, bool attn, bool mlp) {
  if (w == nullptr) return fail(MT_ERR_INVALID_ARG, "weights struct is NULL");
  struct {
    const void* p;
    const char* name;
    bool required;
  } items[] = {
      {w->norm1_w, "norm1_w", attn},
      {w->norm1_b, "norm1_b", attn && L->norm == MT_NORM_LAYER},
      {w->w_qkv, "w_qkv", attn},
      {w->b_qkv, "b_qkv", false},
      {w->w_o, "w_o", attn},
      {w->b_o, "b_o", false},
      {w->norm2_w, "norm2_w", mlp},
      {w->norm2_b, "norm2_b", mlp && L->norm == MT_NORM_LAYER},
      {w->w_fc1, "w_fc1", mlp},
      {w->b_fc1, "b_fc1", false},
      {w->w_fc2, "w_fc2", mlp},
      {w->b_fc2, "b_fc2", false},
  };
  for (auto& it : items) {
    if (it.required && it.p == nullptr) return fail(MT_ERR_INVALID_ARG, "weight %s is NULL", it.name);
    if (it.p != nullptr && !aligned16(it.p)) return fail(MT_ERR_INVALID_ARG, "weight %s is not 16-byte aligned", it.name);
  }
  return MT_OK;
}

int check_call(const mt_layer* L, const void* in, const void* out, int S, int B, Layout* lay) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (in == nullptr || out == nullptr) return fail(MT_ERR_INVALID_ARG, "input or output pointer is NULL");
  if (!aligned16(in) || !aligned16(out)) return fail(MT_ERR_INVALID_ARG, "input/output must be 16-byte aligned");
  if (S <= 0 || B <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive (got %d, %d)", S, B);
  if (static_cast<long long>(S) * B > (1LL << 30)) return fail(MT_ERR_UNSUPPORTED, "seq*batch too large");
  *lay = layout_for(L, S, B);
  if (L->ws == nullptr) return fail(MT_ERR_NO_WORKSPACE, "no workspace set (need %zu bytes)", lay->total);
  if (L->ws_bytes < lay->total)
    return fail(MT_ERR_NO_WORKSPACE, "workspace has %zu bytes, this call needs %zu", L->ws_bytes, lay->total);
  return MT_OK;
}

// ------------------------------------------------------------------ the two blocks
// Token rows in n chunks [row[c], row[c + 1]) (boundaries at multiples of 256): on input, the rows of
// chunk c are ready once event ev[c] has been reached (a copy on another stream); on output, the rows
// of chunk c are final at event ev[c], recorded on the compute stream.
constexpr int kMaxChunks = 4;
struct Chunks {
  int n;
  int row[kMaxChunks + 1];
  cudaEvent_t ev[kMaxChunks];
};

// Attention block: norm1 -> QKV GEMM (+bias, RoPE, scatter) -> flash attention -> output projection.
// out_mode kEpiStore writes the rank's partial; kEpiResid writes h = x + Y + b_o.  in != null: norm1
// and the QKV GEMM run per input chunk, each after its rows have arrived.
int run_attention_block(mt_layer* L, const Layout& lay, const void* x, int S, int B, const mt_weights* w, void* out,
                        int out_mode, cudaStream_t st, const Packed* pk = nullptr, float* lse = nullptr,
                        const Chunks* in = nullptr) {
  const int T = S * B, H = L->hidden, d = L->head_dim;
  cudaError_t e;
  // The RoPE table (positions 0 .. seq or max_seqlen, never more than the T token rows) is written
  // by the norm1 launches, row by row, before the QKV GEMMs read it.
  float2* rope = L->rope_base > 0.f ? region<float2>(L, lay, kRope) : nullptr;
  mt::RopeRows rope_rows{rope, L->d_theta, pk ? pk->max_seqlen : S, d / 2, 0};
  int* pos = nullptr;
  if (pk != nullptr) {
    pos = region<int>(L, lay, kPos);
    count_launch(L);
    e = mt::launch_packed_index(pk->cu, pk->num_seqs, T, pk->max_seqlen, pos, L->d_err, st);
    if (e != cudaSuccess) return cuda_fail(e, "packed-sample index");
  }
  bf16* xn = region<bf16>(L, lay, kXn);
  bf16 *q = region<bf16>(L, lay, kQ), *k = region<bf16>(L, lay, kK);
  __half* v = region<__half>(L, lay, kV);
  const int nqkv = L->q_w + 2 * L->kv_w;
  mt::GemmParams p;
  int rc;
  CUtensorMap tqkv;
  const bool qkv_tma = B == 1;  // q, k, v rows are then the token rows
  if (qkv_tma && (rc = map_qkv_out(&tqkv, q, d, S, static_cast<uint64_t>(L->nh_r) + 2 * L->ng_r))) return rc;
  const int nchunks = in != nullptr ? in->n : 1;
  for (int c = 0; c < nchunks; ++c) {
    const int r0 = in != nullptr ? in->row[c] : 0, rows = in != nullptr ? in->row[c + 1] - r0 : T;
    if (in != nullptr && (e = cudaStreamWaitEvent(st, in->ev[c], 0)) != cudaSuccess)
      return cuda_fail(e, "waiting for the input rows");
    const size_t off = static_cast<size_t>(r0) * H;
    {
      Timed t(L, kSlotNorm1, st);
      rope_rows.row0 = r0;
      e = mt::launch_norm(L->norm == MT_NORM_LAYER, static_cast<const bf16*>(x) + off,
                          static_cast<const bf16*>(w->norm1_w), static_cast<const bf16*>(w->norm1_b), xn + off, rows,
                          H, L->eps, st, nullptr, nullptr, nullptr, rope != nullptr ? &rope_rows : nullptr);
    }
    if (e != cudaSuccess) return cuda_fail(e, "norm1 launch");
    p = gemm_params(rows, nqkv, H, false, L->d_err);
    p.bias = static_cast<const bf16*>(w->b_qkv);
    p.q = q;
    p.k = k;
    p.v = v;
    p.rope = rope;
    p.seq = S;
    p.batch = B;
    p.head_dim = d;
    p.q_w = L->q_w;
    p.kv_w = L->kv_w;
    p.nh = L->nh_r;
    p.ng = L->ng_r;
    p.pos = pos;
    p.row0 = r0;
    if ((rc = run_gemm(L, kSlotQkv, mt::kEpiQkv, xn + off, H, w->w_qkv, nqkv, rows, nqkv, H, p, st, false,
                       qkv_tma ? &tqkv : nullptr)))
      return rc;
  }

  CUtensorMap tq, tk, tv;
  if ((rc = map_3d(&tq, q, d, S, static_cast<uint64_t>(B) * L->nh_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  if ((rc = map_3d(&tk, k, d, S, static_cast<uint64_t>(B) * L->ng_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  if ((rc = map_3d(&tv, v, d, S, static_cast<uint64_t>(B) * L->ng_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  bf16* o = region<bf16>(L, lay, kO);
  mt::AttnParams ap{};
  ap.seq = S;
  ap.batch = B;
  ap.nh = L->nh_r;
  ap.ng = L->ng_r;
  ap.num_qb = ((pk ? pk->max_seqlen : S) + 127) / 128;
  ap.cu = pk ? pk->cu : nullptr;
  ap.num_seqs = pk ? pk->num_seqs : 0;
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  ap.o = o;
  ap.ldo = L->q_w;
  ap.lse = lse;
  ap.err = L->d_err;
  {
    Timed t(L, kSlotAttn, st);
    e = mt::launch_attention(d, tq, tk, tv, ap, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");

  p = gemm_params(T, H, L->q_w, false, L->d_err);
  p.out = static_cast<bf16*>(out);
  p.ldo = H;
  if (out_mode == mt::kEpiResid) {
    p.bias = static_cast<const bf16*>(w->b_o);
    p.resid = static_cast<const bf16*>(x);
    p.ldr = H;
  }
  return run_gemm(L, kSlotO, out_mode, o, L->q_w, w->w_o, H, T, H, L->q_w, p, st);
}

// MLP block: norm2 -> fc1 GEMM (+bias, SwiGLU / GeLU) -> fc2 GEMM.
// out_mode kEpiStore writes the rank's partial; kEpiResid writes y = h + Y + b_fc2.  out_chunks !=
// null: fc2 runs per output chunk and records the chunk's event after it.
int run_mlp_block(mt_layer* L, const Layout& lay, const void* h, int S, int B, const mt_weights* w, void* out,
                  int out_mode, cudaStream_t st, const Chunks* out_chunks = nullptr) {
  const int T = S * B, H = L->hidden;
  bf16* hn = region<bf16>(L, lay, kHn);
  cudaError_t e;
  {
    Timed t(L, kSlotNorm2, st);
    e = mt::launch_norm(L->norm == MT_NORM_LAYER, static_cast<const bf16*>(h),
                                  static_cast<const bf16*>(w->norm2_w), static_cast<const bf16*>(w->norm2_b), hn, T,
                                  H, L->eps, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "norm2 launch");
  bf16* a = region<bf16>(L, lay, kA);
  const bool swiglu = L->act == MT_ACT_SWIGLU;
  mt::GemmParams p = gemm_params(T, L->f_r, H, swiglu, L->d_err);
  p.out = a;
  p.ldo = L->f_r;
  p.bias = static_cast<const bf16*>(w->b_fc1);
  int rc = run_gemm(L, kSlotFc1, swiglu ? mt::kEpiSwiglu : mt::kEpiGelu, hn, H, w->w_fc1, L->f1_r, T, L->f_r, H, p, st);
  if (rc) return rc;
  const int nchunks = out_chunks != nullptr ? out_chunks->n : 1;
  for (int c = 0; c < nchunks; ++c) {
    const int r0 = out_chunks != nullptr ? out_chunks->row[c] : 0;
    const int rows = out_chunks != nullptr ? out_chunks->row[c + 1] - r0 : T;
    p = gemm_params(rows, H, L->f_r, false, L->d_err);
    p.out = static_cast<bf16*>(out) + static_cast<size_t>(r0) * H;
    p.ldo = H;
    if (out_mode == mt::kEpiResid) {
      p.bias = static_cast<const bf16*>(w->b_fc2);
      p.resid = static_cast<const bf16*>(h) + static_cast<size_t>(r0) * H;
      p.ldr = H;
    }
    if ((rc = run_gemm(L, kSlotFc2, out_mode, a + static_cast<size_t>(r0) * L->f_r, L->f_r, w->w_fc2, H, rows, H,
                       L->f_r, p, st)))
      return rc;
    if (out_chunks != nullptr && (e = cudaEventRecord(out_chunks->ev[c], st)) != cudaSuccess)
      return cuda_fail(e, "recording an output chunk");
  }
  return MT_OK;
}

int forward_device(mt_layer* L, const Layout& lay, const void* x, int S, int B, const mt_weights* w, void* y,
                   cudaStream_t st, const Packed* pk = nullptr, const Chunks* in = nullptr,
                   const Chunks* out_chunks = nullptr) {
  bf16* h = region<bf16>(L, lay, kH);
  int rc = run_attention_block(L, lay, x, S, B, w, h, mt::kEpiResid, st, pk, nullptr, in);
  if (rc) return rc;
  return run_mlp_block(L, lay, h, S, B, w, y, L->tp == 1 ? mt::kEpiResid : mt::kEpiStore, st, out_chunks);
}

// The layer with its four GEMMs on E4M3 operands (delayed scaling of the activations, weights
// pre-quantised by the caller).  Same semantics as forward_device otherwise.
int forward_device_fp8(mt_layer* L, const Layout& lay, const void* x, int S, int B, const mt_weights* w,
                       const mt_fp8_weights* w8, void* y, cudaStream_t st) {
  const int T = S * B, H = L->hidden, d = L->head_dim;
  float* scale = L->d_f8;
  float* deq = L->d_f8 + 4;
  unsigned* amax = reinterpret_cast<unsigned*>(L->d_f8 + 8);
  cudaError_t e;
  float2* rope = L->rope_base > 0.f ? region<float2>(L, lay, kRope) : nullptr;  // rows written by norm1
  const mt::RopeRows rope_rows{rope, L->d_theta, S, d / 2, 0};
  uint8_t* xn8 = region<uint8_t>(L, lay, kXn);
  {
    Timed t(L, kSlotNorm1, st);
    e = mt::launch_norm(L->norm == MT_NORM_LAYER, static_cast<const bf16*>(x), static_cast<const bf16*>(w->norm1_w),
                        static_cast<const bf16*>(w->norm1_b), nullptr, T, H, L->eps, st, xn8, scale + 0, amax + 0,
                        rope != nullptr ? &rope_rows : nullptr);
  }
  if (e != cudaSuccess) return cuda_fail(e, "norm1 launch");
  bf16 *q = region<bf16>(L, lay, kQ), *k = region<bf16>(L, lay, kK);
  __half* v = region<__half>(L, lay, kV);
  const int nqkv = L->q_w + 2 * L->kv_w;
  mt::GemmParams p = gemm_params(T, nqkv, H, false, L->d_err);
  p.bias = static_cast<const bf16*>(w->b_qkv);
  p.q = q;
  p.k = k;
  p.v = v;
  p.rope = rope;
  p.seq = S;
  p.batch = B;
  p.head_dim = d;
  p.q_w = L->q_w;
  p.kv_w = L->kv_w;
  p.nh = L->nh_r;
  p.ng = L->ng_r;
  p.deq_a = deq + 0;
  p.deq_b = w8->deq_qkv;
  CUtensorMap tqkv;
  int rc = B == 1 ? map_qkv_out(&tqkv, q, d, S, static_cast<uint64_t>(L->nh_r) + 2 * L->ng_r) : MT_OK;
  if (rc) return rc;
  if ((rc = run_gemm(L, kSlotQkv, mt::kEpiQkv, xn8, H, w8->w_qkv, nqkv, T, nqkv, H, p, st, true,
                     B == 1 ? &tqkv : nullptr)))
    return rc;

  CUtensorMap tq, tk, tv;
  if ((rc = map_3d(&tq, q, d, S, static_cast<uint64_t>(B) * L->nh_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  if ((rc = map_3d(&tk, k, d, S, static_cast<uint64_t>(B) * L->ng_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  if ((rc = map_3d(&tv, v, d, S, static_cast<uint64_t>(B) * L->ng_r, d, static_cast<uint64_t>(S) * d, 128))) return rc;
  uint8_t* o8 = region<uint8_t>(L, lay, kO);
  mt::AttnParams ap{};
  ap.seq = S;
  ap.batch = B;
  ap.nh = L->nh_r;
  ap.ng = L->ng_r;
  ap.num_qb = (S + 127) / 128;
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  ap.ldo = L->q_w;
  ap.err = L->d_err;
  ap.o8 = o8;
  ap.q_scale = scale + 1;
  ap.amax = amax + 1;
  {
    Timed t(L, kSlotAttn, st);
    e = mt::launch_attention(d, tq, tk, tv, ap, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");

  bf16* h = region<bf16>(L, lay, kH);
  p = gemm_params(T, H, L->q_w, false, L->d_err);
  p.out = h;
  p.ldo = H;
  p.bias = static_cast<const bf16*>(w->b_o);
  p.resid = static_cast<const bf16*>(x);
  p.ldr = H;
  p.deq_a = deq + 1;
  p.deq_b = w8->deq_o;
  if ((rc = run_gemm(L, kSlotO, mt::kEpiResid, o8, L->q_w, w8->w_o, H, T, H, L->q_w, p, st, true))) return rc;

  uint8_t* hn8 = region<uint8_t>(L, lay, kHn);
  {
    Timed t(L, kSlotNorm2, st);
    e = mt::launch_norm(L->norm == MT_NORM_LAYER, h, static_cast<const bf16*>(w->norm2_w),
                        static_cast<const bf16*>(w->norm2_b), nullptr, T, H, L->eps, st, hn8, scale + 2, amax + 2);
  }
  if (e != cudaSuccess) return cuda_fail(e, "norm2 launch");
  uint8_t* a8 = region<uint8_t>(L, lay, kA);
  const bool swiglu = L->act == MT_ACT_SWIGLU;
  p = gemm_params(T, L->f_r, H, swiglu, L->d_err);
  p.ldo = L->f_r;
  p.bias = static_cast<const bf16*>(w->b_fc1);
  p.out8 = a8;
  p.q_scale = scale + 3;
  p.amax = amax + 3;
  p.deq_a = deq + 2;
  p.deq_b = w8->deq_fc1;
  if ((rc = run_gemm(L, kSlotFc1, swiglu ? mt::kEpiSwiglu : mt::kEpiGelu, hn8, H, w8->w_fc1, L->f1_r, T, L->f_r, H, p,
                     st, true)))
    return rc;
  p = gemm_params(T, H, L->f_r, false, L->d_err);
  p.out = static_cast<bf16*>(y);
  p.ldo = H;
  if (L->tp == 1) {
    p.bias = static_cast<const bf16*>(w->b_fc2);
    p.resid = h;
    p.ldr = H;
  }
  p.deq_a = deq + 3;
  p.deq_b = w8->deq_fc2;
  if ((rc = run_gemm(L, kSlotFc2, L->tp == 1 ? mt::kEpiResid : mt::kEpiStore, a8, L->f_r, w8->w_fc2, H, T, H, L->f_r,
                     p, st, true)))
    return rc;
  count_launch(L);
  e = mt::launch_fp8_history(L->d_f8, L->f8_len, L->f8_pos, st);
  if (e != cudaSuccess) return cuda_fail(e, "amax history update");
  L->f8_pos = (L->f8_pos + 1) % L->f8_len;
  return MT_OK;
}

// ------------------------------------------------------------------ backward pass (TP=1)
// Plain bf16 GEMM out[M, N] = A B^T with fp32 accumulation, to bf16 `out` or fp32 `out32` (acc32: add
// to it), pitch ldo.  A is stored [M, K] (a_mn = false) or [K, M] (a_mn = true), pitch lda; B is
// stored [N, K] (b_mn = false) or [K, N] (b_mn = true), pitch ldb.  L may be null (no error word,
// no launch count).
int gemm_ab(mt_layer* L, const void* A, size_t lda, bool a_mn, const void* Bm, size_t ldb, bool b_mn, int M, int N,
            int K, void* out, float* out32, size_t ldo, bool acc32, cudaStream_t st, bool c_trans = false,
            bool cut_k = true) {
  CUtensorMap ta, tb, tb64;
  int rc = a_mn ? map_2d(&ta, A, M, K, lda, 64) : map_2d(&ta, A, K, M, lda, 128);
  if (!rc) rc = b_mn ? map_2d(&tb, Bm, N, K, ldb, 64) : map_2d(&tb, Bm, K, N, ldb, 128);
  if (!rc) rc = b_mn ? map_2d(&tb64, Bm, N, K, ldb, 64) : map_2d(&tb64, Bm, K, N, ldb, 64);
  if (rc) return rc;
  mt::GemmParams p = gemm_params(M, N, K, false, L != nullptr ? L->d_err : nullptr);
  p.out = static_cast<bf16*>(out);
  p.out32 = out32;
  p.acc32 = acc32 ? 1 : 0;
  p.ldo = static_cast<int>(ldo);
  p.a_mn = a_mn ? 1 : 0;
  p.b_mn = b_mn ? 1 : 0;
  p.c_trans = c_trans && out32 == nullptr ? 1 : 0;
  plan_gemm(p, mt::kEpiStore, 0, L, false, cut_k);
  CUtensorMap to = ta;
  if ((rc = prepare_out(p, mt::kEpiStore, &to))) return rc;
  count_launch(L);
  cudaError_t e = mt::launch_gemm(mt::kEpiStore, false, ta, tb, tb64, to, ta, p, st);
  return e == cudaSuccess ? MT_OK : cuda_fail(e, "GEMM launch");
}

enum BwRegion {
  kBU = 0, kBA, kBDa, kBDu, kBDhn, kBDh, kBDo, kBDq, kBDk, kBDv, kBDqkv, kBDxn, kBGrow, kBAcc,
  kBLse, kBDsum, kBDoH, kBVh, kBT, kBNum
};

struct BwLayout {
  Layout fwd;
  size_t off[kBNum], size[kBNum], total;
};

// Runs the dK/dV kernel of the attention backward cuts each (key block, kv group) into: doubled
// while the grid has fewer CTAs than SMs and the shortest key block (the last, with the fewest
// query blocks) still has a step for every run.  With few kv groups (one TP rank of a GQA layer)
// the grid would otherwise leave most SMs idle; with enough CTAs a split only adds the partial
// sums' traffic (Llama-3-8B shape, 256 CTAs: the same time with two runs).
int kv_parts(const mt_layer* L, int S, int B) {
  const int nb = (S + 127) / 128, shortest = (L->nh_r / L->ng_r) * ((S + 63) / 64 - 2 * (nb - 1));
  const long ctas = static_cast<long>(nb) * B * L->ng_r;
  int parts = 1;
  while (2 * parts <= mt::kMaxKvParts && 2 * parts <= shortest && ctas * parts < mt::num_sms()) parts *= 2;
  return parts;
}

BwLayout bw_layout(const mt_layer* L, int S, int B) {
  BwLayout b{};
  b.fwd = layout_for(L, S, B);
  const size_t T = static_cast<size_t>(S) * B, H = L->hidden, d = L->head_dim;
  const size_t QKV = L->q_w + 2 * L->kv_w, f = L->f_r, f1 = L->f1_r, qw = L->q_w;
  const size_t maxc = std::max(std::max(QKV, f1), std::max(H, qw));
  b.size[kBU] = T * f1 * 2;
  b.size[kBA] = T * f * 2;
  b.size[kBDa] = T * f * 2;
  b.size[kBDu] = T * f1 * 2;
  b.size[kBDhn] = T * H * 2;
  b.size[kBDh] = T * H * 2;
  b.size[kBDo] = T * qw * 2;
  b.size[kBDq] = static_cast<size_t>(B) * L->nh_r * S * d * 4;
  // dK and dV: room for the most partial runs the attention backward may cut a key block into
  b.size[kBDk] = static_cast<size_t>(B) * L->ng_r * S * d * 4 * mt::kMaxKvParts;
  b.size[kBDv] = static_cast<size_t>(B) * L->ng_r * S * d * 4 * mt::kMaxKvParts;
  b.size[kBDqkv] = T * QKV * 2;
  b.size[kBDxn] = T * H * 2;
  b.size[kBGrow] = 2 * static_cast<size_t>(mt::norm_bwd_blocks(static_cast<int>(T))) * H * 4;  // norm partials
  b.size[kBAcc] = maxc * 4;
  // attention backward: row statistics, head-major dO and V
  const size_t zq = static_cast<size_t>(B) * L->nh_r, zk = static_cast<size_t>(B) * L->ng_r;
  b.size[kBLse] = zq * S * 4;
  b.size[kBDsum] = zq * S * 4;
  b.size[kBDoH] = zq * S * d * 2;
  b.size[kBVh] = zk * S * d * 2;
  // the transposed operand of a weight gradient: the smaller of X and dY, at most H columns (every
  // projection has H on one side)
  b.size[kBT] = T * H * 2;
  size_t o = b.fwd.total;
  for (int r = 0; r < kBNum; ++r) {
    b.off[r] = o;
    o = round_up(o + b.size[r], 1024);
  }
  b.total = o;
  return b;
}

template <typename T>
T* bwr(const mt_layer* L, const BwLayout& b, BwRegion r) {
  return reinterpret_cast<T*>(static_cast<char*>(L->ws) + b.off[r]);
}

// Gradients of one linear Y = X W^T (+ b) given dY (all bf16, dense):
//   dW [N, K] = dY^T X, db = column sums of dY, dX [M, K] = dY W (written to dx if not null).
// The weight gradient (its operand transpose and GEMM) runs on `sw` once dY and X are ready on `st`
// (sw may be st); the bias gradient and dX run on `st`.
int linear_bwd(mt_layer* L, const BwLayout& b, const void* dY, const void* X, const void* W, int M, int N, int K,
               void* dW, void* db, void* dX, cudaStream_t st, cudaStream_t sw) {
  int rc;
  // Y [M, N] = X [M, K] W[N, K]^T.  The GEMM reads an MN-major A at full rate and loses 12-14 % on an
  // MN-major B, so every product here takes its B K-major:
  //   dW = dY^T X with X^T [K, M] (one transpose) as B, dY read as an MN-major A; or, when dY is the
  //        narrower of the two, dW^T = X^T dY with dY^T [N, M] as B, stored transposed;
  //   dX = dY W formed as dX^T = W^T dY^T: W an MN-major A, dY a K-major B, stored transposed.
  if (dW != nullptr) {
    // the transpose buffer is used on `sw` only, so the weight gradients take it in turn
    bf16* tr = bwr<bf16>(L, b, kBT);
    const bool tx = K <= N;  // transpose X (else dY)
    const bool cut_k = sw == st;  // a K-cut tail's waits assume no other kernel of the handle runs beside it
    cudaError_t e = cudaSuccess;
    if (sw != st && ((e = cudaEventRecord(L->dw_fork, st)) != cudaSuccess ||
                     (e = cudaStreamWaitEvent(sw, L->dw_fork, 0)) != cudaSuccess))
      return cuda_fail(e, "weight-gradient fork");
    count_launch(L);
    e = tx ? mt::launch_transpose_bf16(static_cast<const bf16*>(X), K, tr, M, M, K, sw)
           : mt::launch_transpose_bf16(static_cast<const bf16*>(dY), N, tr, M, M, N, sw);
    if (e != cudaSuccess) return cuda_fail(e, "weight-gradient operand transpose");
    if ((rc = tx ? gemm_ab(L, dY, N, true, tr, M, false, N, K, M, dW, nullptr, K, false, sw, false, cut_k)
                 : gemm_ab(L, X, K, true, tr, M, false, K, N, M, dW, nullptr, K, false, sw, true, cut_k)))
      return rc;
  }
  if (db != nullptr) {
    count_launch(L);
    count_launch(L);  // the column sums, then their conversion to bf16
    cudaError_t e = mt::launch_colsum(dY, false, N, M, N, bwr<float>(L, b, kBAcc), static_cast<bf16*>(db), st);
    if (e != cudaSuccess) return cuda_fail(e, "bias gradient");
  }
  if (dX != nullptr && (rc = gemm_ab(L, W, K, true, dY, N, false, K, M, N, dX, nullptr, K, false, st, true))) return rc;
  return MT_OK;
}

int norm_bwd(mt_layer* L, const BwLayout& b, const void* dy, const void* x, const void* gamma, const void* add,
             void* out, void* dgamma, void* dbeta, int T, cudaStream_t st) {
  const int H = L->hidden;
  float* part = bwr<float>(L, b, kBGrow);  // per-CTA partial rows of d gamma, then of d beta
  const int nb = mt::norm_bwd_blocks(T);
  count_launch(L);
  cudaError_t e = mt::launch_norm_bwd(static_cast<const bf16*>(dy), static_cast<const bf16*>(x),
                                      static_cast<const bf16*>(gamma), static_cast<const bf16*>(add),
                                      static_cast<bf16*>(out), part, T, H, L->eps, L->norm == MT_NORM_LAYER, st);
  if (e == cudaSuccess && dgamma != nullptr) {
    count_launch(L);
    count_launch(L);  // the column sums, then their conversion to bf16
    e = mt::launch_colsum(part, true, H, nb, H, bwr<float>(L, b, kBAcc), static_cast<bf16*>(dgamma), st);
  }
  if (e == cudaSuccess && dbeta != nullptr && L->norm == MT_NORM_LAYER) {
    count_launch(L);
    count_launch(L);
    e = mt::launch_colsum(part + static_cast<size_t>(nb) * H, true, H, nb, H, bwr<float>(L, b, kBAcc),
                          static_cast<bf16*>(dbeta), st);
  }
  return e == cudaSuccess ? MT_OK : cuda_fail(e, "norm backward");
}

// The forward intermediates the gradients need, written into the backward workspace: xn, q, k
// (after RoPE), v, o, h (attention block, with each query row's log-sum-exp), hn, u (fc1's
// pre-activation output) and a.  The full-recompute backward runs this first; the training forward
// runs it (plus fc2) so that a later backward can skip it.
int forward_saving(mt_layer* L, const BwLayout& b, const void* x, int S, int B, const mt_weights* w, cudaStream_t st) {
  const Layout& lay = b.fwd;
  const int T = S * B, H = L->hidden, f = L->f_r, f1 = L->f1_r;
  const bool swiglu = L->act == MT_ACT_SWIGLU;
  int rc;
  bf16* h = region<bf16>(L, lay, kH);
  if ((rc = run_attention_block(L, lay, x, S, B, w, h, mt::kEpiResid, st, nullptr, bwr<float>(L, b, kBLse))))
    return rc;
  bf16* hn = region<bf16>(L, lay, kHn);
  count_launch(L);
  cudaError_t e = mt::launch_norm(L->norm == MT_NORM_LAYER, h, static_cast<const bf16*>(w->norm2_w),
                                  static_cast<const bf16*>(w->norm2_b), hn, T, H, L->eps, st);
  if (e != cudaSuccess) return cuda_fail(e, "norm2 launch");
  // fc1 with the forward's activation epilogue, which also keeps the pre-activation u
  mt::GemmParams p = gemm_params(T, f, H, swiglu, L->d_err);
  p.out = bwr<bf16>(L, b, kBA);
  p.ldo = f;
  p.bias = static_cast<const bf16*>(w->b_fc1);
  p.pre = bwr<bf16>(L, b, kBU);
  p.ldp = f1;
  return run_gemm(L, -1, swiglu ? mt::kEpiSwiglu : mt::kEpiGelu, hn, H, w->w_fc1, f1, T, f, H, p, st);
}

// The gradients from the intermediates forward_saving left in the workspace.
int backward_from_saved(mt_layer* L, const BwLayout& b, const void* x, const void* dy, int S, int B,
                        const mt_weights* w, void* dx, const mt_grads* g, cudaStream_t st) {
  const Layout& lay = b.fwd;
  const int T = S * B, H = L->hidden, d = L->head_dim, nh = L->nh_r, ng = L->ng_r;
  const int qw = L->q_w, kvw = L->kv_w, QKV = qw + 2 * kvw, f = L->f_r, f1 = L->f1_r;
  const bool swiglu = L->act == MT_ACT_SWIGLU;
  int rc;
  cudaError_t e;
  bf16* h = region<bf16>(L, lay, kH);
  bf16 *xn = region<bf16>(L, lay, kXn), *hn = region<bf16>(L, lay, kHn), *o = region<bf16>(L, lay, kO);
  bf16 *q = region<bf16>(L, lay, kQ), *k = region<bf16>(L, lay, kK);
  bf16 *u = bwr<bf16>(L, b, kBU), *a = bwr<bf16>(L, b, kBA);

  // ---- MLP
  bf16 *da = bwr<bf16>(L, b, kBDa), *du = bwr<bf16>(L, b, kBDu), *dhn = bwr<bf16>(L, b, kBDhn);
  bf16* dh = bwr<bf16>(L, b, kBDh);
  if ((rc = ensure_dw_stream(L))) return rc;
  cudaStream_t sw = L->dw_stream;  // the weight gradients' GEMMs, beside the chain of dX
  if ((rc = linear_bwd(L, b, dy, a, w->w_fc2, T, H, f, g->w_fc2, w->b_fc2 ? g->b_fc2 : nullptr, da, st, sw)))
    return rc;
  count_launch(L);
  if ((e = mt::launch_act_bwd(u, da, du, T, f, swiglu, st)) != cudaSuccess) return cuda_fail(e, "activation backward");
  if ((rc = linear_bwd(L, b, du, hn, w->w_fc1, T, f1, H, g->w_fc1, w->b_fc1 ? g->b_fc1 : nullptr, dhn, st, sw)))
    return rc;
  if ((rc = norm_bwd(L, b, dhn, h, w->norm2_w, dy, dh, g->norm2_w, g->norm2_b, T, st))) return rc;

  // ---- output projection
  bf16* dO = bwr<bf16>(L, b, kBDo);
  if ((rc = linear_bwd(L, b, dh, o, w->w_o, T, H, qw, g->w_o, w->b_o ? g->b_o : nullptr, dO, st, sw))) return rc;

  // ---- attention, flash-style: P and dS are rebuilt tile by tile from the row log-sum-exp the
  //      forward recompute wrote; fp32 dQ, dK, dV
  float *dq = bwr<float>(L, b, kBDq), *dk = bwr<float>(L, b, kBDk), *dv = bwr<float>(L, b, kBDv);
  float *lse = bwr<float>(L, b, kBLse), *dsum = bwr<float>(L, b, kBDsum);
  bf16 *dOh = bwr<bf16>(L, b, kBDoH), *Vh = bwr<bf16>(L, b, kBVh);
  const int zq = B * nh, zk = B * ng;
  const size_t sd = static_cast<size_t>(S) * d;
  int kvp = 1;  // partial dK/dV buffers the RoPE pack sums
  // dO head-major; V from the forward's head-major fp16 copy (the bf16 dO pairs with a bf16 V)
  count_launch(L);
  if ((e = mt::launch_head_slices(dO, static_cast<size_t>(B) * qw, static_cast<size_t>(qw), static_cast<size_t>(d),
                                  nh, zq, dOh, static_cast<size_t>(d), S, d, st)) != cudaSuccess)
    return cuda_fail(e, "attention backward operands");
  count_launch(L);
  if ((e = mt::launch_f16_to_bf16(region<__half>(L, lay, kV), Vh, static_cast<size_t>(zk) * sd, st)) != cudaSuccess)
    return cuda_fail(e, "attention backward operands");
  count_launch(L);
  if ((e = mt::launch_row_dot(dO, o, dsum, S, B, nh, d, st)) != cudaSuccess) return cuda_fail(e, "rowsum(dO o O)");
  {
    CUtensorMap m[6];
    const uint64_t Zq = zq, Zk = zk;
    if ((rc = map_3d(&m[0], q, d, S, Zq, d, sd, 128)) || (rc = map_3d(&m[1], dOh, d, S, Zq, d, sd, 128)) ||
        (rc = map_3d(&m[2], k, d, S, Zk, d, sd, 128)) || (rc = map_3d(&m[3], Vh, d, S, Zk, d, sd, 128)) ||
        (rc = map_3d(&m[4], q, d, S, Zq, d, sd, 64)) || (rc = map_3d(&m[5], dOh, d, S, Zq, d, sd, 64)))
      return rc;
    mt::AttnBwdParams ap{};
    ap.seq = S;
    ap.batch = B;
    ap.nh = nh;
    ap.ng = ng;
    ap.num_qb = (S + 127) / 128;
    ap.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    ap.lse = lse;
    ap.dsum = dsum;
    ap.dq = dq;
    ap.dk = dk;
    ap.dv = dv;
    ap.err = L->d_err;
    ap.kv_parts = kv_parts(L, S, B);
    ap.part_stride = static_cast<size_t>(zk) * sd;
    kvp = ap.kv_parts;
    // dQ on the copy stream beside dK/dV: fork after D = rowsum(dO o O), join before the RoPE pack
    if ((rc = ensure_copy_stream(L))) return rc;
    cudaStream_t cs = L->copy_stream;
    if ((e = cudaEventRecord(L->fork_ev, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs, L->fork_ev, 0)) != cudaSuccess)
      return cuda_fail(e, "attention backward fork");
    Timed t(L, kSlotAttnBwd, st);  // both kernels: from the fork to the join
    count_launch(L);
    if ((e = mt::launch_attention_bwd(d, m, ap, st, cs)) != cudaSuccess) return cuda_fail(e, "attention backward");
    if ((e = cudaEventRecord(L->join_ev, cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, L->join_ev, 0)) != cudaSuccess)
      return cuda_fail(e, "attention backward join");
  }
  bf16* dqkv = bwr<bf16>(L, b, kBDqkv);
  const float2* rope = L->rope_base > 0.f ? region<float2>(L, lay, kRope) : nullptr;
  count_launch(L);
  if ((e = mt::launch_rope_bwd_pack(dq, dk, dv, kvp, static_cast<size_t>(zk) * sd, rope, dqkv, S, B, nh, ng, d,
                                    st)) != cudaSuccess)
    return cuda_fail(e, "RoPE backward");

  // ---- QKV projection and the input norm
  bf16* dxn = bwr<bf16>(L, b, kBDxn);
  if ((rc = linear_bwd(L, b, dqkv, xn, w->w_qkv, T, QKV, H, g->w_qkv, w->b_qkv ? g->b_qkv : nullptr, dxn, st, sw)))
    return rc;
  if ((rc = norm_bwd(L, b, dxn, x, w->norm1_w, dh, dx, g->norm1_w, g->norm1_b, T, st))) return rc;
  if ((e = cudaEventRecord(L->dw_join, sw)) != cudaSuccess || (e = cudaStreamWaitEvent(st, L->dw_join, 0)) != cudaSuccess)
    return cuda_fail(e, "weight-gradient join");
  return MT_OK;
}

// Full activation recompute: the forward intermediates, then the gradients.
int backward_device(mt_layer* L, const BwLayout& b, const void* x, const void* dy, int S, int B, const mt_weights* w,
                    void* dx, const mt_grads* g, cudaStream_t st) {
  const int rc = forward_saving(L, b, x, S, B, w, st);
  return rc ? rc : backward_from_saved(L, b, x, dy, S, B, w, dx, g, st);
}

}  // namespace

namespace mt {
int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}
}  // namespace mt

// ====================================================================== exported C ABI
namespace {
// The checks shared by the backward and training-forward entry points (g may be NULL for the
// training forward, which takes y in place of dy and dx).
int check_train_call(mt_layer* L, const void* x, const void* dy, int seq, int batch, const mt_weights* w,
                     const void* dx, const mt_grads* g, bool need_grads, BwLayout* b) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (L->tp != 1) return fail(MT_ERR_UNSUPPORTED, "the backward pass is implemented for tp_size == 1");
  if (x == nullptr || dy == nullptr || dx == nullptr || (need_grads && g == nullptr))
    return fail(MT_ERR_INVALID_ARG, need_grads ? "x, dy, dx and grads must not be NULL" : "x and y must not be NULL");
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx)) return fail(MT_ERR_INVALID_ARG, "x/dy/dx/y must be 16-byte aligned");
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive");
  if (seq % 8) return fail(MT_ERR_UNSUPPORTED, "the backward pass needs seq % 8 == 0");
  if (L->hidden > 8192) return fail(MT_ERR_UNSUPPORTED, "the backward pass needs hidden <= 8192");
  if (need_grads) {
    const void* gp[] = {g->norm1_w, g->norm1_b, g->w_qkv, g->b_qkv, g->w_o, g->b_o,
                        g->norm2_w, g->norm2_b, g->w_fc1, g->b_fc1, g->w_fc2, g->b_fc2};
    for (const void* p : gp)
      if (p != nullptr && !aligned16(p)) return fail(MT_ERR_INVALID_ARG, "gradient buffers must be 16-byte aligned");
  }
  *b = bw_layout(L, seq, batch);
  if (L->ws == nullptr || L->ws_bytes < b->total)
    return fail(MT_ERR_NO_WORKSPACE, "the backward pass needs a workspace of %zu bytes", b->total);
  return check_weights(L, w, true, true);
}
}  // namespace

extern "C" {

int mt_layer_create(int hidden, int heads, int query_groups, int head_dim, int ffn, int norm, int act,
                    float rope_base, int tp_size, int tp_rank, mt_layer** out) {
  if (out == nullptr) return fail(MT_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (hidden <= 0 || heads <= 0 || query_groups <= 0 || head_dim <= 0 || ffn <= 0 || tp_size <= 0)
    return fail(MT_ERR_INVALID_ARG, "sizes must be positive");
  if (tp_rank < 0 || tp_rank >= tp_size) return fail(MT_ERR_INVALID_ARG, "tp_rank %d outside [0, %d)", tp_rank, tp_size);
  if (norm != MT_NORM_RMS && norm != MT_NORM_LAYER) return fail(MT_ERR_INVALID_ARG, "unknown norm %d", norm);
  if (act != MT_ACT_SWIGLU && act != MT_ACT_GELU_TANH) return fail(MT_ERR_INVALID_ARG, "unknown activation %d", act);
  if (!(rope_base >= 0.f) || std::isinf(rope_base)) return fail(MT_ERR_INVALID_ARG, "rope_base must be finite and >= 0");
  if (head_dim != 64 && head_dim != 128) return fail(MT_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", head_dim);
  if (heads % query_groups) return fail(MT_ERR_UNSUPPORTED, "heads %% query_groups != 0");
  if (heads % tp_size || query_groups % tp_size || ffn % tp_size)
    return fail(MT_ERR_UNSUPPORTED, "heads, query_groups and ffn must be divisible by tp_size");
  if (hidden % 8 || hidden > 8192) return fail(MT_ERR_UNSUPPORTED, "hidden must be a multiple of 8 and <= 8192");
  if ((ffn / tp_size) % 8) return fail(MT_ERR_UNSUPPORTED, "ffn/tp_size must be a multiple of 8");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(MT_ERR_UNSUPPORTED, "this library is built for sm_103 (GB300); device %d is sm_%d%d", dev, major, minor);

  mt_layer* L = new mt_layer{};
  L->hidden = hidden;
  L->heads = heads;
  L->groups = query_groups;
  L->head_dim = head_dim;
  L->ffn = ffn;
  L->norm = norm;
  L->act = act;
  L->tp = tp_size;
  L->rank = tp_rank;
  L->rope_base = rope_base;
  L->eps = 1e-5f;
  L->nh_r = heads / tp_size;
  L->ng_r = query_groups / tp_size;
  L->f_r = ffn / tp_size;
  L->f1_r = act == MT_ACT_SWIGLU ? 2 * L->f_r : L->f_r;
  L->q_w = L->nh_r * head_dim;
  L->kv_w = L->ng_r * head_dim;
  L->device = dev;
  e = cudaMalloc(&L->d_err, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(L->d_err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&L->d_kws, static_cast<size_t>(kKsSlots) * 256 * 256 * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&L->d_kflags, kKsTiles * 16 * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(L->d_kflags, 0, kKsTiles * 16 * sizeof(int));
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&L->done_ev, cudaEventDisableTiming);
  if (e == cudaSuccess && rope_base > 0.f) {
    const int half = head_dim / 2;
    double theta[64];
    for (int i = 0; i < half; ++i) theta[i] = std::pow(static_cast<double>(rope_base), -2.0 * i / head_dim);
    e = cudaMalloc(&L->d_theta, half * sizeof(double));
    if (e == cudaSuccess) e = cudaMemcpy(L->d_theta, theta, half * sizeof(double), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    mt_layer_destroy(L);
    return cuda_fail(e, "mt_layer_create allocation");
  }
  *out = L;
  return ok();
}

int mt_layer_set_eps(mt_layer* L, float eps) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (!(eps > 0.f) || std::isinf(eps)) return fail(MT_ERR_INVALID_ARG, "eps must be positive and finite");
  L->eps = eps;
  return ok();
}

int mt_layer_workspace_bytes(const mt_layer* L, int seq, int batch, size_t* bytes) {
  if (L == nullptr || bytes == nullptr) return fail(MT_ERR_INVALID_ARG, "handle or bytes is NULL");
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive");
  *bytes = layout_for(L, seq, batch).total;
  return ok();
}

int mt_layer_set_workspace(mt_layer* L, void* dev_ptr, size_t bytes) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (dev_ptr != nullptr && (reinterpret_cast<uintptr_t>(dev_ptr) & 255u))
    return fail(MT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  L->ws = dev_ptr;
  L->ws_bytes = dev_ptr ? bytes : 0;
  return ok();
}

int mt_layer_workspace_region(const mt_layer* L, int seq, int batch, int which, size_t* offset, size_t* bytes) {
  if (L == nullptr || offset == nullptr || bytes == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive");
  if (which < 0 || which > kRope) return fail(MT_ERR_INVALID_ARG, "unknown region %d", which);
  const Layout lay = layout_for(L, seq, batch);
  *offset = lay.off[which];
  *bytes = lay.size[which];
  return ok();
}

int mt_layer_forward(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* y_partial,
                     void* cuda_stream) {
  Layout lay;
  int rc = check_call(L, x, y_partial, seq, batch, &lay);
  if (rc) return rc;
  if ((rc = check_weights(L, w, true, true))) return rc;
  rc = forward_device(L, lay, x, seq, batch, w, y_partial, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_layer_forward_attn(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* attn_out,
                          void* cuda_stream) {
  Layout lay;
  int rc = check_call(L, x, attn_out, seq, batch, &lay);
  if (rc) return rc;
  if ((rc = check_weights(L, w, true, false))) return rc;
  rc = run_attention_block(L, lay, x, seq, batch, w, attn_out, mt::kEpiStore, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_layer_forward_mlp(mt_layer* L, const void* h, int seq, int batch, const mt_weights* w, void* y_partial,
                         void* cuda_stream) {
  Layout lay;
  int rc = check_call(L, h, y_partial, seq, batch, &lay);
  if (rc) return rc;
  if ((rc = check_weights(L, w, false, true))) return rc;
  rc = run_mlp_block(L, lay, h, seq, batch, w, y_partial, mt::kEpiStore, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_layer_workspace_bytes_packed(const mt_layer* L, int total_tokens, int num_seqs, int max_seqlen, size_t* bytes) {
  if (L == nullptr || bytes == nullptr) return fail(MT_ERR_INVALID_ARG, "handle or bytes is NULL");
  if (total_tokens <= 0 || num_seqs <= 0 || max_seqlen <= 0 || max_seqlen > total_tokens)
    return fail(MT_ERR_INVALID_ARG, "need total_tokens > 0, num_seqs > 0, 0 < max_seqlen <= total_tokens");
  *bytes = layout_packed(L, total_tokens, max_seqlen).total;
  return ok();
}

int mt_layer_forward_packed(mt_layer* L, const void* x, int total_tokens, const int* cu_seqlens, int num_seqs,
                            int max_seqlen, const mt_weights* w, void* y_partial, void* cuda_stream) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (x == nullptr || y_partial == nullptr || cu_seqlens == nullptr)
    return fail(MT_ERR_INVALID_ARG, "x, y_partial and cu_seqlens must not be NULL");
  if (!aligned16(x) || !aligned16(y_partial) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(MT_ERR_INVALID_ARG, "x/y must be 16-byte and cu_seqlens 4-byte aligned");
  if (total_tokens <= 0 || num_seqs <= 0 || max_seqlen <= 0 || max_seqlen > total_tokens)
    return fail(MT_ERR_INVALID_ARG, "need total_tokens > 0, num_seqs > 0, 0 < max_seqlen <= total_tokens");
  if (total_tokens > (1 << 30)) return fail(MT_ERR_UNSUPPORTED, "too many tokens");
  const Layout lay = layout_packed(L, total_tokens, max_seqlen);
  if (L->ws == nullptr || L->ws_bytes < lay.total)
    return fail(MT_ERR_NO_WORKSPACE, "workspace missing or smaller than the %zu bytes this call needs", lay.total);
  int rc = check_weights(L, w, true, true);
  if (rc) return rc;
  const Packed pk{cu_seqlens, num_seqs, max_seqlen};
  rc = forward_device(L, lay, x, total_tokens, 1, w, y_partial, static_cast<cudaStream_t>(cuda_stream), &pk);
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_layer_forward_host(mt_layer* L, const void* x_host, int seq, int batch, const mt_weights* w, void* y_host,
                          void* cuda_stream) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (x_host == nullptr || y_host == nullptr) return fail(MT_ERR_INVALID_ARG, "host buffers must not be NULL");
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive");
  Layout lay = layout_for(L, seq, batch);
  if (L->ws == nullptr || L->ws_bytes < lay.total)
    return fail(MT_ERR_NO_WORKSPACE, "workspace missing or smaller than %zu bytes", lay.total);
  int rc = check_weights(L, w, true, true);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  void* xd = region<void>(L, lay, kXStage);
  void* yd = region<void>(L, lay, kYStage);
  const size_t bytes = lay.size[kXStage];
  const int T = seq * batch;
  // Row chunks at multiples of the 256-row GEMM tile, about 1024 rows or more each (two to four).
  // The first input chunk's copy and the last output chunk's copy are not hidden, so smaller chunks
  // hide more, while every QKV or fc2 chunk below one wave of tiles still costs a whole tile time.
  // 4096 tokens on one box: two chunks 1.341-1.360 ms per step, four 1.292-1.314 ms, eight input
  // chunks (with four output chunks) 1.367-1.379 ms.
  const int n = T < 512 ? 1 : std::min(kMaxChunks, std::max(2, T / 1024));
  if (n > 1 && pinned(x_host) && pinned(y_host)) {
    // Overlap the copies with the layer: x arrives in n row chunks on the copy stream and norm1 + QKV
    // of chunk c run as soon as it is in; fc2 runs per chunk and each chunk of y is copied back while
    // the next is computed.  The stream `st` waits for the last copy.
    if ((rc = ensure_copy_stream(L))) return rc;
    cudaStream_t cs = L->copy_stream;
    cudaEvent_t* ev = L->copy_ev;  // start (then: copies done) | x chunks [n] | y chunks [n]
    Chunks in{n, {}, {}}, out{n, {}, {}};
    for (int c = 0; c <= n; ++c) in.row[c] = out.row[c] = c == n ? T : (c * (T / n)) / 256 * 256;
    for (int c = 0; c < n; ++c) {
      in.ev[c] = ev[1 + c];
      out.ev[c] = ev[1 + kMaxChunks + c];
    }
    const size_t row_bytes = static_cast<size_t>(L->hidden) * 2;
    const uint8_t* xs = static_cast<const uint8_t*>(x_host);
    uint8_t* ys = static_cast<uint8_t*>(y_host);
    uint8_t* xdb = static_cast<uint8_t*>(xd);
    uint8_t* ydb = static_cast<uint8_t*>(yd);
    cudaError_t e = cudaEventRecord(ev[0], st);  // the host buffers' earlier users on `st` come first
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[0], 0);
    for (int c = 0; c < n && e == cudaSuccess; ++c) {
      const size_t o = in.row[c] * row_bytes, nb = (in.row[c + 1] - in.row[c]) * row_bytes;
      e = cudaMemcpyAsync(xdb + o, xs + o, nb, cudaMemcpyHostToDevice, cs);
      if (e == cudaSuccess) e = cudaEventRecord(in.ev[c], cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of x");
    if ((rc = forward_device(L, lay, xd, seq, batch, w, yd, st, nullptr, &in, &out))) return rc;
    for (int c = 0; c < n && e == cudaSuccess; ++c) {
      const size_t o = out.row[c] * row_bytes, nb = (out.row[c + 1] - out.row[c]) * row_bytes;
      e = cudaStreamWaitEvent(cs, out.ev[c], 0);
      if (e == cudaSuccess) e = cudaMemcpyAsync(ys + o, ydb + o, nb, cudaMemcpyDeviceToHost, cs);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev[0], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[0], 0);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy of y");
    return done(L, st);
  }
  cudaError_t e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of x");
  rc = forward_device(L, lay, xd, seq, batch, w, yd, st);
  if (rc) return rc;
  e = cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy of y");
  return done(L, st);
}

int mt_layer_status(mt_layer* L) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  // wait for the handle's own work only: the end of its last call and its copy stream
  cudaError_t e = L->done_pending ? cudaEventSynchronize(L->done_ev) : cudaSuccess;
  if (e != cudaSuccess) return cuda_fail(e, "waiting for the handle's last call");
  L->done_pending = false;
  int rc = ensure_copy_stream(L);
  if (rc) return rc;
  cudaStream_t cs = L->copy_stream;
  int code = 0;
  e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&code, L->d_err, sizeof(int), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (code != 0) {
    // a launch that gave up may have left K-split arrivals counted: start the next one from zero
    e = cudaMemsetAsync(L->d_kflags, 0, kKsTiles * 16 * sizeof(int), cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->d_err, 0, sizeof(int), cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  }
  if (code == MT_ERR_INVALID_ARG)
    return fail(MT_ERR_INVALID_ARG, "cu_seqlens were found inconsistent on the device (not 0 .. total_tokens, "
                                    "decreasing, or a sample longer than max_seqlen); outputs are invalid");
  if (code != 0)
    return fail(MT_ERR_DEVICE_TIMEOUT, "a kernel stopped waiting on a barrier (device code %d); outputs are invalid",
                code);
  return ok();
}

const char* mt_last_error(void) { return g_last_error.c_str(); }

void mt_layer_destroy(mt_layer* L) {
  if (L == nullptr) return;
  if (L->d_err) cudaFree(L->d_err);
  if (L->d_theta) cudaFree(L->d_theta);
  if (L->d_f8) cudaFree(L->d_f8);
  if (L->d_kws) cudaFree(L->d_kws);
  if (L->d_kflags) cudaFree(L->d_kflags);
  for (auto& r : L->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : L->pool) cudaEventDestroy(e);
  for (auto e : L->copy_ev)
    if (e) cudaEventDestroy(e);
  if (L->fork_ev) cudaEventDestroy(L->fork_ev);
  if (L->join_ev) cudaEventDestroy(L->join_ev);
  if (L->copy_stream) cudaStreamDestroy(L->copy_stream);
  if (L->dw_fork) cudaEventDestroy(L->dw_fork);
  if (L->dw_join) cudaEventDestroy(L->dw_join);
  if (L->dw_stream) cudaStreamDestroy(L->dw_stream);
  if (L->done_ev) cudaEventDestroy(L->done_ev);
  delete L;
}

int mt_layer_profile_enable(mt_layer* L, int slot_mask) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (slot_mask < 0 || slot_mask > MT_PROFILE_ALL) return fail(MT_ERR_INVALID_ARG, "slot mask 0x%x out of range", slot_mask);
  L->profile_mask = slot_mask;
  return ok();
}

int mt_layer_launch_count(const mt_layer* L, unsigned long long* count) {
  if (L == nullptr || count == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  *count = L->launch_count;
  return ok();
}

int mt_layer_profile_read(mt_layer* L, int* launches, double* total_ms) {
  if (L == nullptr || launches == nullptr || total_ms == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  for (int i = 0; i < MT_PROFILE_SLOTS; ++i) {
    launches[i] = 0;
    total_ms[i] = 0.0;
  }
  int rc = MT_OK;
  for (auto& r : L->recs) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess && rc == MT_OK) rc = cuda_fail(e, "reading profile events");
    launches[r.slot] += 1;
    total_ms[r.slot] += ms;
    L->pool.push_back(r.a);
    L->pool.push_back(r.b);
  }
  L->recs.clear();
  return rc ? rc : ok();
}

int mt_gemm_set_pairing(int mode) {
  if (mode < 0 || mode > 2) return fail(MT_ERR_INVALID_ARG, "pairing mode must be 0, 1 or 2 (got %d)", mode);
  g_pairing.store(mode);
  return ok();
}

int mt_attn_set_heads_per_cta(int mode) {
  if (mode < 0 || mode > 2) return fail(MT_ERR_INVALID_ARG, "attention heads-per-CTA mode must be 0, 1 or 2 (got %d)", mode);
  mt::set_attention_heads_mode(mode);
  return ok();
}

int mt_gemm_set_tail_split(int mode) {
  if (mode < 0 || mode > 1) return fail(MT_ERR_INVALID_ARG, "tail split mode must be 0 or 1 (got %d)", mode);
  g_tail.store(mode);
  return ok();
}

int mt_gemm_plan(int M, int N, int K, int epilogue, int head_dim, int fp8, int with_handle, int sms, int pair_slots,
                 int* plan) {
  if (plan == nullptr) return fail(MT_ERR_INVALID_ARG, "plan is NULL");
  if (M <= 0 || N <= 0 || K <= 0) return fail(MT_ERR_INVALID_ARG, "M, N, K must be positive");
  if (epilogue < mt::kEpiStore || epilogue > mt::kEpiGelu)
    return fail(MT_ERR_INVALID_ARG, "epilogue must be 0 .. 4 (got %d)", epilogue);
  if (epilogue == mt::kEpiQkv && head_dim != 64 && head_dim != 128)
    return fail(MT_ERR_INVALID_ARG, "head_dim must be 64 or 128 for the QKV epilogue (got %d)", head_dim);
  if (sms < 2 || pair_slots < 1 || pair_slots > sms / 2)
    return fail(MT_ERR_INVALID_ARG, "need sms >= 2 and 1 <= pair_slots <= sms / 2 (got %d, %d)", sms, pair_slots);
  mt::GemmParams p = gemm_params(M, N, K, epilogue == mt::kEpiSwiglu, nullptr);
  plan_gemm_on(p, epilogue, epilogue == mt::kEpiQkv ? head_dim : 0, with_handle != 0, fp8 != 0, sms, pair_slots);
  const int out[8] = {p.pair, p.tiles_m, p.tiles_n, p.split, p.ksplit, p.full_units, p.num_units, p.epi_split};
  for (int i = 0; i < 8; ++i) plan[i] = out[i];
  return ok();
}

int mt_gemm_bf16_t(const void* A, int a_layout, const void* B, int b_layout, void* C, int M, int N, int K,
                   void* cuda_stream) {
  if (A == nullptr || B == nullptr || C == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL operand");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return fail(MT_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  if (M <= 0 || N <= 0 || K <= 0) return fail(MT_ERR_INVALID_ARG, "M, N, K must be positive");
  if ((a_layout != 0 && a_layout != 1) || (b_layout != 0 && b_layout != 1))
    return fail(MT_ERR_INVALID_ARG, "layouts must be 0 or 1 (got %d, %d)", a_layout, b_layout);
  if ((a_layout ? M : K) % 8 || (b_layout ? N : K) % 8 || N % 8)
    return fail(MT_ERR_UNSUPPORTED, "the contiguous dimension of each operand and N must be multiples of 8");
  const int rc = gemm_ab(nullptr, A, a_layout ? M : K, a_layout != 0, B, b_layout ? N : K, b_layout != 0, M, N, K, C,
                         nullptr, N, false, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : ok();
}

int mt_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, void* cuda_stream) {
  if (A == nullptr || B == nullptr || C == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL operand");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return fail(MT_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  if (M <= 0 || N <= 0 || K <= 0) return fail(MT_ERR_INVALID_ARG, "M, N, K must be positive");
  if (K % 8 || N % 8) return fail(MT_ERR_UNSUPPORTED, "K and N must be multiples of 8");
  mt::GemmParams p = gemm_params(M, N, K, false, nullptr);
  p.out = static_cast<bf16*>(C);
  p.ldo = N;
  int rc = run_gemm(nullptr, 0, mt::kEpiStore, A, K, B, N, M, N, K, p, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : ok();
}

int mt_layer_fp8_enable(mt_layer* L, int amax_history_len) {
  if (L == nullptr) return fail(MT_ERR_INVALID_ARG, "handle is NULL");
  if (amax_history_len < 1 || amax_history_len > (1 << 16))
    return fail(MT_ERR_INVALID_ARG, "amax_history_len must be in [1, 65536]");
  if (L->d_f8) cudaFree(L->d_f8);
  L->d_f8 = nullptr;
  const size_t n = 16 + 4 * static_cast<size_t>(amax_history_len);
  cudaError_t e = cudaMalloc(&L->d_f8, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMemset(L->d_f8, 0, n * sizeof(float));
  const float ones[8] = {1, 1, 1, 1, 1, 1, 1, 1};
  if (e == cudaSuccess) e = cudaMemcpy(L->d_f8, ones, sizeof(ones), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 scaling state");
  L->f8_len = amax_history_len;
  L->f8_pos = 0;
  return ok();
}

int mt_layer_fp8_set_scales(mt_layer* L, const float* scales) {
  if (L == nullptr || scales == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  if (L->d_f8 == nullptr) return fail(MT_ERR_INVALID_ARG, "call mt_layer_fp8_enable first");
  float head[16] = {0};
  for (int i = 0; i < 4; ++i) {
    if (!(scales[i] > 0.f) || std::isinf(scales[i])) return fail(MT_ERR_INVALID_ARG, "scales must be positive and finite");
    head[i] = scales[i];
    head[4 + i] = 1.0f / scales[i];
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemset(L->d_f8, 0, (16 + 4 * static_cast<size_t>(L->f8_len)) * sizeof(float));
  if (e == cudaSuccess) e = cudaMemcpy(L->d_f8, head, sizeof(head), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "setting FP8 scales");
  L->f8_pos = 0;
  return ok();
}

int mt_layer_fp8_state(mt_layer* L, float* scales, float* last_amax) {
  if (L == nullptr || scales == nullptr || last_amax == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  if (L->d_f8 == nullptr) return fail(MT_ERR_INVALID_ARG, "call mt_layer_fp8_enable first");
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(scales, L->d_f8, 4 * sizeof(float), cudaMemcpyDeviceToHost);
  const int last = (L->f8_pos + L->f8_len - 1) % L->f8_len;
  for (int t = 0; t < 4 && e == cudaSuccess; ++t)
    e = cudaMemcpy(last_amax + t, L->d_f8 + 16 + static_cast<size_t>(t) * L->f8_len + last, sizeof(float),
                   cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading FP8 state");
  return ok();
}

int mt_layer_forward_fp8(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w,
                         const mt_fp8_weights* w8, void* y_partial, void* cuda_stream) {
  Layout lay;
  int rc = check_call(L, x, y_partial, seq, batch, &lay);
  if (rc) return rc;
  if (L->d_f8 == nullptr) return fail(MT_ERR_INVALID_ARG, "call mt_layer_fp8_enable first");
  if (L->hidden % 16 || L->f_r % 16)
    return fail(MT_ERR_UNSUPPORTED, "the FP8 path needs hidden and ffn/tp_size multiples of 16");
  if (w8 == nullptr) return fail(MT_ERR_INVALID_ARG, "fp8 weights struct is NULL");
  const void* wp[] = {w8->w_qkv, w8->w_o, w8->w_fc1, w8->w_fc2};
  const float* dp[] = {w8->deq_qkv, w8->deq_o, w8->deq_fc1, w8->deq_fc2};
  for (int i = 0; i < 4; ++i)
    if (wp[i] == nullptr || !aligned16(wp[i]) || dp[i] == nullptr)
      return fail(MT_ERR_INVALID_ARG, "fp8 weight %d or its dequantisation factor is NULL/misaligned", i);
  mt_weights wn = *w;  // norms and biases are bf16; the projections come from w8
  wn.w_qkv = w8->w_qkv;
  wn.w_o = w8->w_o;
  wn.w_fc1 = w8->w_fc1;
  wn.w_fc2 = w8->w_fc2;
  if ((rc = check_weights(L, &wn, true, true))) return rc;
  rc = forward_device_fp8(L, lay, x, seq, batch, w, w8, y_partial, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_quantize_e4m3(const void* src, size_t n, void* dst, float* amax_deq, void* cuda_stream) {
  if (src == nullptr || dst == nullptr || amax_deq == nullptr) return fail(MT_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(src) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(amax_deq) & 7u))
    return fail(MT_ERR_INVALID_ARG, "src/dst must be 16-byte and amax_deq 8-byte aligned");
  if (n == 0 || n % 8) return fail(MT_ERR_UNSUPPORTED, "n must be a positive multiple of 8");
  cudaError_t e = mt::launch_quantize_e4m3(static_cast<const bf16*>(src), n, static_cast<uint8_t*>(dst), amax_deq,
                                           static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "E4M3 quantisation launch");
  return ok();
}

int mt_gemm_e4m3(const void* A, const void* B, void* C, int M, int N, int K, const float* deq_a, const float* deq_b,
                 void* cuda_stream) {
  if (A == nullptr || B == nullptr || C == nullptr || deq_a == nullptr || deq_b == nullptr)
    return fail(MT_ERR_INVALID_ARG, "NULL operand");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return fail(MT_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  if (M <= 0 || N <= 0 || K <= 0) return fail(MT_ERR_INVALID_ARG, "M, N, K must be positive");
  if (K % 16 || N % 8) return fail(MT_ERR_UNSUPPORTED, "K must be a multiple of 16 and N of 8");
  mt::GemmParams p = gemm_params(M, N, K, false, nullptr);
  p.out = static_cast<bf16*>(C);
  p.ldo = N;
  p.deq_a = deq_a;
  p.deq_b = deq_b;
  int rc = run_gemm(nullptr, 0, mt::kEpiStore, A, K, B, N, M, N, K, p, static_cast<cudaStream_t>(cuda_stream), true);
  return rc ? rc : ok();
}

int mt_layer_backward_workspace_bytes(const mt_layer* L, int seq, int batch, size_t* bytes) {
  if (L == nullptr || bytes == nullptr) return fail(MT_ERR_INVALID_ARG, "handle or bytes is NULL");
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive");
  *bytes = bw_layout(L, seq, batch).total;
  return ok();
}

int mt_layer_backward(mt_layer* L, const void* x, const void* dy, int seq, int batch, const mt_weights* w, void* dx,
                      const mt_grads* g, void* cuda_stream) {
  BwLayout b;
  int rc = check_train_call(L, x, dy, seq, batch, w, dx, g, true, &b);
  if (rc) return rc;
  rc = backward_device(L, b, x, dy, seq, batch, w, dx, g, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_layer_forward_train(mt_layer* L, const void* x, int seq, int batch, const mt_weights* w, void* y,
                           void* cuda_stream) {
  BwLayout b;
  int rc = check_train_call(L, x, x, seq, batch, w, y, nullptr, false, &b);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if ((rc = forward_saving(L, b, x, seq, batch, w, st))) return rc;
  // fc2 with the residual: y = h + a W_fc2^T + b_fc2, as the forward's last GEMM
  const int T = seq * batch, H = L->hidden, f = L->f_r;
  mt::GemmParams p = gemm_params(T, H, f, false, L->d_err);
  p.out = static_cast<bf16*>(y);
  p.ldo = H;
  p.bias = static_cast<const bf16*>(w->b_fc2);
  p.resid = region<bf16>(L, b.fwd, kH);
  p.ldr = H;
  if ((rc = run_gemm(L, kSlotFc2, mt::kEpiResid, bwr<bf16>(L, b, kBA), f, w->w_fc2, H, T, H, f, p, st))) return rc;
  return done(L, st);
}

int mt_layer_backward_saved(mt_layer* L, const void* x, const void* dy, int seq, int batch, const mt_weights* w,
                            void* dx, const mt_grads* g, void* cuda_stream) {
  BwLayout b;
  int rc = check_train_call(L, x, dy, seq, batch, w, dx, g, true, &b);
  if (rc) return rc;
  rc = backward_from_saved(L, b, x, dy, seq, batch, w, dx, g, static_cast<cudaStream_t>(cuda_stream));
  return rc ? rc : done(L, static_cast<cudaStream_t>(cuda_stream));
}

int mt_sp_reduce_add_norm(const void* const* partials, int num_partials, const void* resid, const void* bias,
                          const void* norm_w, const void* norm_b, int norm, float eps, int tokens, int hidden, int row0,
                          int rows, void* h_out, void* hn_out, void* cuda_stream) {
  if (partials == nullptr || resid == nullptr || norm_w == nullptr || h_out == nullptr || hn_out == nullptr)
    return fail(MT_ERR_INVALID_ARG, "NULL argument");
  if (num_partials < 1 || num_partials > mt::kMaxSpParts)
    return fail(MT_ERR_UNSUPPORTED, "num_partials must be in [1, %d]", mt::kMaxSpParts);
  if (norm != MT_NORM_RMS && norm != MT_NORM_LAYER) return fail(MT_ERR_INVALID_ARG, "unknown norm %d", norm);
  if (norm == MT_NORM_LAYER && norm_b == nullptr) return fail(MT_ERR_INVALID_ARG, "LayerNorm needs norm_b");
  if (!(eps > 0.f) || std::isinf(eps)) return fail(MT_ERR_INVALID_ARG, "eps must be positive and finite");
  if (tokens <= 0 || hidden <= 0 || rows < 0 || row0 < 0 || row0 + rows > tokens)
    return fail(MT_ERR_INVALID_ARG, "rows [%d, %d) outside [0, %d)", row0, row0 + rows, tokens);
  if (hidden % 8 || hidden > 8192) return fail(MT_ERR_UNSUPPORTED, "hidden must be a multiple of 8 and <= 8192");
  mt::SpParams p{};
  for (int i = 0; i < num_partials; ++i) {
    if (partials[i] == nullptr || !aligned16(partials[i])) return fail(MT_ERR_INVALID_ARG, "partial %d is NULL or misaligned", i);
    p.parts[i] = static_cast<const bf16*>(partials[i]);
  }
  const void* ptrs[] = {resid, bias, norm_w, norm_b, h_out, hn_out};
  for (const void* q : ptrs)
    if (q != nullptr && !aligned16(q)) return fail(MT_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  p.nparts = num_partials;
  p.row0 = static_cast<size_t>(row0);
  p.rows = rows;
  p.H = hidden;
  p.resid = static_cast<const bf16*>(resid);
  p.bias = static_cast<const bf16*>(bias);
  p.gamma = static_cast<const bf16*>(norm_w);
  p.beta = static_cast<const bf16*>(norm_b);
  p.eps = eps;
  p.h = static_cast<bf16*>(h_out);
  p.hn = static_cast<bf16*>(hn_out);
  cudaError_t e = mt::launch_sp_add_norm(norm == MT_NORM_LAYER, p, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "sequence-parallel epilogue launch");
  return ok();
}

int mt_selftest_bounded_wait(int limit_us) {
  if (limit_us < 1 || limit_us > 1000000) return fail(MT_ERR_INVALID_ARG, "limit_us must be in [1, 1e6]");
  int* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  cudaMemset(d, 0, sizeof(int));
  e = mt::launch_wait_selftest(d, static_cast<unsigned long long>(limit_us) * 1000ull, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int code = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&code, d, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self test");
  if (code == MT_ERR_DEVICE_TIMEOUT) return fail(MT_ERR_DEVICE_TIMEOUT, "bounded wait gave up after %d us", limit_us);
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------- allocation-free variant
// Scratch for mt_layer_forward_static: a fixed area in the library's own device image.  Its name
// is only a host-side stand-in in host code; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_area[MT_STATIC_AREA_BYTES];

namespace {
constexpr size_t kStaticHeader = 1024;  // error word at offset 0, RoPE frequencies at 256
constexpr int kMaxDevices = 128;
std::mutex g_static_mu;
struct StaticSlot {
  unsigned long long ctx_id;  // the CUDA context the address belongs to
  void* ptr;
};
StaticSlot g_static[kMaxDevices];

// Id of the context current on this thread (0 if none is current yet).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_ctx = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  if (get_ctx == nullptr || get_id == nullptr) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qb != cudaDriverEntryPointSuccess)
      return 0;
    get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the static area on `dev` (the current device).  It is looked up once per
// device and context: a context created anew (after cudaDeviceReset, say) gets a fresh lookup.
int static_area(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(MT_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  const unsigned long long id = current_context_id();
  StaticSlot& slot = g_static[dev];
  if (slot.ptr == nullptr || id == 0 || slot.ctx_id != id) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_area);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch area");
    slot.ptr = p;
    slot.ctx_id = current_context_id();  // the lookup has made the context current if none was
  }
  *out = slot.ptr;
  return MT_OK;
}

// Per-call set-up of the static area, as kernel arguments (so no host memory is read by a copy):
// clears the error word and writes the RoPE frequencies.
struct StaticSetup {
  double theta[64];
  int half;
};

__global__ void static_setup_kernel(int* err, double* theta, StaticSetup s) {
  const int i = threadIdx.x;
  if (i == 0) *err = 0;
  if (theta != nullptr && i < s.half) theta[i] = s.theta[i];
}
}  // namespace

extern "C" int mt_layer_forward_static(int hidden, int heads, int query_groups, int head_dim, int ffn, int norm,
                                       int act, float rope_base, int tp_size, int tp_rank, float eps, const void* x,
                                       int seq, int batch, const mt_weights* w, void* y_partial, void* cuda_stream) {
  if (hidden <= 0 || heads <= 0 || query_groups <= 0 || head_dim <= 0 || ffn <= 0 || tp_size <= 0)
    return fail(MT_ERR_INVALID_ARG, "sizes must be positive");
  if (tp_rank < 0 || tp_rank >= tp_size) return fail(MT_ERR_INVALID_ARG, "tp_rank %d outside [0, %d)", tp_rank, tp_size);
  if (norm != MT_NORM_RMS && norm != MT_NORM_LAYER) return fail(MT_ERR_INVALID_ARG, "unknown norm %d", norm);
  if (act != MT_ACT_SWIGLU && act != MT_ACT_GELU_TANH) return fail(MT_ERR_INVALID_ARG, "unknown activation %d", act);
  if (!(rope_base >= 0.f) || std::isinf(rope_base)) return fail(MT_ERR_INVALID_ARG, "rope_base must be finite and >= 0");
  if (!(eps > 0.f) || std::isinf(eps)) return fail(MT_ERR_INVALID_ARG, "eps must be positive and finite");
  if (head_dim != 64 && head_dim != 128) return fail(MT_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", head_dim);
  if (heads % query_groups) return fail(MT_ERR_UNSUPPORTED, "heads %% query_groups != 0");
  if (heads % tp_size || query_groups % tp_size || ffn % tp_size)
    return fail(MT_ERR_UNSUPPORTED, "heads, query_groups and ffn must be divisible by tp_size");
  if (hidden % 8 || hidden > 8192) return fail(MT_ERR_UNSUPPORTED, "hidden must be a multiple of 8 and <= 8192");
  if ((ffn / tp_size) % 8) return fail(MT_ERR_UNSUPPORTED, "ffn/tp_size must be a multiple of 8");

  // A handle on the stack: same fields as mt_layer_create fills, but every device buffer points
  // into the static area.
  mt_layer L{};
  L.hidden = hidden;
  L.heads = heads;
  L.groups = query_groups;
  L.head_dim = head_dim;
  L.ffn = ffn;
  L.norm = norm;
  L.act = act;
  L.tp = tp_size;
  L.rank = tp_rank;
  L.rope_base = rope_base;
  L.eps = eps;
  L.nh_r = heads / tp_size;
  L.ng_r = query_groups / tp_size;
  L.f_r = ffn / tp_size;
  L.f1_r = act == MT_ACT_SWIGLU ? 2 * L.f_r : L.f_r;
  L.q_w = L.nh_r * head_dim;
  L.kv_w = L.ng_r * head_dim;
  L.profile_mask = 0;
  if (seq <= 0 || batch <= 0) return fail(MT_ERR_INVALID_ARG, "seq and batch must be positive (got %d, %d)", seq, batch);
  const size_t need = layout_for(&L, seq, batch).total;
  const size_t have = static_cast<size_t>(MT_STATIC_AREA_BYTES) - kStaticHeader;
  if (need > have)
    return fail(MT_ERR_UNSUPPORTED, "this call needs %zu bytes of scratch; the static area holds %zu (seq*batch too large)",
                need, have);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(MT_ERR_UNSUPPORTED, "this library is built for sm_103 (GB300); device %d is sm_%d%d", dev, major, minor);
  void* base = nullptr;
  int rc = static_area(dev, &base);
  if (rc) return rc;
  L.device = dev;
  L.d_err = static_cast<int*>(base);
  L.d_theta = rope_base > 0.f ? reinterpret_cast<double*>(static_cast<char*>(base) + 256) : nullptr;
  L.ws = static_cast<char*>(base) + kStaticHeader;
  L.ws_bytes = have;

  Layout lay;
  if ((rc = check_call(&L, x, y_partial, seq, batch, &lay))) return rc;
  if ((rc = check_weights(&L, w, true, true))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  StaticSetup setup{};
  setup.half = head_dim / 2;
  for (int i = 0; i < setup.half; ++i)
    setup.theta[i] = std::pow(static_cast<double>(rope_base), -2.0 * i / head_dim);  // as mt_layer_create
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(64);
  cfg.stream = st;
  e = cudaLaunchKernelEx(&cfg, static_setup_kernel, L.d_err, L.d_theta, setup);  // the error word starts at zero
  if (e != cudaSuccess) return cuda_fail(e, "static area set-up launch");
  rc = forward_device(&L, lay, x, seq, batch, w, y_partial, st);
  return rc ? rc : ok();
}

extern "C" int mt_layer_forward_static_status(void* cuda_stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  void* base = nullptr;
  int rc = static_area(dev, &base);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int code = 0;  // the copy to pageable memory returns once the stream's earlier work and the copy are done
  e = cudaMemcpyAsync(&code, base, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the static area's error word");
  if (code != 0)
    return fail(MT_ERR_DEVICE_TIMEOUT,
                "a kernel of the last static call stopped waiting on a barrier (device code %d); its outputs are invalid",
                code);
  return ok();
}

