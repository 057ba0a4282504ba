// Causal GQA flash attention on the 5th-generation tensor cores.
//
// o_h = softmax(q_h k_g^T / sqrt(d) + causal mask) v_g,  g = h / (nh/ng)
// (core_attention with AttnMaskType.causal in the layer spec of "快速入门" §3.1; GQA through
// num_query_groups of "ai阅读megatron" TransformerConfig; FlashAttention is the prior art the
// pages name: exact attention computed block by block with an online softmax, O(S) memory.)
//
// Two forms share one scheme, chosen by launch_attention from d, the heads per kv group and the
// number of CTAs:
//   attn_tp_kernel<D>       an even number of heads per group: one CTA takes two heads of one group
//                           for a 128-query block, so every K/V tile feeds both (the GQA/MQA
//                           workloads); P stays in tensor memory;
//   attn_db_kernel<D>       one head per CTA with two score buffers in tensor memory: an odd
//                           number of heads per group (MHA at d = 128), or too few two-head CTAs
//                           to fill the SMs twice over (then the longest query block's chain of
//                           key blocks sets the time);
//   attn2_kernel<64, true>  d = 64 with an odd number of heads per group (MHA): two heads of two
//                           groups, each ring slot holding both groups' tiles.
// CTAs are issued longest-first (the last query blocks see the most keys).  In every form warp 0
// loads the Q tile(s) and then K and V tiles [128 keys x d] by TMA; one thread of warp 1 issues
// S_j = Q K_j^T into a TMEM score buffer and O += P_j V_j into a TMEM accumulator, reading V as an
// MN-major operand (its d index contiguous); the softmax warps (one query row per thread) read S_j
// from TMEM, mask the diagonal block, keep a running maximum and sum in the log2 domain, write
// P_j = 2^(s c - m) as fp16 (into shared memory in the 128-byte-swizzled layout the MMA reads in
// attn2_kernel, over S_j in tensor memory in attn_tp_kernel), and rescale O in TMEM only when the running
// maximum grows by more than 2^8 (between rescales P stays below 256).  At the end O / l is written as bf16 (or E4M3) to o[t, h*d + i] and,
// when asked, m + log2(l) to lse for the backward pass.
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

constexpr int BQ = 128, BKV = 128;
static_assert(BKV == 128, "a row of S is read with one 128-column TMEM load");
constexpr int P_ATOM = BQ * 128;  // one 64-key half of a P tile: [128 rows x 64 fp16], 16 KB

// Maximum of a row of S (BKV scores in registers) over eight independent chains of three-input
// maxima (chain k takes elements 2k and 2k+1 of every 16), so the reduction is not one long chain.
__device__ __forceinline__ float row_max(const float* s) {
  float m8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m8[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
  for (int i = 16; i < BKV; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], s[i + 2 * k], s[i + 2 * k + 1]);
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// What one CTA works on: query block qb of a sequence whose rows start at q_row0 - qb*128 and
// whose keys start at kv_row0 (rows of the [b, head, s, d] q, k, v buffers), `len` tokens long;
// batch row b, head (or first head of the pair) h.
struct Work {
  int qb, b, h, q_row0, kv_row0, len;
};

// Dense batches: blockIdx -> (query block, longest first; batch row; head slot).  Packed samples:
// (query block, longest first; sample; head slot); returns false when the block lies past the end
// of its sample (or the sample's bounds are invalid) so the CTA has nothing to do.
__device__ __forceinline__ bool decode_work(const AttnParams& p, int heads_slots, int head_step, Work& w) {
  const int bid = static_cast<int>(blockIdx.x);
  if (p.cu == nullptr) {
    const int per = p.batch * heads_slots;
    w.qb = p.num_qb - 1 - bid / per;
    const int rem = bid % per;
    w.b = rem / heads_slots;
    w.h = head_step * (rem - w.b * heads_slots);
    w.q_row0 = w.qb * BQ;
    w.kv_row0 = 0;
    w.len = p.seq;
    return true;
  }
  const int per = p.num_seqs * heads_slots;
  w.qb = p.num_qb - 1 - bid / per;
  const int rem = bid % per;
  const int sid = rem / heads_slots;
  w.b = 0;
  w.h = head_step * (rem - sid * heads_slots);
  const int start = p.cu[sid];
  w.len = p.cu[sid + 1] - start;
  if (start < 0 || w.len <= w.qb * BQ || start + w.len > p.seq) return false;
  w.q_row0 = start + w.qb * BQ;
  w.kv_row0 = start;
  return true;
}

// ------------------------------------------------------------------ two heads per CTA, P in shared memory
// The form used for MHA at d = 64 (two heads of two groups, TG); attn_tp_kernel below replaces it
// for two heads of one group.  The CTA holds the Q tiles of two heads for one 128-row query block.
//   TMEM: head t's scores S_t in columns [256t, 256t+128) and its output O_t in [256t+128, +d).
//   The softmax warps of a head read S_t into registers and release it at once (s_free), so the
//   tensor core computes S_t(j+1) while they turn S_t(j) into P_t(j); P goes to shared memory (fp16,
//   128-byte swizzle, per head) and O_t += P_t V_j reads it from there.
//   Shared memory: Q of both heads, a three-slot ring of K and V tiles and the two P tiles.  Tiles
//   enter the ring in the order K0, K1, V0, K2, V1, K3, ..., each taking the slot of the tile three
//   places earlier: V_j loads as soon as both S(j) are done and K_{j+2} as soon as both P V(j-1)
//   are, so each tile has about one block of lead time.  The softmax forms P_t(j) in registers
//   before it waits for P_t(j-1) V_{j-1}, and only the shared-memory stores wait.
//   10 warps put three warps on some SM sub-partitions, whose 16K-register files then allow 168
//   registers per thread.
// The softmax role for one head (four warps, one query row per thread, warp w on TMEM lane quadrant
// `quad`): per key block it waits for S in tensor memory, releases it at once, masks the diagonal
// block, forms P = 2^(s c - m) in registers, waits for the previous P V product (then rescales O
// if the running maximum grew by more than 2^8) and stores P into its shared-memory tile in the
// 128-byte-swizzled layout the P V MMA reads.  At the end O / l goes to o (bf16, or E4M3 with its
// amax) and m + log2(l) to lse.  `arrive` signals a barrier the MMA thread waits on.
template <int D, typename Arrive>
__device__ __forceinline__ void softmax_head(const AttnParams& p, const Work& wk, int h, int quad, int lane,
                                             uint32_t tS, uint32_t tO, uint8_t* ptile, uint32_t s_full,
                                             uint32_t s_free, uint32_t p_full, uint32_t o_done,
                                             volatile int* abort_flag, Arrive arrive) {
  const int qb = wk.qb, b = wk.b, nkv = qb + 1;
  const int r = quad * 32 + lane;
  const bool row_ok = qb * BQ + r < wk.len;  // inside its sequence
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const float c = p.scale_log2;
  uint8_t* prow = ptile + r * 128;
  const int sw = r & 7;
  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    bool w = mbar_wait(s_full, j & 1, p.err, abort_flag);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float s[BKV];
    tmem_ld128(tS + lane_off, s);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive(s_free);  // the tensor core may overwrite S now
    if (j == qb) {
#pragma unroll
      for (int i = 0; i < BKV; ++i)
        if (i > r) s[i] = -INFINITY;
    }
    const float mx = row_max(s);
    const float m_new = fmaxf(m_used, mx * c);
    const bool grow = __any_sync(0xffffffffu, m_new > m_used + 8.0f);
    float alpha = 1.f;
    if (grow) {
      alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m_used - m_new);
      m_used = m_new;
    }
    // P = 2^(s c - m) in packed halves, formed in registers while the tensor core still runs
    // P(j-1) V_{j-1}: one fp32x2 FMA, one fp16x2 conversion and one fp16x2 exponential per pair
    // of scores (the argument is at most 8 after the lazy rescaling, so its fp16 rounding moves P
    // by under 0.6%, the order of P's own 16-bit rounding); row sums in four fp16x2 partial sums
    // per 64 keys, widened to fp32 once per block.
    uint32_t pk[BKV / 2];
    float rs = 0.f;
    {
      const float2 cc = make_float2(c, c), mm = make_float2(-m_used, -m_used);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        __half2 acc[4] = {__float2half2_rn(0.f), __float2half2_rn(0.f), __float2half2_rn(0.f),
                          __float2half2_rn(0.f)};
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int i = 64 * hf + 2 * q;
          const float2 xy = ffma2(make_float2(s[i], s[i + 1]), cc, mm);
          pk[32 * hf + q] = ex2_f16x2(pack_f16x2(xy.x, xy.y));
          acc[q & 3] = __hadd2(acc[q & 3], *reinterpret_cast<const __half2*>(&pk[32 * hf + q]));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(acc[k]);
          rs += f.x + f.y;
        }
      }
    }
    l = l * alpha + rs;
    if (j > 0) {  // P(j-1) V_{j-1} finished: P may be overwritten and O is stable
      w = mbar_wait(o_done, (j - 1) & 1, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      if (grow) {
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          float o[32];
          tmem_ld32(tO + lane_off + cc * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tO + lane_off + cc * 32, o);
        }
      }
    }
    // each 8-key chunk at its swizzled position of the 128-byte rows the P V MMA reads
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint32_t* e4 = pk + 32 * hf + 4 * ch;
        *reinterpret_cast<uint4*>(prow + hf * P_ATOM + ((ch ^ sw) << 4)) = make_uint4(e4[0], e4[1], e4[2], e4[3]);
      }
    fence_proxy_async_smem();  // the P stores become visible to the tensor core
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive(p_full);
  }
  if (ok) {
    const bool w = mbar_wait(o_done, (nkv - 1) & 1, p.err, abort_flag);
    if (__all_sync(0xffffffffu, w)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const size_t orow = (static_cast<size_t>(wk.q_row0 + r) * p.batch + b) * p.ldo + h * D;
      if (p.lse != nullptr && row_ok)
        p.lse[(static_cast<size_t>(b) * p.nh + h) * p.seq + wk.q_row0 + r] = m_used + log2f(l);
      const float qs = p.o8 != nullptr ? __ldg(p.q_scale) : 1.f;
      float mx = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + lane_off + cc * 32, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= inv_l;
          if (p.o8 != nullptr) {  // E4M3 output for the FP8 output projection
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(o[i]));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint2*>(p.o8 + orow + cc * 32 + q4 * 8) = pack_e4m3x8(o + q4 * 8, qs);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint4*>(p.o + orow + cc * 32 + q4 * 8) = pack_bf16x8(o + q4 * 8);
          }
        }
      }
      if (p.o8 != nullptr) {
        mx = warp_max(mx);
        if (lane == 0) atomic_max_abs(p.amax, mx);
      }
    }
  }
}

// TG (two groups): the CTA's two heads belong to different kv groups (MHA, or an odd number of
// heads per group) and every ring slot holds both groups' tiles, head t's at offset t * 16 KB; d = 64.
template <int D, bool TG = false>
struct Geo2 {
  static_assert(!TG || D == 64, "a ring slot holds two groups' tiles only at d = 64");
  static constexpr int ATOM = 128 * 128;        // [128 rows x 64 fp16/bf16] swizzle block, 16 KB
  static constexpr int Q_BYTES = BQ * D * 2;    // per head
  static constexpr int KV_BYTES = (TG ? 2 : 1) * BKV * D * 2;  // K or V tiles [128 keys x d]: d/64 atoms each
  static constexpr int P_BYTES = BQ * BKV * 2;  // per head: two key halves of 16 KB
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * Q_BYTES;  // three-slot ring shared by K and V tiles
  static constexpr int OFF_P = OFF_KV + 3 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr size_t SMEM_USED = 1024 + OFF_BAR + 256;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM (TMEM)
  static constexpr uint32_t IDESC_S = idesc_bf16(BQ, BKV);
  static constexpr uint32_t IDESC_O = idesc_f16(BQ, D) | (1u << 16);  // fp16 P (K-major), fp16 V (MN-major)
};
static_assert(Geo2<64, true>::SMEM_USED <= 232448, "attention tiles exceed the shared memory of a CTA");

template <int D, bool TG>
__global__ void __launch_bounds__(320, 1)
    attn2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using G = Geo2<D, TG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + G::OFF_BAR);
  // bars: q_full | kv_full[3] | kv_empty[3] | s_full[2] | s_free[2] | p_full[2] |
  //       o_done[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  // tile number n of the load sequence sits in ring slot n % 3, in that slot's (n / 3)-th use
  auto kv_full = [&](int n) { return bar0 + 8u * (1 + n % 3); };
  auto kv_empty = [&](int n) { return bar0 + 8u * (4 + n % 3); };
  auto use_parity = [](int n) { return static_cast<uint32_t>((n / 3) & 1); };
  auto s_full = [&](int t) { return bar0 + 8u * (7 + t); };
  auto s_free = [&](int t) { return bar0 + 8u * (9 + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (11 + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (13 + t); };
  const uint32_t drain = bar0 + 8u * 15;
  auto sQa = [&](int t) { return smem_u32(base + G::OFF_Q + t * G::Q_BYTES); };
  auto sKV = [&](int n) { return smem_u32(base + G::OFF_KV + (n % 3) * G::KV_BYTES); };
  auto sPa = [&](int t) { return smem_u32(base + G::OFF_P + t * G::P_BYTES); };

  pdl_wait();  // q, k, v (and cu_seqlens) are written by the kernels before
  pdl_trigger();
  Work wk;
  if (!decode_work(p, p.nh >> 1, 2, wk)) return;  // uniform over the CTA, before any barrier or TMEM use
  const int qb = wk.qb, b = wk.b, h0 = wk.h;
  const int g = h0 / (p.nh / p.ng), g1 = (h0 + 1) / (p.nh / p.ng);  // the heads' kv groups (equal unless TG)
  constexpr uint32_t HEAD_OFF = TG ? G::ATOM : 0u;  // head 1's tile inside a ring slot
  const int nkv = qb + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(kv_full(i), 1);
      mbar_init(kv_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_free(i), 4);
      mbar_init(p_full(i), 4);
      mbar_init(o_done(i), 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto tS = [&](int t) { return tmem_base + 256u * t; };
  auto tO = [&](int t) { return tmem_base + 256u * t + 128u; };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * G::Q_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sQa(t) + a * G::ATOM, &tmQ, q_full, a * 64, wk.q_row0, b * p.nh + h0 + t);
      // Load sequence K0, K1, V0, K2, V1, K3, V2, ..., K(n-1), V(n-2), V(n-1) through the ring:
      // tile n reuses the slot of tile n - 3, so V_j waits only for S(j) (K_j's slot) and K_{j+2}
      // for P V(j-1) (V_{j-1}'s slot), each a block ahead of its own use.
      int issued = 0;
      auto load = [&](const CUtensorMap* map, int j) -> bool {
        const int n = issued;
        if (!mbar_wait(kv_empty(n), use_parity(n) ^ 1u, p.err, abort_flag)) return false;
        mbar_arrive_expect_tx(kv_full(n), G::KV_BYTES);
        if (TG) {  // both heads' groups, one [128 x 64] box each
          tma_load_3d(sKV(n), map, kv_full(n), 0, wk.kv_row0 + j * BKV, b * p.ng + g);
          tma_load_3d(sKV(n) + HEAD_OFF, map, kv_full(n), 0, wk.kv_row0 + j * BKV, b * p.ng + g1);
        } else {
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sKV(n) + a * G::ATOM, map, kv_full(n), a * 64, wk.kv_row0 + j * BKV, b * p.ng + g);
        }
        ++issued;
        return true;
      };
      bool ok = load(&tmK, 0) && (nkv < 2 || load(&tmK, 1));
      for (int j = 0; ok && j < nkv; ++j) {
        ok = load(&tmV, j);
        if (ok && j + 2 < nkv) ok = load(&tmK, j + 2);
      }
      if (!ok) {  // let this CTA's own copies in flight land
        mbar_wait_slow(q_full, 0, nullptr, nullptr, kDrainLimitNs);
        for (int n = issued - 1; n >= 0 && n >= issued - 3; --n)
          mbar_wait_slow(kv_full(n), use_parity(n), nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // tile numbers of K_j and V_j in the loader's sequence
      auto tile_k = [](int j) { return j < 2 ? j : 2 * j - 1; };
      auto tile_v = [nkv](int j) { return (nkv > 1 ? 2 : 1) + 2 * j - ((j == nkv - 1 && nkv >= 2) ? 1 : 0); };
      auto issue_s = [&](int t, int n) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * G::ATOM + (k & 3) * 32;
          mma_bf16_ss(tS(t), sw128_desc(sQa(t) + off), sw128_desc(sKV(n) + t * HEAD_OFF + off), G::IDESC_S,
                      k > 0 ? 1u : 0u);
        }
        mma_commit(s_full(t));
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag) && mbar_wait(kv_full(0), use_parity(0), p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        mma_commit(kv_empty(0));
      }
      for (int j = 0; ok && j < nkv; ++j) {
        // S(j+1) of both heads as soon as their softmax has taken S(j) into registers
        if (j + 1 < nkv) {
          const int nk = tile_k(j + 1);
          if (!mbar_wait(kv_full(nk), use_parity(nk), p.err, abort_flag)) {
            ok = false;
            break;
          }
          for (int t = 0; t < 2 && ok; ++t) {
            if (!mbar_wait(s_free(t), j & 1, p.err, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, nk);
          }
          if (!ok) break;
          mma_commit(kv_empty(nk));
        }
        // O_t += P_t(j) V_j once the softmax has written P_t(j)
        const int nv = tile_v(j);
        const uint32_t sV = sKV(nv);
        if (!mbar_wait(kv_full(nv), use_parity(nv), p.err, abort_flag)) {
          ok = false;
          break;
        }
        for (int t = 0; t < 2 && ok; ++t) {
          if (!mbar_wait(p_full(t), j & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BKV / 16; ++k) {
            const uint32_t pa = sPa(t) + (k >> 2) * G::ATOM + (k & 3) * 32;
            mma_bf16_ss(tO(t), sw128_desc(pa), sw128_desc_mn(sV + t * HEAD_OFF + k * 2048, G::ATOM), G::IDESC_O,
                        (j > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(o_done(t));
        }
        if (!ok) break;
        mma_commit(kv_empty(nv));
      }
      mma_commit(drain);
      mbar_wait_slow(drain, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int t = (warp - 2) >> 2;  // which head of the pair
    softmax_head<D>(p, wk, h0 + t, warp & 3, lane, tS(t), tO(t), base + G::OFF_P + t * G::P_BYTES, s_full(t),
                    s_free(t), p_full(t), o_done(t), abort_flag, [](uint32_t bar) { mbar_arrive(bar); });
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ two heads of one group, P in TMEM
// The variant for an even number of query heads per kv group (GQA/MQA), with the probabilities kept
// in tensor memory: the softmax warps of head t write P_t(j) (fp16) over the first 64 columns of
// S_t(j), which they have read into registers, and O_t += P_t(j) V_j takes P as its A operand from
// tensor memory.  No shared-memory P tile and no generic-to-async proxy fence; the freed shared
// memory holds a deeper ring of K and V tiles (NS slots, loaded K0, V0, K1, V1, ... in the order
// the MMAs use them).
//   TMEM: head t's S_t (and P_t) in columns [256t, 256t+128), O_t in [256t+128, 256t+128+d).
//   MMA order: S_A(0), S_B(0); then per key block j: P_A V_j, S_A(j+1), P_B V_j, S_B(j+1).  The
//   MMAs of one thread run in issue order, so S_t(j+1) overwrites S_t's columns only after
//   P_t(j) V_j has read P_t(j) from them; the softmax of one head runs while the tensor core
//   works on the other head's pair of products.  One barrier per head (s_full) completes after
//   S_t(j) -- and so also after P_t(j-1) V_{j-1}, which makes O_t stable for a rescale -- and, one
//   block after the last, when O_t is final; p_full tells the MMA thread that P_t(j) is written
//   (and any rescale of O_t done).
template <int D, int NH>
struct GeoT {
  static constexpr int ATOM = 128 * 128;          // [128 rows x 64 bf16] swizzle block, 16 KB
  static constexpr int Q_BYTES = BQ * D * 2;      // per head
  static constexpr int KV_BYTES = BKV * D * 2;    // one K or V tile [128 keys x d]
  static constexpr int NS = D == 128 ? (NH == 2 ? 5 : 6) : 8;  // ring slots (NH: heads per CTA)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = NH * Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NS * KV_BYTES;
  static constexpr size_t SMEM_USED = 1024 + OFF_BAR + 256;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM
  // two heads: S and O of each (4 x 128 columns); one head: two S buffers and O (3 x 128)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = idesc_bf16(BQ, BKV);
  static constexpr uint32_t IDESC_O = idesc_f16(BQ, D) | (1u << 16);  // fp16 P (K-major), fp16 V (MN-major)
};
static_assert(GeoT<128, 2>::SMEM_USED <= 232448 && GeoT<64, 2>::SMEM_USED <= 232448 &&
                  GeoT<128, 1>::SMEM_USED <= 232448 && GeoT<64, 1>::SMEM_USED <= 232448,
              "attention tiles exceed the shared memory of a CTA");

// Softmax of one head (four warps, one query row per thread) for attn_tp_kernel and attn_db_kernel:
// per key block it waits for S, masks the diagonal block, forms P = 2^(s c - m) as fp16 pairs,
// rescales O when the running maximum grew by more than 2^8, writes P over S's first 64 columns
// and signals p_full.  DB (attn_db_kernel): block j's scores are in the buffer at tS + 128 (j & 1),
// completed on the barrier s_full + 8 (j & 1) (phase j / 2); P(j) is signalled on p_full + 8 (j & 1)
// (a warp may run one block ahead of the others, so consecutive blocks use different barriers);
// o_done completes after each P V product and o_final after the last: a rescale first waits for
// the previous product, the final O for all of them.
template <int D, bool DB = false>
__device__ __forceinline__ void softmax_head_tm(const AttnParams& p, const Work& wk, int h, int quad, int lane,
                                                uint32_t tS, uint32_t tO, uint32_t s_full, uint32_t p_full,
                                                volatile int* abort_flag, uint32_t o_done = 0, uint32_t o_final = 0) {
  const int qb = wk.qb, b = wk.b, nkv = qb + 1;
  const int r = quad * 32 + lane;
  const bool row_ok = qb * BQ + r < wk.len;  // inside its sequence
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const float c = p.scale_log2;
  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    const uint32_t tSj = DB ? tS + 128u * (j & 1) : tS;
    const bool w = DB ? mbar_wait(s_full + 8u * (j & 1), (j >> 1) & 1, p.err, abort_flag)
                      : mbar_wait(s_full, j & 1, p.err, abort_flag);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float s[BKV];
    tmem_ld128(tSj + lane_off, s);
    if (j == qb) {  // diagonal block: key j*128+i visible iff i <= r
#pragma unroll
      for (int i = 0; i < BKV; ++i)
        if (i > r) s[i] = -INFINITY;
    }
    const float mx = row_max(s);
    const float m_new = fmaxf(m_used, mx * c);
    const bool grow = __any_sync(0xffffffffu, m_new > m_used + 8.0f);
    float alpha = 1.f;
    if (grow) {
      alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m_used - m_new);
      m_used = m_new;
    }
    // P = 2^(s c - m) in packed halves (one fp32x2 FMA, one fp16x2 conversion and one fp16x2
    // exponential per pair of scores; the argument is at most 8 after the lazy rescaling); row sums
    // in four fp16x2 partial sums per 64 keys, widened to fp32 once per block.
    uint32_t pk[BKV / 2];
    float rs = 0.f;
    {
      const float2 cc = make_float2(c, c), mm = make_float2(-m_used, -m_used);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        __half2 acc[4] = {__float2half2_rn(0.f), __float2half2_rn(0.f), __float2half2_rn(0.f),
                          __float2half2_rn(0.f)};
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int i = 64 * hf + 2 * q;
          const float2 xy = ffma2(make_float2(s[i], s[i + 1]), cc, mm);
          pk[32 * hf + q] = ex2_f16x2(pack_f16x2(xy.x, xy.y));
          acc[q & 3] = __hadd2(acc[q & 3], *reinterpret_cast<const __half2*>(&pk[32 * hf + q]));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(acc[k]);
          rs += f.x + f.y;
        }
      }
    }
    l = l * alpha + rs;
    if (DB && grow && j > 0) {  // O is stable once P(j-1) V_{j-1} has completed
      const bool wo = mbar_wait(o_done, (j - 1) & 1, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, wo)) {
        ok = false;
        break;
      }
      tc_fence_after();
    }
    if (grow && j > 0) {  // (two heads: P(j-1) V_{j-1} precedes S(j), so O is stable)
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + lane_off + cc * 32, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        tmem_st32(tO + lane_off + cc * 32, o);
      }
    }
    tmem_st64(tSj + lane_off, pk);  // key 2i (low half) and 2i+1 of P in column i
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(DB ? p_full + 8u * (j & 1) : p_full);
  }
  if (ok) {
    const bool w = DB ? mbar_wait(o_final, 0, p.err, abort_flag)
                      : mbar_wait(s_full, nkv & 1, p.err, abort_flag);  // the last P V product is done
    if (__all_sync(0xffffffffu, w)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const size_t orow = (static_cast<size_t>(wk.q_row0 + r) * p.batch + b) * p.ldo + h * D;
      if (p.lse != nullptr && row_ok)
        p.lse[(static_cast<size_t>(b) * p.nh + h) * p.seq + wk.q_row0 + r] = m_used + log2f(l);
      const float qs = p.o8 != nullptr ? __ldg(p.q_scale) : 1.f;
      float mx = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + lane_off + cc * 32, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= inv_l;
          if (p.o8 != nullptr) {  // E4M3 output for the FP8 output projection
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(o[i]));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint2*>(p.o8 + orow + cc * 32 + q4 * 8) = pack_e4m3x8(o + q4 * 8, qs);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint4*>(p.o + orow + cc * 32 + q4 * 8) = pack_bf16x8(o + q4 * 8);
          }
        }
      }
      if (p.o8 != nullptr) {
        mx = warp_max(mx);
        if (lane == 0) atomic_max_abs(p.amax, mx);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_tp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  constexpr int NH = 2;
  using G = GeoT<D, NH>;
  constexpr int NS = G::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + G::OFF_BAR);
  // bars: q_full | kv_full[NS] | kv_empty[NS] | s_full[2] | p_full[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6 + 2 * NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  // tile n of the load sequence (K_j = 2j, V_j = 2j + 1) sits in ring slot n % NS, in that slot's
  // (n / NS)-th use
  auto kv_full = [&](int n) { return bar0 + 8u * (1 + n % NS); };
  auto kv_empty = [&](int n) { return bar0 + 8u * (1 + NS + n % NS); };
  auto use_parity = [](int n) { return static_cast<uint32_t>((n / NS) & 1); };
  auto s_full = [&](int t) { return bar0 + 8u * (1 + 2 * NS + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (3 + 2 * NS + t); };
  const uint32_t drain = bar0 + 8u * (5 + 2 * NS);
  auto sQa = [&](int t) { return smem_u32(base + G::OFF_Q + t * G::Q_BYTES); };
  auto sKV = [&](int n) { return smem_u32(base + G::OFF_KV + (n % NS) * G::KV_BYTES); };

  pdl_wait();  // q, k, v (and cu_seqlens) are written by the kernels before
  pdl_trigger();
  Work wk;
  if (!decode_work(p, p.nh / NH, NH, wk)) return;  // uniform over the CTA, before any barrier or TMEM use
  const int qb = wk.qb, b = wk.b, h0 = wk.h;
  const int g = h0 / (p.nh / p.ng);  // both heads' kv group (an even number of heads per group)
  const int nkv = qb + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(kv_full(i), 1);
      mbar_init(kv_empty(i), 1);
    }
    for (int i = 0; i < NH; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto tS = [&](int t) { return tmem_base + 256u * t; };
  auto tO = [&](int t) { return tmem_base + 256u * t + 128u; };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, NH * G::Q_BYTES);
#pragma unroll
      for (int t = 0; t < NH; ++t)
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sQa(t) + a * G::ATOM, &tmQ, q_full, a * 64, wk.q_row0, b * p.nh + h0 + t);
      int issued = 0;
      bool ok = true;
      for (int n = 0; ok && n < 2 * nkv; ++n) {
        const CUtensorMap* map = (n & 1) ? &tmV : &tmK;
        if (!mbar_wait(kv_empty(n), use_parity(n) ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(kv_full(n), G::KV_BYTES);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sKV(n) + a * G::ATOM, map, kv_full(n), a * 64, wk.kv_row0 + (n >> 1) * BKV, b * p.ng + g);
        ++issued;
      }
      if (!ok) {  // let this CTA's own copies in flight land
        mbar_wait_slow(q_full, 0, nullptr, nullptr, kDrainLimitNs);
        for (int n = issued - 1; n >= 0 && n >= issued - NS; --n)
          mbar_wait_slow(kv_full(n), use_parity(n), nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      auto issue_s = [&](int t, int n) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * G::ATOM + (k & 3) * 32;
          mma_bf16_ss(tS(t), sw128_desc(sQa(t) + off), sw128_desc(sKV(n) + off), G::IDESC_S, k > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag) && mbar_wait(kv_full(0), use_parity(0), p.err, abort_flag);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NH; ++t) {
          issue_s(t, 0);
          mma_commit(s_full(t));
        }
        mma_commit(kv_empty(0));
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int nv = 2 * j + 1, nk = 2 * j + 2;  // tiles V_j and K_{j+1}
        // both tiles' waits back to back, ahead of the block's MMAs: a wait stops the MMA stream, and a
        // second wait right after the first costs far less than one between MMAs
        if (!mbar_wait(kv_full(nv), use_parity(nv), p.err, abort_flag) ||
            (j + 1 < nkv && !mbar_wait(kv_full(nk), use_parity(nk), p.err, abort_flag))) {
          ok = false;
          break;
        }
        for (int t = 0; t < NH && ok; ++t) {
          if (!mbar_wait(p_full(t), j & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BKV / 16; ++k)
            mma_f16_ts(tO(t), tS(t) + 8u * k, sw128_desc_mn(sKV(nv) + k * 2048, G::ATOM), G::IDESC_O,
                       (j > 0 || k > 0) ? 1u : 0u);
          if (j + 1 < nkv) issue_s(t, nk);
          mma_commit(s_full(t));
        }
        if (!ok) break;
        mma_commit(kv_empty(nv));
        if (j + 1 < nkv) mma_commit(kv_empty(nk));
      }
      mma_commit(drain);
      mbar_wait_slow(drain, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int t = (warp - 2) >> 2;  // which head of the pair
    softmax_head_tm<D>(p, wk, h0 + t, warp & 3, lane, tS(t), tO(t), s_full(t), p_full(t), abort_flag);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, G::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ one head, two score buffers
// attn_db_kernel: one head per CTA (an odd number of heads per group, or too few two-head CTAs),
// with two TMEM score buffers so that the tensor core computes S(j+1) while the softmax warps turn
// S(j) into P(j), and one thread of warp 1 issues, after S(0) and S(1):
//   per key block j: P(j) V_j (P from score buffer j % 2), then S(j+2) into the same buffer.
// The MMAs run in issue order, so S(j+2) overwrites P(j) only after P(j) V_j has read it.  A
// rescale of O in block j waits for P(j-1) V_{j-1} (o_done), which S(j) no longer implies.
// Every parity wait sees its barrier at most one phase from the awaited one: S(j) completing
// implies P(j-2) V_{j-2} completed, and S(j+2), P(j) V_j and a warp's block j+2 all wait for
// block j's P from every softmax warp.
//   TMEM: score buffers in columns [0, 128) and [128, 256), O in [256, 256 + d).
//   Tiles enter the ring in the order the MMAs use them: K0, K1, then V_j, K_{j+2} per block.
template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_db_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using G = GeoT<D, 1>;
  constexpr int NS = G::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + G::OFF_BAR);
  // bars: q_full | kv_full[NS] | kv_empty[NS] | s_full[2] | p_full[2] | o_done | o_final | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 + 2 * NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  // tile n of the load sequence sits in ring slot n % NS, in that slot's (n / NS)-th use
  auto kv_full = [&](int n) { return bar0 + 8u * (1 + n % NS); };
  auto kv_empty = [&](int n) { return bar0 + 8u * (1 + NS + n % NS); };
  auto use_parity = [](int n) { return static_cast<uint32_t>((n / NS) & 1); };
  const uint32_t s_full = bar0 + 8u * (1 + 2 * NS);  // buffer b's barrier at s_full + 8 b
  const uint32_t p_full = bar0 + 8u * (3 + 2 * NS);  // block j's at p_full + 8 (j & 1)
  const uint32_t o_done = bar0 + 8u * (5 + 2 * NS);
  const uint32_t o_final = bar0 + 8u * (6 + 2 * NS);
  const uint32_t drain = bar0 + 8u * (7 + 2 * NS);
  const uint32_t sQ = smem_u32(base + G::OFF_Q);
  auto sKV = [&](int n) { return smem_u32(base + G::OFF_KV + (n % NS) * G::KV_BYTES); };

  pdl_wait();  // q, k, v (and cu_seqlens) are written by the kernels before
  pdl_trigger();
  Work wk;
  if (!decode_work(p, p.nh, 1, wk)) return;  // uniform over the CTA, before any barrier or TMEM use
  const int qb = wk.qb, b = wk.b, h = wk.h;
  const int g = h / (p.nh / p.ng);
  const int nkv = qb + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(kv_full(i), 1);
      mbar_init(kv_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8u * i, 1);
      mbar_init(p_full + 8u * i, 4);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tS = tmem_base, tO = tmem_base + 256u;  // score buffer b at tS + 128 b

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, G::Q_BYTES);
#pragma unroll
      for (int a = 0; a < D / 64; ++a) tma_load_3d(sQ + a * G::ATOM, &tmQ, q_full, a * 64, wk.q_row0, b * p.nh + h);
      int n = 0;
      // one tile (K or V of key block kb) into the next ring slot
      auto load = [&](const CUtensorMap* map, int kb) {
        if (!mbar_wait(kv_empty(n), use_parity(n) ^ 1u, p.err, abort_flag)) return false;
        mbar_arrive_expect_tx(kv_full(n), G::KV_BYTES);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sKV(n) + a * G::ATOM, map, kv_full(n), a * 64, wk.kv_row0 + kb * BKV, b * p.ng + g);
        ++n;
        return true;
      };
      bool ok = load(&tmK, 0) && (nkv < 2 || load(&tmK, 1));
      for (int j = 0; ok && j < nkv; ++j) ok = load(&tmV, j) && (j + 2 >= nkv || load(&tmK, j + 2));
      if (!ok) {  // let this CTA's own copies in flight land
        mbar_wait_slow(q_full, 0, nullptr, nullptr, kDrainLimitNs);
        for (int m = n - 1; m >= 0 && m >= n - NS; --m)
          mbar_wait_slow(kv_full(m), use_parity(m), nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int n = 0;  // next tile of the load sequence
      auto issue_s = [&](int buf) {  // S into score buffer `buf` from the K tile n
        const uint32_t ks = sKV(n);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * G::ATOM + (k & 3) * 32;
          mma_bf16_ss(tS + 128u * buf, sw128_desc(sQ + off), sw128_desc(ks + off), G::IDESC_S, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full + 8u * buf);
        mma_commit(kv_empty(n));
        ++n;
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag) && mbar_wait(kv_full(0), use_parity(0), p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        if (nkv > 1) {
          ok = mbar_wait(kv_full(n), use_parity(n), p.err, abort_flag);
          if (ok) issue_s(1);
        }
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int buf = j & 1;
        if (!mbar_wait(kv_full(n), use_parity(n), p.err, abort_flag) ||  // V_j
            !mbar_wait(p_full + 8u * buf, (j >> 1) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vs = sKV(n);
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k)
          mma_f16_ts(tO, tS + 128u * buf + 8u * k, sw128_desc_mn(vs + k * 2048, G::ATOM), G::IDESC_O,
                     (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(o_done);
        if (j + 1 == nkv) mma_commit(o_final);
        mma_commit(kv_empty(n));
        ++n;
        if (j + 2 < nkv) {
          if (!mbar_wait(kv_full(n), use_parity(n), p.err, abort_flag)) {  // K_{j+2}
            ok = false;
            break;
          }
          issue_s(buf);
        }
      }
      mma_commit(drain);
      mbar_wait_slow(drain, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    softmax_head_tm<D, true>(p, wk, h, warp & 3, lane, tS, tO, s_full, p_full, abort_flag, o_done, o_final);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, G::TMEM_COLS);
  }
}

template <int D, int NH>
cudaError_t launch_tp(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p,
                      cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(NH == 2 ? attn_tp_kernel<D> : attn_db_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(GeoT<D, NH>::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned grid = static_cast<unsigned>(p.num_qb) * (p.cu ? p.num_seqs : p.batch) * (p.nh / NH);
  return launch_pdl(NH == 2 ? attn_tp_kernel<D> : attn_db_kernel<D>, dim3(grid), dim3(64 + 128 * NH),
                    GeoT<D, NH>::SMEM, stream, tmQ, tmK, tmV, p);
}

template <int D, bool TG>
cudaError_t launch_d2(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p,
                      cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn2_kernel<D, TG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Geo2<D, TG>::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned grid = static_cast<unsigned>(p.num_qb) * (p.cu ? p.num_seqs : p.batch) * (p.nh / 2);
  return launch_pdl(attn2_kernel<D, TG>, dim3(grid), dim3(320), Geo2<D, TG>::SMEM, stream, tmQ, tmK, tmV, p);
}

// Heads per CTA (set_attention_heads_mode): 0 automatic, 1 one head always, 2 two heads wherever
// the form allows.
std::atomic<int> g_heads_mode{0};

}  // namespace

void set_attention_heads_mode(int mode) { g_heads_mode.store(mode); }

cudaError_t launch_attention(int head_dim, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, cudaStream_t stream) {
  if (p.num_qb <= 0) return cudaSuccess;
  if (head_dim != 64 && head_dim != 128) return cudaErrorInvalidValue;
  const int mode = g_heads_mode.load();
  const bool even = ((p.nh / p.ng) & 1) == 0;  // an even number of query heads per kv group
  // d = 64 with an odd number of heads per group (MHA): two heads of two groups per CTA
  if (mode != 1 && head_dim == 64 && !even && (p.nh & 1) == 0) return launch_d2<64, true>(tmQ, tmK, tmV, p, stream);
  // two heads of one group per CTA when the two-head CTAs fill the SMs at least twice over
  const long pair_ctas = static_cast<long>(p.num_qb) * (p.cu ? p.num_seqs : p.batch) * (p.nh / 2);
  if (even && mode != 1 && (mode == 2 || pair_ctas >= 2L * num_sms()))
    return head_dim == 64 ? launch_tp<64, 2>(tmQ, tmK, tmV, p, stream) : launch_tp<128, 2>(tmQ, tmK, tmV, p, stream);
  return head_dim == 64 ? launch_tp<64, 1>(tmQ, tmK, tmV, p, stream) : launch_tp<128, 1>(tmQ, tmK, tmV, p, stream);
}

}  // namespace mt
