// Backward pass of the causal GQA attention, flash-style: P and dS are formed tile by tile on
// chip from the forward's per-row log-sum-exp and never reach memory
// (training step of "ai阅读megatron"; activation recompute, "快速入门" §8).  For one head, with
// scores S = Q K^T, P = softmax(S / sqrt(d)) and D_i = dO_i . O_i:
//     dS = P o (dP - D) / sqrt(d),  dP = dO V^T,
//     dV = P^T dO,  dK = dS^T Q,  dQ = dS K   (dK, dV summed over the query heads of a group).
// Two kernels, each a producer warp (TMA), two MMA-issuing threads (tcgen05: one for the score
// products, one for the gradient products, so that neither's waits stall the other) and sixteen
// elementwise warps (one row per thread, four warps per TMEM lane quadrant):
//   attn_bwd_dq_kernel:   one CTA per (128 queries, head); steps over 128-key blocks j <= i:
//                         Q in TMEM, S and dP into TMEM, dS (bf16) into TMEM, dQ += dS K in TMEM.
//   attn_bwd_dkdv_kernel: one CTA per (128 keys, kv group, run); steps over the group's heads and
//                         the 64-query blocks i >= j: S^T and dP^T into TMEM, P^T and dS^T (bf16) into
//                         TMEM, dV += P^T dO and dK += dS^T Q in TMEM.  With kv_parts > 1 the steps of
//                         a (key block, group) are cut into that many runs on separate CTAs, each
//                         writing partial sums to its own dK/dV buffer (the caller adds them).
// The two kernels share no output, so the caller may run them on two streams at once.
// The caller provides head-major copies of dO and V (dO by head_slices_kernel below); the second operands of the
// gradient products (K for dQ, dO for dV, Q for dK) are the tiles already staged for the score
// products, read as MN-major operands.
#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

constexpr int ATOM128 = 128 * 128;  // [128 rows x 64] bf16 block with the 128-byte swizzle, 16 KB
constexpr int ATOM64 = 64 * 128;    // [64 rows x 64] block, 8 KB

// `desc` advanced by `bytes` (a multiple of 16): the start-address field holds (address & 0x3FFFF) >> 4
// and no shared-memory address of a CTA reaches 2^18, so the advance is a plain add that never
// carries out of the field.  Lets a loop build each descriptor once and step it.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// ------------------------------------------------------------------ prep
// Batched copy of the R x C slices src_z = src + (z / zdiv) * sb + (z % zdiv) * sh (row pitch sp) into
// dst + z R dp (row pitch dp): the head-major copy of dO.
__global__ void head_slices_kernel(const bf16* __restrict__ src, size_t sp, size_t sb, size_t sh, int zdiv,
                                   bf16* __restrict__ dst, size_t dp, int R, int C) {
  const int z = blockIdx.z;
  const uint16_t* s = reinterpret_cast<const uint16_t*>(src + (z / zdiv) * sb + (z % zdiv) * sh);
  uint16_t* d = reinterpret_cast<uint16_t*>(dst) + static_cast<size_t>(z) * R * dp;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) d[static_cast<size_t>(r) * dp + c] = s[static_cast<size_t>(r) * sp + c];
  }
}

// The same copy, 16 bytes (8 columns) per thread, when C, the pitches and the slice offsets are
// multiples of 8 elements (16-byte aligned rows): x indexes 8-column groups, y rows.
__global__ void head_slices_vec_kernel(const bf16* __restrict__ src, size_t sp, size_t sb, size_t sh, int zdiv,
                                       bf16* __restrict__ dst, size_t dp, int R, int C8) {
  const int z = blockIdx.z;
  const bf16* s = src + (z / zdiv) * sb + (z % zdiv) * sh;
  bf16* d = dst + static_cast<size_t>(z) * R * dp;
  const int c = blockIdx.x * blockDim.x + threadIdx.x, r = blockIdx.y * blockDim.y + threadIdx.y;
  if (r < R && c < C8)
    *reinterpret_cast<uint4*>(d + static_cast<size_t>(r) * dp + 8 * c) =
        *reinterpret_cast<const uint4*>(s + static_cast<size_t>(r) * sp + 8 * c);
}

// D[(b * nh + h) * S + s] = sum_c dO[s b, h c] * O[s b, h c]  (both [S * B, nh * d] bf16, d = 64 or
// 128): d / 8 lanes per (token, head), each taking 8 columns, so a warp covers 32 / (d / 8) rows.
__global__ void row_dot_kernel(const bf16* __restrict__ dO, const bf16* __restrict__ O, float* __restrict__ Dsum,
                               int S, int B, int nh, int d) {
  const int L = d >> 3;  // lanes per row, a power of two dividing 32
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t rowi = tid / L;
  const int sub = static_cast<int>(tid % L);
  const size_t rows = static_cast<size_t>(S) * B * nh;
  const int h = static_cast<int>(rowi % nh);
  const size_t t = rowi / nh;  // token s * B + b
  float acc = 0.f;
  if (rowi < rows) {
    const size_t off = t * static_cast<size_t>(nh) * d + static_cast<size_t>(h) * d + sub * 8;
    float a[8], o[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(dO + off), a);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(O + off), o);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += a[e] * o[e];
  }
  for (int o = L >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);  // inside the row's lanes
  if (rowi < rows && sub == 0) {
    const int b = static_cast<int>(t % B), s = static_cast<int>(t / B);
    Dsum[(static_cast<size_t>(b) * nh + h) * S + s] = acc;
  }
}

// Bounded wait shared by the roles below (records the error and raises the CTA's abort flag).
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, int* err, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ dQ
// One CTA per (128 queries, head), stepping over the 128-key blocks j <= i, so that every product
// has N = 128 (N = d for dQ).  Q moves to tensor memory once, as the A operand of S, and the
// elementwise warps write dS there too, as the A operand of dQ += dS K (two bf16 per 32-bit
// column): the tensor core then reads only K, V and dO from shared memory, which holds dO, a
// three-slot K ring and a two-slot V ring.  K_j feeds S_j (read K-major) and, one step later,
// dQ += dS_j K_j (read MN-major), so its slot is released after that; V_j feeds dP_j only.  One
// barrier per step (two in turn) completes when both K_j and V_j have landed.
//   TMEM: S [0, 128), dP [128, 256), dQ [256, 256 + d), Q [384, 384 + d/2), dS [448, 512).
//   Two issuing threads: warp 1 issues S_n and dP_n for every step, the last warp dQ += dS_n K_n once
//   dS_n is written, so that neither's waits stall the other's products; a K slot is free once
//   both have committed its last product.
//   Sixteen elementwise warps, four per TMEM lane quadrant, each taking 32 of a step's 128 columns.
template <int D>
struct GeoQ {
  static constexpr int QD_BYTES = 128 * D * 2;      // Q_i or dO_i: D/64 blocks of [128 x 64]
  static constexpr int KV_BYTES = 128 * D * 2;      // K_j or V_j: D/64 blocks of [128 x 64]
  static constexpr int NK = 3, NV = 2;              // K and V ring slots
  static constexpr int OFF_DO = 0;
  static constexpr int OFF_QS = QD_BYTES;           // Q, on its way to tensor memory
  static constexpr int OFF_K = OFF_QS + QD_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
  static constexpr size_t SMEM_USED = 1024 + OFF_BAR + 256;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;  // one CTA per SM (TMEM)
  static constexpr int EW = 16;                     // elementwise warps
  static constexpr int THREADS = 96 + 32 * EW;      // producer, S/dP issuer, elementwise, dQ issuer
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128);
  static constexpr uint32_t IDESC_Q = idesc_bf16_bmn(128, D);  // B = K_j read MN-major
};
static_assert(GeoQ<128>::SMEM_USED <= 232448, "dQ tiles exceed the shared memory of a CTA");

// Each thread writes 16 consecutive 32-bit columns of its own TMEM lane and waits for the write.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(GeoQ<D>::THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const AttnBwdParams p) {
  using G = GeoQ<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + G::OFF_BAR);
  // bars: q_full | kv_full[2] | k_empty[3] | v_empty[2] | q_tm | s_full | s_free | ds_full | ds_free | done | sp_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0, q_tm = bar0 + 8u * 8, s_full = bar0 + 8u * 9, s_free = bar0 + 8u * 10,
                 ds_full = bar0 + 8u * 11, ds_free = bar0 + 8u * 12, done = bar0 + 8u * 13, sp_done = bar0 + 8u * 14;
  auto kv_full = [&](int n) { return bar0 + 8u * (1 + (n & 1)); };
  auto k_empty = [&](int n) { return bar0 + 8u * (3 + n % G::NK); };
  auto v_empty = [&](int n) { return bar0 + 8u * (6 + n % G::NV); };
  const uint32_t sDO = smem_u32(base + G::OFF_DO), sQS = smem_u32(base + G::OFF_QS);
  auto sK = [&](int n) { return smem_u32(base + G::OFF_K + (n % G::NK) * G::KV_BYTES); };
  auto sV = [&](int n) { return smem_u32(base + G::OFF_V + (n % G::NV) * G::KV_BYTES); };

  pdl_wait();
  pdl_trigger();
  const int per = p.batch * p.nh;
  const int qb = p.num_qb - 1 - static_cast<int>(blockIdx.x) / per;  // longest rows first
  const int zq = static_cast<int>(blockIdx.x) % per;                  // b * nh + h
  const int b = zq / p.nh, h = zq % p.nh;
  const int zk = b * p.ng + h / (p.nh / p.ng);
  const int nst = qb + 1;  // 128-key blocks j <= qb (keys past seq arrive as zeros and are masked)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(kv_full(0), 1);
    mbar_init(kv_full(1), 1);
    for (int i = 0; i < G::NK; ++i) mbar_init(k_empty(i), 2);  // after S_n (warp 1) and dQ_n (last warp)
    for (int i = 0; i < G::NV; ++i) mbar_init(v_empty(i), 1);
    mbar_init(q_tm, D / 8);  // the warps that move Q: D/32 per lane quadrant
    mbar_init(s_full, 1);
    mbar_init(s_free, G::EW);
    mbar_init(ds_full, G::EW);
    mbar_init(ds_free, 1);
    mbar_init(done, 1);
    mbar_init(sp_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmDO);
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
  const uint32_t tS = tmem_base, tP = tmem_base + 128u, tQ = tmem_base + 256u, tQa = tmem_base + 384u,
                 tDS = tmem_base + 448u;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * G::QD_BYTES);
#pragma unroll
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(sQS + a * ATOM128, &tmQ, q_full, a * 64, qb * 128, zq);
        tma_load_3d(sDO + a * ATOM128, &tmDO, q_full, a * 64, qb * 128, zq);
      }
      int issued = 0;
      bool ok = true;
      for (int n = 0; n < nst; ++n) {
        if (!mbar_wait(k_empty(n), ((n / G::NK) & 1) ^ 1u, p.err, abort_flag) ||
            !mbar_wait(v_empty(n), ((n / G::NV) & 1) ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(kv_full(n), 2 * G::KV_BYTES);
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(sK(n) + a * ATOM128, &tmK, kv_full(n), a * 64, n * 128, zk);
          tma_load_3d(sV(n) + a * ATOM128, &tmV, kv_full(n), a * 64, n * 128, zk);
        }
        ++issued;
      }
      if (!ok) {  // let this CTA's own copies in flight land
        mbar_wait_slow(q_full, 0, nullptr, nullptr, kDrainLimitNs);
        for (int n = issued - 1; n >= 0 && n >= issued - 2; --n)
          mbar_wait_slow(kv_full(n), (n >> 1) & 1, nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // S_n = Q K_n^T (Q from tensor memory) and dP_n = dO V_n^T
      uint64_t ddo[D / 16];  // dO stays put: its descriptors are built once
#pragma unroll
      for (int k = 0; k < D / 16; ++k) ddo[k] = sw128_desc(sDO + (k >> 2) * ATOM128 + (k & 3) * 32);
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag) && mbar_wait(q_tm, 0, p.err, abort_flag);
      for (int n = 0; ok && n < nst; ++n) {
        if (!mbar_wait(kv_full(n), (n >> 1) & 1, p.err, abort_flag) ||
            (n >= 1 && !mbar_wait(s_free, (n - 1) & 1, p.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = sw128_desc(sK(n)), dv = sw128_desc(sV(n));
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_f16_ts(tS, tQa + 8u * k, desc_add(dk, (k >> 2) * ATOM128 + (k & 3) * 32), G::IDESC_S, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_bf16_ss(tP, ddo[k], desc_add(dv, (k >> 2) * ATOM128 + (k & 3) * 32), G::IDESC_S, k > 0 ? 1u : 0u);
        mma_commit(s_full);
        mma_commit(v_empty(n));
        mma_commit(k_empty(n));
      }
      mma_commit(sp_done);
      mbar_wait_slow(sp_done, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else if (warp == 2 + G::EW) {
    if (lane == 0) {  // dQ += dS_m K_m, dS from tensor memory, K_m read MN-major
      bool ok = true;
      for (int m = 0; ok && m < nst; ++m) {
        if (!mbar_wait(ds_full, m & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = sw128_desc_mn(sK(m), ATOM128);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ts(tQ, tDS + 8u * k, desc_add(dk, k * 2048), G::IDESC_Q, (m > 0 || k > 0) ? 1u : 0u);
        mma_commit(ds_free);
        mma_commit(k_empty(m));
      }
      mma_commit(done);
      mbar_wait_slow(done, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int quad = warp & 3, c4 = (warp - 2) >> 2;  // columns [32 c4, 32 c4 + 32) of a step
    const int r = quad * 32 + lane;
    const int qi = qb * 128 + r;  // query row
    const bool row_ok = qi < p.seq;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const size_t rix = static_cast<size_t>(zq) * p.seq + qi;
    // P / sqrt(d) = 2^(s c - lse + log2(1/sqrt(d))): the scale folds into the exponent; a row past
    // seq gets P = 0 through lse = +inf
    const float lse = row_ok ? p.lse[rix] - log2f(p.scale) : __int_as_float(0x7f800000);
    const float dsum = row_ok ? p.dsum[rix] : 0.f;
    bool ok = true;
    if (c4 < D / 32) {  // Q into tensor memory: this warp's 32 elements as 16 columns of bf16 pairs
      ok = wait_all(q_full, 0, p.err, abort_flag);
      if (ok) {
        const uint8_t* row = base + G::OFF_QS + (c4 >> 1) * ATOM128 + r * 128;
        uint32_t w[16];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + (((4 * (c4 & 1) + ch) ^ (r & 7)) << 4));
          w[4 * ch] = v.x;
          w[4 * ch + 1] = v.y;
          w[4 * ch + 2] = v.z;
          w[4 * ch + 3] = v.w;
        }
        tmem_st16(tQa + lane_off + 16 * c4, w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_tm);
      }
    }
    for (int n = 0; ok && n < nst; ++n) {
      if (!wait_all(s_full, n & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t su[32], du[32];
      tmem_ld32_issue(tS + lane_off + 32 * c4, su);
      tmem_ld32_issue(tP + lane_off + 32 * c4, du);
      tmem_ld32_wait(su);
      tmem_ld32_wait(du);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      uint32_t w[16];  // dS as bf16 pairs
      if (n < qb) {  // below the diagonal block every key is visible
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = ex2_approx(__uint_as_float(su[c]) * p.scale_log2 - lse);
          const float p1 = ex2_approx(__uint_as_float(su[c + 1]) * p.scale_log2 - lse);
          w[c >> 1] = pack_bf16x2(p0 * (__uint_as_float(du[c]) - dsum), p1 * (__uint_as_float(du[c + 1]) - dsum));
        }
      } else {
        const int key0 = n * 128 + 32 * c4;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = key0 + c <= qi ? ex2_approx(__uint_as_float(su[c]) * p.scale_log2 - lse) : 0.f;
          const float p1 = key0 + c + 1 <= qi ? ex2_approx(__uint_as_float(su[c + 1]) * p.scale_log2 - lse) : 0.f;
          w[c >> 1] = pack_bf16x2(p0 * (__uint_as_float(du[c]) - dsum), p1 * (__uint_as_float(du[c + 1]) - dsum));
        }
      }
      if (n >= 1 && !wait_all(ds_free, (n - 1) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      tmem_st16(tDS + lane_off + 16 * c4, w);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    if (ok && wait_all(done, 0, p.err, abort_flag)) {
      tc_fence_after();
      if (c4 < D / 32) {
        float v[32];
        tmem_ld32(tQ + lane_off + 32 * c4, v);
        if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(p.dq + rix * D + 32 * c4);
#pragma unroll
          for (int g = 0; g < 8; ++g) dst[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ dK, dV
// One CTA per (128 keys, kv group), stepping over the group's heads and, per head, the 64-query
// blocks i >= j.  K and V stay in shared memory (the A operands of S^T = K Q^T and dP^T = V dO^T);
// a ring of Q and dO blocks feeds those products (read K-major) and the gradient products
// dV += P^T dO and dK += dS^T Q (read MN-major).  S^T and dP^T are double-buffered in tensor
// memory; the elementwise warps write P^T over S^T and dS^T over dP^T (bf16 pairs in the first 32
// columns of each), the A operands of the gradient products, and the sums over the group's heads
// happen in the dV and dK accumulators.
//   TMEM: buffer b: S^T [128 b, 128 b + 64), dP^T [128 b + 64, 128 b + 128); dV [256, 256 + d),
//         dK [384, 384 + d).
//   Two issuing threads: warp 1 issues S^T_n and dP^T_n into buffer n % 2 once the gradient
//   products of step n - 2 have read it, the last warp dV and dK once P^T_n and dS^T_n are written;
//   a ring slot is free once both have committed its last product.
//   Sixteen elementwise warps, four per TMEM lane quadrant, each taking 16 of a step's 64 columns;
//   the four warps of a quadrant meet at a named barrier between reading S^T, dP^T and writing
//   P^T, dS^T over them (a warp's P^T columns hold other warps' S^T columns).
template <int D>
struct GeoKV {
  static constexpr int KV_BYTES = 128 * D * 2;            // K_j or V_j: D/64 blocks of [128 x 64]
  static constexpr int QD_BYTES = 64 * D * 2;             // Q_i or dO_i: D/64 blocks of [64 x 64]
  static constexpr int STAGE = 2 * QD_BYTES;
  static constexpr int NSTG = D == 128 ? 5 : 8;           // query blocks in flight
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_BYTES;
  static constexpr int OFF_ST = 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_ST + NSTG * STAGE;
  static constexpr size_t SMEM_USED = 1024 + OFF_BAR + 256;
  static constexpr size_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr int EW = 16;
  static constexpr int THREADS = 96 + 32 * EW;            // producer, S/dP issuer, elementwise, gradient issuer
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 64);
  static constexpr uint32_t IDESC_G = idesc_bf16_bmn(128, D);  // B = dO_i or Q_i read MN-major
};
static_assert(GeoKV<128>::SMEM_USED <= 232448, "dK/dV tiles exceed the shared memory of a CTA");

// 16 consecutive fp32 columns of the thread's TMEM lane, split into issue and wait (see tmem_ld32_issue).
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}
// Each thread writes 8 consecutive 32-bit columns of its own TMEM lane (no wait).
__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier of the four elementwise warps that share TMEM lane quadrant q (ids 1-4).
__device__ __forceinline__ void quad_sync(int q) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + q) : "memory");
}

template <int D>
__global__ void __launch_bounds__(GeoKV<D>::THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                         const AttnBwdParams p) {
  using G = GeoKV<D>;
  constexpr int NS = G::NSTG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + G::OFF_BAR);
  // bars: kv_full | st_full[NS] | st_empty[NS] | s_full[2] | pt_full[2] | g_done[2] | done | sp_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9 + 2 * NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t kv_full = bar0, done = bar0 + 8u * (7 + 2 * NS), sp_done = bar0 + 8u * (8 + 2 * NS);
  // step n uses buffer n & 1; its barriers complete phase n / 2
  auto s_full = [&](int n) { return bar0 + 8u * (1 + 2 * NS + (n & 1)); };
  auto pt_full = [&](int n) { return bar0 + 8u * (3 + 2 * NS + (n & 1)); };
  auto g_done = [&](int n) { return bar0 + 8u * (5 + 2 * NS + (n & 1)); };
  auto st_full = [&](int n) { return bar0 + 8u * (1 + n % NS); };
  auto st_empty = [&](int n) { return bar0 + 8u * (1 + NS + n % NS); };
  const uint32_t sK = smem_u32(base + G::OFF_K), sV = smem_u32(base + G::OFF_V);
  auto sQ = [&](int n) { return smem_u32(base + G::OFF_ST + (n % NS) * G::STAGE); };
  auto sDO = [&](int n) { return smem_u32(base + G::OFF_ST + (n % NS) * G::STAGE + G::QD_BYTES); };

  pdl_wait();
  pdl_trigger();
  const int per = p.batch * p.ng * p.kv_parts;
  const int kb = static_cast<int>(blockIdx.x) / per;  // key block 0 has the most query blocks
  const int zk = static_cast<int>(blockIdx.x) % per / p.kv_parts;  // b * ng + g
  const int part = static_cast<int>(blockIdx.x) % p.kv_parts;
  const int b = zk / p.ng, g = zk % p.ng;
  const int rep = p.nh / p.ng;
  const int nq64 = (p.seq + 63) / 64;
  const int i0 = 2 * kb;            // first 64-query block that sees a key of this block
  const int per_head = nq64 - i0;   // >= 1 for every launched key block
  // steps (head of the group, query block), flattened; this CTA takes the run [n0, n0 + nst), which
  // is not empty (the launcher cuts at most as many runs as the shortest key block has steps)
  const int n0 = part * (rep * per_head) / p.kv_parts;
  const int nst = (part + 1) * (rep * per_head) / p.kv_parts - n0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(st_full(i), 1);
      mbar_init(st_empty(i), 2);  // after S^T/dP^T (warp 1) and after dV/dK (last warp)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(pt_full(i), G::EW);
      mbar_init(g_done(i), 1);
    }
    mbar_init(done, 1);
    mbar_init(sp_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
    tma_prefetch(&tmQ);
    tma_prefetch(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto tS = [&](int n) { return tmem_base + 128u * (n & 1); };        // S^T, then P^T
  auto tP = [&](int n) { return tmem_base + 128u * (n & 1) + 64u; };  // dP^T, then dS^T
  const uint32_t tV = tmem_base + 256u, tK = tmem_base + 384u;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * G::KV_BYTES);
#pragma unroll
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(sK + a * ATOM128, &tmK, kv_full, a * 64, kb * 128, zk);
        tma_load_3d(sV + a * ATOM128, &tmV, kv_full, a * 64, kb * 128, zk);
      }
      int issued = 0;
      bool ok = true;
      for (int n = 0; n < nst; ++n) {
        const int zq = b * p.nh + g * rep + (n0 + n) / per_head;
        const int qi0 = (i0 + (n0 + n) % per_head) * 64;
        if (!mbar_wait(st_empty(n), ((n / NS) & 1) ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(st_full(n), G::STAGE);
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(sQ(n) + a * ATOM64, &tmQ, st_full(n), a * 64, qi0, zq);
          tma_load_3d(sDO(n) + a * ATOM64, &tmDO, st_full(n), a * 64, qi0, zq);
        }
        ++issued;
      }
      if (!ok) {
        mbar_wait_slow(kv_full, 0, nullptr, nullptr, kDrainLimitNs);
        for (int n = issued - 1; n >= 0 && n >= issued - NS; --n)
          mbar_wait_slow(st_full(n), (n / NS) & 1, nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // S^T = K Q^T and dP^T = V dO^T for one 64-query block
      uint64_t dk[D / 16], dv[D / 16];  // K and V stay put: their descriptors are built once
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        dk[k] = sw128_desc(sK + (k >> 2) * ATOM128 + (k & 3) * 32);
        dv[k] = sw128_desc(sV + (k >> 2) * ATOM128 + (k & 3) * 32);
      }
      bool ok = mbar_wait(kv_full, 0, p.err, abort_flag);
      for (int n = 0; ok && n < nst; ++n) {
        if (!mbar_wait(st_full(n), (n / NS) & 1, p.err, abort_flag) ||
            (n >= 2 && !mbar_wait(g_done(n), ((n >> 1) - 1) & 1, p.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dq = sw128_desc(sQ(n)), ddo = sw128_desc(sDO(n));
        const uint32_t ts = tS(n), tp = tP(n);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_bf16_ss(ts, dk[k], desc_add(dq, (k >> 2) * ATOM64 + (k & 3) * 32), G::IDESC_S, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_bf16_ss(tp, dv[k], desc_add(ddo, (k >> 2) * ATOM64 + (k & 3) * 32), G::IDESC_S, k > 0 ? 1u : 0u);
        mma_commit(s_full(n));
        mma_commit(st_empty(n));
      }
      mma_commit(sp_done);
      mbar_wait_slow(sp_done, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else if (warp == 2 + G::EW) {
    if (lane == 0) {  // dV += P^T dO and dK += dS^T Q (P^T, dS^T from tensor memory; dO, Q MN-major)
      bool ok = true;
      for (int m = 0; ok && m < nst; ++m) {
        if (!mbar_wait(pt_full(m), (m >> 1) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dq = sw128_desc_mn(sQ(m), ATOM64), ddo = sw128_desc_mn(sDO(m), ATOM64);
        const uint32_t ts = tS(m), tp = tP(m);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ts(tV, ts + 8u * k, desc_add(ddo, k * 2048), G::IDESC_G, (m > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ts(tK, tp + 8u * k, desc_add(dq, k * 2048), G::IDESC_G, (m > 0 || k > 0) ? 1u : 0u);
        mma_commit(g_done(m));
        mma_commit(st_empty(m));
      }
      mma_commit(done);
      mbar_wait_slow(done, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int quad = warp & 3, c4 = (warp - 2) >> 2;  // query columns [16 c4, 16 c4 + 16) of a step
    const int r = quad * 32 + lane;
    const int kj = kb * 128 + r;  // key row
    const bool row_ok = kj < p.seq;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // the statistics of a step's columns come by 16-byte loads when rows are 16-byte aligned
    const bool vec = (p.seq & 3) == 0 && (reinterpret_cast<uintptr_t>(p.lse) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.dsum) & 15) == 0;
    // every warp of a quadrant passes the quadrant barrier once per step, also after a failed wait
    // (it then skips the step's work), so that no warp is left at the barrier
    bool ok = true;
    for (int n = 0; n < nst; ++n) {
      if (!ok) {
        quad_sync(quad);
        continue;
      }
      const int zq = b * p.nh + g * rep + (n0 + n) / per_head;
      const int qc0 = (i0 + (n0 + n) % per_head) * 64 + 16 * c4;  // this warp's first query column
      // the 16 columns' row statistics, the same for every lane (one broadcast load each); columns
      // past seq read the last row's (their P^T and dS^T multiply zero rows of dO and Q)
      // dsum is kept as D / sqrt(d), so that dS^T = P^T (dP^T / sqrt(d) - D / sqrt(d)) is one FMA and a product
      float lse[16], dsum[16];
      const size_t s0 = static_cast<size_t>(zq) * p.seq;
      if (vec && qc0 + 16 <= p.seq) {
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(p.lse + s0 + qc0 + c));
          const float4 d = __ldg(reinterpret_cast<const float4*>(p.dsum + s0 + qc0 + c));
          lse[c] = a.x;
          lse[c + 1] = a.y;
          lse[c + 2] = a.z;
          lse[c + 3] = a.w;
          dsum[c] = d.x * p.scale;
          dsum[c + 1] = d.y * p.scale;
          dsum[c + 2] = d.z * p.scale;
          dsum[c + 3] = d.w * p.scale;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int q = min(qc0 + c, p.seq - 1);
          lse[c] = __ldg(p.lse + s0 + q);
          dsum[c] = __ldg(p.dsum + s0 + q) * p.scale;
        }
      }
      if (!wait_all(s_full(n), (n >> 1) & 1, p.err, abort_flag)) {
        ok = false;
        quad_sync(quad);
        continue;
      }
      tc_fence_after();
      const uint32_t ts = tS(n) + lane_off, tp = tP(n) + lane_off;
      uint32_t su[16], du[16];
      tmem_ld16_issue(ts + 16 * c4, su);
      tmem_ld16_issue(tp + 16 * c4, du);
      tmem_ld16_wait(su);
      tmem_ld16_wait(du);
      tc_fence_before();
      quad_sync(quad);  // the quadrant's four warps have read S^T and dP^T
      tc_fence_after();
      uint32_t wp[8], wd[8];  // P^T and dS^T as bf16 pairs
      const bool below = qc0 >= kb * 128 + 127;  // every key of the block precedes every query of these columns
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        float p0 = ex2_approx(__uint_as_float(su[c]) * p.scale_log2 - lse[c]);
        float p1 = ex2_approx(__uint_as_float(su[c + 1]) * p.scale_log2 - lse[c + 1]);
        if (!below) {
          p0 = qc0 + c >= kj ? p0 : 0.f;
          p1 = qc0 + c + 1 >= kj ? p1 : 0.f;
        }
        wp[c >> 1] = pack_bf16x2(p0, p1);
        wd[c >> 1] = pack_bf16x2(p0 * fmaf(__uint_as_float(du[c]), p.scale, -dsum[c]),
                                 p1 * fmaf(__uint_as_float(du[c + 1]), p.scale, -dsum[c + 1]));
      }
      tmem_st8_nowait(ts + 8 * c4, wp);
      tmem_st8_nowait(tp + 8 * c4, wd);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pt_full(n));
    }
    if (ok && wait_all(done, 0, p.err, abort_flag)) {
      tc_fence_after();
      const size_t row = static_cast<size_t>(zk) * p.seq + kj;
      constexpr int W = D / 4;  // columns of dV and dK per warp
      float v[W], k32[W];
      if (W == 32) {
        tmem_ld32(tV + lane_off + W * c4, v);
        tmem_ld32(tK + lane_off + W * c4, k32);
      } else {
        uint32_t a[16], c[16];
        tmem_ld16_issue(tV + lane_off + W * c4, a);
        tmem_ld16_issue(tK + lane_off + W * c4, c);
        tmem_ld16_wait(a);
        tmem_ld16_wait(c);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[i] = __uint_as_float(a[i]);
          k32[i] = __uint_as_float(c[i]);
        }
      }
      if (row_ok) {
        const size_t off = part * p.part_stride + row * D + W * c4;  // this run's partial sums
        float4* dv = reinterpret_cast<float4*>(p.dv + off);
        float4* dk = reinterpret_cast<float4*>(p.dk + off);
#pragma unroll
        for (int q = 0; q < W / 4; ++q) {
          dv[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          dk[q] = make_float4(k32[4 * q], k32[4 * q + 1], k32[4 * q + 2], k32[4 * q + 3]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap* maps, const AttnBwdParams& p, cudaStream_t st, cudaStream_t st_dq) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(GeoQ<D>::SMEM));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(GeoKV<D>::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned nb = static_cast<unsigned>((p.seq + 127) / 128);
  // maps: Q, dO, K, V as 128-row boxes; Q, dO as 64-row boxes.  dK/dV first: its longest blocks
  // (key block 0 sees every query block) set the critical path, so they start before any dQ block.
  cudaError_t e = launch_pdl(attn_bwd_dkdv_kernel<D>, dim3(nb * p.batch * p.ng * p.kv_parts), dim3(GeoKV<D>::THREADS),
                             GeoKV<D>::SMEM, st, maps[2], maps[3], maps[4], maps[5], p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_dq_kernel<D>, dim3(nb * p.batch * p.nh), dim3(GeoQ<D>::THREADS), GeoQ<D>::SMEM, st_dq,
                    maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace

cudaError_t launch_head_slices(const bf16* src, size_t sp, size_t sb, size_t sh, int zdiv, int Z, bf16* dst, size_t dp,
                               int R, int C, cudaStream_t st) {
  if (Z <= 0 || R <= 0 || C <= 0) return cudaSuccess;
  const bool vec = C % 8 == 0 && sp % 8 == 0 && sb % 8 == 0 && sh % 8 == 0 && dp % 8 == 0 &&
                   reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0;
  if (vec)
    head_slices_vec_kernel<<<dim3((C / 8 + 15) / 16, (R + 15) / 16, Z), dim3(16, 16), 0, st>>>(src, sp, sb, sh, zdiv,
                                                                                              dst, dp, R, C / 8);
  else
    head_slices_kernel<<<dim3((C + 31) / 32, (R + 31) / 32, Z), dim3(32, 8), 0, st>>>(src, sp, sb, sh, zdiv, dst, dp, R,
                                                                                     C);
  return cudaGetLastError();
}

cudaError_t launch_row_dot(const bf16* dO, const bf16* O, float* Dsum, int S, int B, int nh, int d, cudaStream_t st) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const size_t threads = static_cast<size_t>(S) * B * nh * (d / 8);
  if (threads == 0) return cudaSuccess;
  row_dot_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(dO, O, Dsum, S, B, nh, d);
  return cudaGetLastError();
}

cudaError_t launch_attention_bwd(int head_dim, const CUtensorMap* maps, const AttnBwdParams& p, cudaStream_t st,
                                 cudaStream_t st_dq) {
  if (p.seq <= 0) return cudaSuccess;
  // every run of steps must be non-empty: the last key block has the fewest, (nh / ng) x (query
  // blocks of 64 from its first on), and part_stride must keep whole rows of D floats
  const int nb = (p.seq + 127) / 128, shortest = (p.nh / p.ng) * ((p.seq + 63) / 64 - 2 * (nb - 1));
  if (p.kv_parts < 1 || p.kv_parts > kMaxKvParts || p.kv_parts > shortest || p.part_stride % head_dim != 0)
    return cudaErrorInvalidValue;
  if (head_dim == 64) return launch_bwd_d<64>(maps, p, st, st_dq);
  if (head_dim == 128) return launch_bwd_d<128>(maps, p, st, st_dq);
  return cudaErrorInvalidValue;
}

}  // namespace mt
