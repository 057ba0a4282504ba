// Dense bf16 GEMM on the 5th-generation tensor cores with fused epilogues:
//   out[M, N] = epilogue( A[M, K] * B[N, K]^T )
// A is a row-major activation (tokens x features) and B a weight stored [out, in], so both
// operands are K-major ("Megatron-LM 深度学习与源码分析文档", Part 2 §2: Y = XW, with the
// column-parallel QKV / fc1 and the row-parallel output projection / fc2 all of this form).
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] per stage, 128-byte swizzle,
//               a 4-stage shared-memory ring guarded by full/empty mbarriers.
//   warp 1      one thread issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM
//               accumulators (2 x 256 fp32 columns) and commits stages / finished tiles.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one output row per
//               thread), fused bias / residual / RoPE / SwiGLU / GeLU, bf16 stores; the second
//               accumulator lets the next tile's main loop run meanwhile.
// Tile order is chosen on the host per GEMM (bands of m- or n-tiles sized so the band's operand stays
// in L2, see GemmParams), and the tiles of the last, partial wave are cut into 2 or 4 narrower
// pieces along N so that the tail wave is shorter (wave quantisation on 152 SMs).
#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB (two 128-row boxes)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
// Epilogue staging for TMA stores: per epilogue warp two [32 rows x 32 columns] bf16 boxes (2 KB each),
// after the 1 KB that holds the barriers.
constexpr int EPI_BOX_BYTES = 32 * 32 * 2;
constexpr int EPI_STAGE_BYTES = 8 * 2 * EPI_BOX_BYTES;
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 1024 + EPI_STAGE_BYTES;

// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ void add_vec32(float* v, const bf16* src, int col, int limit) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (col + 8 * g < limit) {
      float f[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(src + col + 8 * g), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * g + e] += f[e];
    }
  }
}

__device__ __forceinline__ void store_vec32(bf16* dst_row, int col, int limit, const float* v) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    if (col + 8 * g < limit) *reinterpret_cast<uint4*>(dst_row + col + 8 * g) = pack_bf16x8(v + 8 * g);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 0.5 u (1 + tanh(z)), z = sqrt(2/pi) (u + 0.044715 u^3), with 1 + tanh(z) = 2 - 2 / (1 + e^(2z)) formed from
// one base-2 exponential and one reciprocal (both special-function instructions; at |z| -> inf the
// reciprocal goes to 0 or 1 and the result to u or 0)
__device__ __forceinline__ float gelu_tanh(float u) {
  const float k0 = 0.7978845608028654f, k1 = 0.044715f, two_log2e = 2.8853900817779268f;
  const float z = k0 * (u + k1 * u * u * u);
  return u * (1.0f - rcp_approx(1.0f + ex2_approx(z * two_log2e)));
}

// silu(g) = g sigmoid(g), sigmoid(g) = 1 / (1 + e^-g): one base-2 exponential and one reciprocal
__device__ __forceinline__ float silu(float g) { return g * rcp_approx(1.0f + ex2_approx(-g * 1.4426950408889634f)); }

// One work unit: tile (tm, tn) of the raster, piece `sub` of `split` along N.
struct Unit {
  int tm, tn, sub, split;
  int kpart, ks, tail;  // K range kpart of ks (ks = 1: all of K); tail: the tile's index in the tail wave
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u) {
  Unit w;
  int tile;
  w.kpart = 0;
  w.ks = 1;
  w.tail = 0;
  if (u < p.full_units) {
    tile = u;
    w.sub = 0;
    w.split = 1;
  } else if (p.ksplit > 1) {
    const int v = u - p.full_units;
    w.tail = v / p.ksplit;
    tile = p.full_units + w.tail;
    w.sub = 0;
    w.split = 1;
    w.kpart = v - w.tail * p.ksplit;
    w.ks = p.ksplit;
  } else {
    const int v = u - p.full_units;
    tile = p.full_units + v / p.split;
    w.sub = v % p.split;
    w.split = p.split;
  }
  if (p.band_m) {
    const int per_band = p.band * p.tiles_n;
    const int bi = tile / per_band, r = tile - bi * per_band;
    const int gm = min(p.band, p.tiles_m - bi * p.band);
    w.tm = bi * p.band + r % gm;
    w.tn = r / gm;
  } else {
    const int per_band = p.band * p.tiles_m;
    const int bi = tile / per_band, r = tile - bi * per_band;
    const int gn = min(p.band, p.tiles_n - bi * p.band);
    w.tn = bi * p.band + r % gn;
    w.tm = r / gn;
  }
  return w;
}

// Output columns of a unit: [c0, c0 + width).  SwiGLU tiles cover 128 outputs (256 accumulator
// columns: gate then up); the others 256.
template <int MODE>
__device__ __forceinline__ int unit_width(const Unit& w) {
  return (MODE == kEpiSwiglu ? 128 : BN) / w.split;
}
template <int MODE>
__device__ __forceinline__ int unit_col0(const Unit& w) {
  return w.tn * (MODE == kEpiSwiglu ? 128 : BN) + w.sub * unit_width<MODE>(w);
}

// K blocks [unit_kb0, unit_kb1) of a unit: all of them, or K range kpart of ks (balanced).
__device__ __forceinline__ int unit_kb0(const Unit& w, int num_kb) { return w.kpart * num_kb / w.ks; }
__device__ __forceinline__ int unit_kb1(const Unit& w, int num_kb) { return (w.kpart + 1) * num_kb / w.ks; }

// K-split partial sums of one epilogue warp (its 32 rows of one CTA): one slot per K range after
// the first, 8 chunks of 32 accumulator columns each, a chunk stored as [8][lane 32] float4 so
// that a warp's store or load of 512 B is contiguous.
constexpr int kKsWarpF4 = 8 * 256;           // float4 per warp and slot
constexpr int kKsSlotF4 = 2 * 4 * kKsWarpF4;  // float4 per slot (two CTAs, four quadrants)

__device__ __forceinline__ int ld_acquire_gpu(const int* a) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int* a, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__device__ __forceinline__ void scale32(float* v, float f) {
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] *= f;
}

// 32 outputs as E4M3 codes (pitch in bytes), masked per 8 columns.
__device__ __forceinline__ void store_e4m3x32(uint8_t* dst_row, int col, int limit, const float* v, float qs) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    if (col + 8 * g < limit) *reinterpret_cast<uint2*>(dst_row + col + 8 * g) = pack_e4m3x8(v + 8 * g, qs);
}

// Eight bf16 values at src[col + 8g], g < 4, as 16-byte vectors; zeros past `limit` (or for a row
// outside the output).
__device__ __forceinline__ void load_vec32(const bf16* src, int col, int limit, bool valid, uint4 (&o)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    o[g] = (valid && col + 8 * g < limit) ? *reinterpret_cast<const uint4*>(src + col + 8 * g) : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void add_loaded32(float* v, const uint4 (&a)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float f[8];
    unpack_bf16x8(a[g], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[8 * g + e] += f[e];
  }
}

// Epilogue of the bf16-output modes (store, residual, GeLU) as a two-deep software pipeline over
// the warp's 32-column chunks: the TMEM load of chunk i + 1 and the global load of its residual
// row segment are in flight while chunk i is formed and stored, so one chunk's latency (TMEM, then
// L2) is not paid again for every chunk.  SwiGLU, whose chunk holds twice the accumulator columns,
// starts the next chunk's TMEM loads once the current chunk is packed to bf16, before its stores.
// Same arithmetic, in the same order, as the one-chunk-at-a-time form.
// The chunk's 32 bf16 outputs of this thread's row, through the warp's staging box and one TMA
// store per chunk (p.tma_out), or as four 16-byte stores.  Box row `lane` holds the thread's 64 bytes,
// its 16-byte piece c at position c ^ ((lane >> 1) & 3) (the 64-byte swizzle of the output tensor
// map, which also keeps the warp's shared-memory stores free of bank conflicts).  The staging box
// alternates between two buffers; a buffer is rewritten once the store issued two chunks earlier has
// read it.
struct EpiStore {
  const CUtensorMap* map;
  uint8_t* stage;  // this warp's two boxes
  int y0;          // output row of box row 0
  int n;           // chunks stored so far
  // residual epilogue: the residual box of a chunk is loaded by TMA into the box the chunk's output
  // will be staged in (rmap: the residual [M, N] in the same 32 x 32 boxes; rbar: this warp's two
  // mbarriers, one per box)
  const CUtensorMap* rmap;
  uint32_t rbar;
  int* err;
};

// Residual box of the warp's `g`-th chunk (box g & 1) at output column `col`: once every store of
// this warp has finished reading its boxes (the box's previous output), one TMA load completing on
// the box's mbarrier.
__device__ __forceinline__ void resid_box_load(EpiStore& es, int g, int col) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    if (es.n > 0) cp_bulk_wait_read<0>();
    const uint32_t bar = es.rbar + 8u * (g & 1);
    mbar_arrive_expect_tx(bar, EPI_BOX_BYTES);
    tma_load_2d(smem_u32(es.stage + (g & 1) * EPI_BOX_BYTES), es.rmap, bar, col, es.y0);
  }
  __syncwarp();
}

// p.c_trans: the tile is stored transposed, element (row, col) at out[col * ldo + row] (the output
// tensor map then spans [N rows][M columns]); box row e holds output row col + e, whose 32 elements
// are the warp's 32 rows, one 2-byte store per lane and e (a warp covers a whole 64-byte box row,
// free of bank conflicts).
__device__ __forceinline__ void store_chunk(const GemmParams& p, EpiStore& es, bf16* out_row, int col, bool valid,
                                            const float* v) {
  const int lane = threadIdx.x & 31;
  if (!p.tma_out) {
    if (!valid) return;
    if (p.c_trans) {
      bf16* dst = p.out + es.y0 + lane;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (col + e < p.N) dst[static_cast<size_t>(col + e) * p.ldo] = __float2bfloat16_rn(v[e]);
    } else {
      store_vec32(out_row, col, p.N, v);
    }
    return;
  }
  uint8_t* box = es.stage + (es.n & 1) * EPI_BOX_BYTES;
  if (es.n >= 2) {
    if (lane == 0) cp_bulk_wait_read<1>();
    __syncwarp();
  }
  if (p.c_trans) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      *reinterpret_cast<bf16*>(box + e * 64 + ((((lane >> 3) ^ (e >> 1)) & 3) << 4) + (lane & 7) * 2) =
          __float2bfloat16_rn(v[e]);
  } else {
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(box + lane * 64 + ((c ^ sw) << 4)) = pack_bf16x8(v + 8 * c);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (p.c_trans) tma_store_2d(es.map, smem_u32(box), es.y0, col);
    else tma_store_2d(es.map, smem_u32(box), col, es.y0);
    cp_bulk_commit();
  }
  ++es.n;
}

// 32 values of this thread's row (8-element groups packed by `pack`) through the warp's next staging
// box, stored with one TMA store at (x, y, z) of the 3-D output map (the QKV epilogue's q, k, v heads).
template <typename Pack>
__device__ __forceinline__ void store_box3(EpiStore& es, const float* v, int x, int y, int z, Pack pack) {
  const int lane = threadIdx.x & 31;
  uint8_t* box = es.stage + (es.n & 1) * EPI_BOX_BYTES;
  if (es.n >= 2) {
    if (lane == 0) cp_bulk_wait_read<1>();
    __syncwarp();
  }
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(box + lane * 64 + ((c ^ sw) << 4)) = pack(v + 8 * c);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(es.map, smem_u32(box), x, y, z);
    cp_bulk_commit();
  }
  ++es.n;
}

template <int MODE, bool F8>
__device__ __forceinline__ void epilogue_tile_bf16(const GemmParams& p, uint32_t tacc, int m0, int c0, int width,
                                                   int r_in_tile, int lo, int hi, EpiStore& es) {
  const int row = m0 + r_in_tile;
  const bool valid = row < p.M;
  const float deq = F8 ? __ldg(p.deq_a) * __ldg(p.deq_b) : 1.f;
  const int end = min(hi, p.N - c0);
  const int n = end > lo ? (end - lo + 31) / 32 : 0;
  if (n == 0) return;
  bf16* out_row = p.out + static_cast<size_t>(row) * p.ldo;
  es.y0 = row - (threadIdx.x & 31);
  if constexpr (MODE == kEpiSwiglu) {
    uint32_t g[32], u[32];
    tmem_ld32_issue(tacc + lo, g);
    tmem_ld32_issue(tacc + width + lo, u);  // the up half follows the `width` gate columns
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
      const int col = c0 + lo + 32 * i;
      tmem_ld32_wait(g);
      tmem_ld32_wait(u);
      float v[32], w[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        v[e] = __uint_as_float(g[e]);
        w[e] = __uint_as_float(u[e]);
      }
      if (i + 1 < n) {
        tmem_ld32_issue(tacc + lo + 32 * (i + 1), g);
        tmem_ld32_issue(tacc + width + lo + 32 * (i + 1), u);
      }
      if (F8) {
        scale32(v, deq);
        scale32(w, deq);
      }
      if (valid) {
        if (p.bias != nullptr) {
          add_vec32(v, p.bias, col, p.N);
          add_vec32(w, p.bias + p.N, col, p.N);
        }
        if (p.pre != nullptr) {
          bf16* pre_row = p.pre + static_cast<size_t>(row) * p.ldp;
          store_vec32(pre_row, col, p.N, v);
          store_vec32(pre_row + p.N, col, p.N, w);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = silu(v[e]) * w[e];
      }
      store_chunk(p, es, out_row, col, valid, v);
    }
  } else {
    if constexpr (MODE == kEpiResid) {
      if (p.tma_out) {  // residual boxes by TMA into the staging boxes, one chunk ahead
        const int lane = threadIdx.x & 31, sw = (lane >> 1) & 3;
        uint32_t g32[32];
        tmem_ld32_issue(tacc + lo, g32);
        resid_box_load(es, es.n, c0 + lo);
#pragma unroll 1
        for (int i = 0; i < n; ++i) {
          const int col = c0 + lo + 32 * i, g = es.n;
          tmem_ld32_wait(g32);
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(g32[e]);
          if (i + 1 < n) {
            tmem_ld32_issue(tacc + lo + 32 * (i + 1), g32);
            resid_box_load(es, g + 1, col + 32);
          }
          const bool got = mbar_wait(es.rbar + 8u * (g & 1), (g >> 1) & 1, es.err, nullptr);
          if (!__all_sync(0xffffffffu, got)) {  // recorded in the error word; let the next box's load land
            if (i + 1 < n && lane == 0)
              mbar_wait_slow(es.rbar + 8u * ((g + 1) & 1), ((g + 1) >> 1) & 1, nullptr, nullptr, kDrainLimitNs);
            return;
          }
          uint8_t* box = es.stage + (g & 1) * EPI_BOX_BYTES + lane * 64;
          if (valid) {
            if (F8) scale32(v, deq);
            if (p.bias != nullptr) add_vec32(v, p.bias, col, p.N);
            uint4 rr[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) rr[c] = *reinterpret_cast<const uint4*>(box + ((c ^ sw) << 4));
            add_loaded32(v, rr);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(box + ((c ^ sw) << 4)) = pack_bf16x8(v + 8 * c);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(es.map, smem_u32(box - lane * 64), col, es.y0);
            cp_bulk_commit();
          }
          ++es.n;
        }
        return;
      }
    }
    const bf16* resid = MODE == kEpiResid ? p.resid + static_cast<size_t>(row) * p.ldr : nullptr;
    uint32_t ga[32], gb[32];
    uint4 ra[4], rb[4];
    auto issue = [&](int i, uint32_t (&r32)[32], uint4 (&res)[4]) {
      const int c = lo + 32 * i;
      tmem_ld32_issue(tacc + c, r32);
      if (MODE == kEpiResid) load_vec32(resid, c0 + c, p.N, valid, res);
    };
    auto finish = [&](int i, const uint32_t (&r32)[32], const uint4 (&res)[4]) {
      const int col = c0 + lo + 32 * i;
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r32[e]);
      if (valid) {
        if (F8) scale32(v, deq);
        if (p.bias != nullptr) add_vec32(v, p.bias, col, p.N);
        if (MODE == kEpiResid) add_loaded32(v, res);
        if (MODE == kEpiGelu) {
          if (p.pre != nullptr) store_vec32(p.pre + static_cast<size_t>(row) * p.ldp, col, p.N, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = gelu_tanh(v[e]);
        }
      }
      store_chunk(p, es, out_row, col, valid, v);
    };
    issue(0, ga, ra);
#pragma unroll 1
    for (int i = 0; i < n; i += 2) {
      tmem_ld32_wait(ga);
      if (i + 1 < n) issue(i + 1, gb, rb);
      finish(i, ga, ra);
      if (i + 1 < n) {
        tmem_ld32_wait(gb);
        if (i + 2 < n) issue(i + 2, ga, ra);
        finish(i + 1, gb, rb);
      }
    }
  }
}

template <int MODE, bool F8>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tacc, int m0, int c0, int width,
                                              int r_in_tile, int lo, int hi, EpiStore& es) {
  if constexpr (MODE == kEpiStore || MODE == kEpiResid || MODE == kEpiGelu || MODE == kEpiSwiglu) {
    if (p.out8 == nullptr && (MODE != kEpiStore || p.out32 == nullptr)) {
      epilogue_tile_bf16<MODE, F8>(p, tacc, m0, c0, width, r_in_tile, lo, hi, es);
      return;
    }
  }
  const int row = m0 + r_in_tile;
  const bool valid = row < p.M;
  const float deq = F8 ? __ldg(p.deq_a) * __ldg(p.deq_b) : 1.f;
  const bool out8 = (MODE == kEpiSwiglu || MODE == kEpiGelu) && p.out8 != nullptr;
  const float qs = out8 ? __ldg(p.q_scale) : 1.f;
  float amax = 0.f;
  if constexpr (MODE == kEpiStore || MODE == kEpiResid || MODE == kEpiGelu) {
#pragma unroll 1
    for (int c = lo; c < hi; c += 32) {
      const int col = c0 + c;
      if (col >= p.N) break;  // uniform across the warp
      float v[32];
      tmem_ld32(tacc + c, v);
      if (valid) {
        if (F8) scale32(v, deq);
        if (p.bias != nullptr) add_vec32(v, p.bias, col, p.N);
        if constexpr (MODE == kEpiResid) add_vec32(v, p.resid + static_cast<size_t>(row) * p.ldr, col, p.N);
        if constexpr (MODE == kEpiGelu) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = gelu_tanh(v[e]);
        }
        if (out8) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (col + e < p.N) amax = fmaxf(amax, fabsf(v[e]));
          store_e4m3x32(p.out8 + static_cast<size_t>(row) * p.ldo, col, p.N, v, qs);
        } else if (MODE == kEpiStore && p.out32 != nullptr) {
          float* dst = p.out32 + static_cast<size_t>(row) * p.ldo + col;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if (col + 4 * g < p.N) {
              float4 o = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
              if (p.acc32) {
                const float4 prev = reinterpret_cast<const float4*>(dst)[g];
                o.x += prev.x;
                o.y += prev.y;
                o.z += prev.z;
                o.w += prev.w;
              }
              reinterpret_cast<float4*>(dst)[g] = o;
            }
          }
        } else {
          store_vec32(p.out + static_cast<size_t>(row) * p.ldo, col, p.N, v);
        }
      }
    }
  } else if constexpr (MODE == kEpiSwiglu) {
#pragma unroll 1
    for (int c = lo; c < hi; c += 32) {
      const int col = c0 + c;
      if (col >= p.N) break;
      float g[32], u[32];
      tmem_ld32(tacc + c, g);
      tmem_ld32(tacc + width + c, u);  // the up half follows the `width` gate columns
      if (valid) {
        if (F8) {
          scale32(g, deq);
          scale32(u, deq);
        }
        if (p.bias != nullptr) {
          add_vec32(g, p.bias, col, p.N);
          add_vec32(u, p.bias + p.N, col, p.N);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) g[e] = silu(g[e]) * u[e];
        if (out8) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (col + e < p.N) amax = fmaxf(amax, fabsf(g[e]));
          store_e4m3x32(p.out8 + static_cast<size_t>(row) * p.ldo, col, p.N, g, qs);
        } else {
          store_vec32(p.out + static_cast<size_t>(row) * p.ldo, col, p.N, g);
        }
      }
    }
  } else if (p.tma_out) {
    // kEpiQkv, batch 1: q, k and v are one [heads q | k | v][token][d] tensor, so the head of column
    // `col` is col / d; each 32-column piece of a head goes out as one TMA store of 32 tokens
    const int d = p.head_dim, half = d >> 1;
    const int lane = threadIdx.x & 31;
    const int y0 = row - lane + p.row0;  // token row of box row 0
    const int rpos = (valid && p.pos != nullptr) ? p.pos[row + p.row0] : row + p.row0;  // RoPE position
    auto bf16x8 = [](const float* f) { return pack_bf16x8(f); };
    auto f16x8 = [](const float* f) { return pack_f16x8(f); };
#pragma unroll 1
    for (int hc = lo; hc < hi; hc += d) {
      const int col = c0 + hc;
      if (col >= p.N) break;
      const int hz = col / d;
      if (col < p.q_w + p.kv_w && p.rope != nullptr) {
        // rotate-half: (x_i, x_{i+d/2}) -> (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s)
#pragma unroll 1
        for (int i0 = 0; i0 < half; i0 += 32) {
          float x1[32], x2[32];
          tmem_ld32(tacc + hc + i0, x1);
          tmem_ld32(tacc + hc + half + i0, x2);
          if (valid) {
            if (F8) {
              scale32(x1, deq);
              scale32(x2, deq);
            }
            if (p.bias != nullptr) {
              add_vec32(x1, p.bias, col + i0, p.N);
              add_vec32(x2, p.bias, col + half + i0, p.N);
            }
            const float4* cs = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(rpos) * half + i0);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float4 t = cs[e];  // (cos, sin) of elements 2e and 2e+1
              const float a0 = x1[2 * e], b0 = x2[2 * e], a1 = x1[2 * e + 1], b1 = x2[2 * e + 1];
              x1[2 * e] = a0 * t.x - b0 * t.y;
              x2[2 * e] = b0 * t.x + a0 * t.y;
              x1[2 * e + 1] = a1 * t.z - b1 * t.w;
              x2[2 * e + 1] = b1 * t.z + a1 * t.w;
            }
          }
          store_box3(es, x1, i0, y0, hz, bf16x8);
          store_box3(es, x2, half + i0, y0, hz, bf16x8);
        }
      } else {
        const bool is_v = col >= p.q_w + p.kv_w;
#pragma unroll 1
        for (int i0 = 0; i0 < d; i0 += 32) {
          float x[32];
          tmem_ld32(tacc + hc + i0, x);
          if (valid) {
            if (F8) scale32(x, deq);
            if (p.bias != nullptr) add_vec32(x, p.bias, col + i0, p.N);
          }
          if (is_v)
            store_box3(es, x, i0, y0, hz, f16x8);
          else
            store_box3(es, x, i0, y0, hz, bf16x8);
        }
      }
    }
  } else {  // kEpiQkv: `width` is a multiple of head_dim, so every head lies inside one unit
    const int d = p.head_dim, half = d >> 1;
    const int trow = row + p.row0;               // token row
    const int s = valid ? trow / p.batch : 0;  // row of the [b, head, s, d] buffers
    const int b = valid ? trow - s * p.batch : 0;
    const int rpos = (valid && p.pos != nullptr) ? p.pos[trow] : s;    // RoPE position
#pragma unroll 1
    for (int hc = lo; hc < hi; hc += d) {
      const int col = c0 + hc;
      if (col >= p.N) break;
      bf16* dst = nullptr;
      __half* vdst = nullptr;
      if (col < p.q_w) {
        const int hh = col / d;
        dst = p.q + ((static_cast<size_t>(b) * p.nh + hh) * p.seq + s) * d;
      } else if (col < p.q_w + p.kv_w) {
        const int gg = (col - p.q_w) / d;
        dst = p.k + ((static_cast<size_t>(b) * p.ng + gg) * p.seq + s) * d;
      } else {
        const int gg = (col - p.q_w - p.kv_w) / d;
        vdst = p.v + ((static_cast<size_t>(b) * p.ng + gg) * p.seq + s) * d;
      }
      if (vdst == nullptr && p.rope != nullptr) {
        // rotate-half: (x_i, x_{i+d/2}) -> (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s)
#pragma unroll 1
        for (int i0 = 0; i0 < half; i0 += 32) {
          float x1[32], x2[32];
          tmem_ld32(tacc + hc + i0, x1);
          tmem_ld32(tacc + hc + half + i0, x2);
          if (valid) {
            if (F8) {
              scale32(x1, deq);
              scale32(x2, deq);
            }
            if (p.bias != nullptr) {
              add_vec32(x1, p.bias, col + i0, p.N);
              add_vec32(x2, p.bias, col + half + i0, p.N);
            }
            const float4* cs = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(rpos) * half + i0);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float4 t = cs[e];  // (cos, sin) of elements 2e and 2e+1
              const float a0 = x1[2 * e], b0 = x2[2 * e], a1 = x1[2 * e + 1], b1 = x2[2 * e + 1];
              x1[2 * e] = a0 * t.x - b0 * t.y;
              x2[2 * e] = b0 * t.x + a0 * t.y;
              x1[2 * e + 1] = a1 * t.z - b1 * t.w;
              x2[2 * e + 1] = b1 * t.z + a1 * t.w;
            }
            store_vec32(dst, i0, d, x1);
            store_vec32(dst, half + i0, d, x2);
          }
        }
      } else {
#pragma unroll 1
        for (int i0 = 0; i0 < d; i0 += 32) {
          float x[32];
          tmem_ld32(tacc + hc + i0, x);
          if (valid) {
            if (F8) scale32(x, deq);
            if (p.bias != nullptr) add_vec32(x, p.bias, col + i0, p.N);
            if (vdst != nullptr) {
#pragma unroll
              for (int g8 = 0; g8 < 4; ++g8) *reinterpret_cast<uint4*>(vdst + i0 + 8 * g8) = pack_f16x8(x + 8 * g8);
            } else {
              store_vec32(dst, i0, d, x);
            }
          }
        }
      }
    }
  }
  if (out8) {  // every lane arrives here (the loops above break uniformly)
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) atomic_max_abs(p.amax, amax);
  }
}

// Epilogue warps: two per TMEM lane quadrant.  With p.epi_split == 2 both store part of a unit's
// `width` columns (part 0 the first half, rounded down to 32 columns, QKV: to whole heads; part 1
// the rest; a unit too narrow to split goes to part 0 alone); with 1 the first warp of each quadrant
// stores all of them and the second stays idle.
constexpr int EPI_WARPS = 8;
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;  // TMA warp, MMA warp, epilogue warps
template <int MODE>
__device__ __forceinline__ void epilogue_part(const GemmParams& p, int width, int part, int& lo, int& hi) {
  const int gran = MODE == kEpiQkv ? p.head_dim : 32;
  const int mid = p.epi_split == 2 ? (width / 2) / gran * gran : 0;
  lo = part == 0 ? 0 : (mid == 0 ? width : mid);
  hi = part == 0 ? (mid == 0 ? width : mid) : width;
}

// ------------------------------------------------------------------ kernel
template <int MODE, bool F8>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmO,
                const __grid_constant__ CUtensorMap tmR, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + STAGES * STAGE_BYTES);
  // bars: full[STAGES] | empty[STAGES] | tmem_full[2] | tmem_empty[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 4 * p.epi_split);  // the active epilogue warps
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 2 * EPI_WARPS; ++i) mbar_init(bar0 + 256u + 8u * i, 1);  // residual boxes
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    tma_prefetch(&tmB64);
    if (p.tma_out) tma_prefetch(&tmO);
    if (p.tma_out && MODE == kEpiResid) tma_prefetch(&tmR);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the setup above overlaps the end of the previous kernel
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  constexpr int KB = F8 ? 128 : BK;  // K elements per stage: one 128-byte swizzle row either way
  const int num_kb = (p.K + KB - 1) / KB;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = decode_unit(p, u);
        const int m0 = w.tm * BM;
        const int width = unit_width<MODE>(w);
        const int c0 = unit_col0<MODE>(w);
        // B rows of this unit: SwiGLU gate rows [c0, c0+width) then the matching up rows;
        // otherwise rows [c0, c0+width).  Boxes of 128 rows, or 64 for the narrowest pieces.
        const int b_rows = MODE == kEpiSwiglu ? 2 * width : width;
        const uint32_t stage_bytes = A_BYTES + b_rows * 128;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full(stage);
          mbar_arrive_expect_tx(fb, stage_bytes);
          const uint32_t a_dst = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
          if (!F8 && p.a_mn) {  // A stored [K, M]: two [64 K x 64 M] blocks
            tma_load_2d(a_dst, &tmA, fb, m0, kb * KB);
            tma_load_2d(a_dst + 8192, &tmA, fb, m0 + 64, kb * KB);
          } else {
            tma_load_2d(a_dst, &tmA, fb, kb * KB, m0);
          }
          if (!F8 && MODE == kEpiStore && p.b_mn) {  // B stored [K, N]: width / 64 blocks of [64 K x 64 N]
            for (int a = 0; a < width / 64; ++a) tma_load_2d(b_dst + a * 8192, &tmB, fb, c0 + 64 * a, kb * KB);
          } else if (MODE == kEpiSwiglu) {
            const CUtensorMap* mb = width == 128 ? &tmB : &tmB64;
            tma_load_2d(b_dst, mb, fb, kb * KB, c0);
            tma_load_2d(b_dst + width * 128, mb, fb, kb * KB, c0 + p.b_row_step);
          } else if (width == 256) {
            tma_load_2d(b_dst, &tmB, fb, kb * KB, c0);
            tma_load_2d(b_dst + B_BYTES / 2, &tmB, fb, kb * KB, c0 + 128);
          } else {
            tma_load_2d(b_dst, width == 128 ? &tmB : &tmB64, fb, kb * KB, c0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let this CTA's own copies in flight land before its shared memory goes away
        for (int s = 0; s < STAGES; ++s)
          if (s < stage || issued >= STAGES)
            mbar_wait_slow(full(s), s < stage ? phase : (phase ^ 1u), nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
        const Unit w = decode_unit(p, u);
        const int width = unit_width<MODE>(w);
        const int n_mma = MODE == kEpiSwiglu ? 2 * width : width;
        const uint32_t idesc = F8 ? idesc_e4m3(BM, n_mma)
                                  : (idesc_bf16(BM, n_mma) | (p.a_mn ? 1u << 15 : 0u) | (p.b_mn ? 1u << 16 : 0u));
        const int acc = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(tempty(acc), use ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full(stage), phase, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K-major tiles advance 32 B per 16-deep K step, MN-major tiles 2048 B (16 K rows)
          const uint32_t a_s = smem_u32(sA + stage * A_BYTES), b_s = smem_u32(sB + stage * B_BYTES);
          const uint64_t ad = (!F8 && p.a_mn) ? sw128_desc_mn(a_s, 8192) : sw128_desc(a_s);
          const uint64_t bd = (!F8 && p.b_mn) ? sw128_desc_mn(b_s, 8192) : sw128_desc(b_s);
          const uint64_t astep = (!F8 && p.a_mn) ? 128ull : 2ull, bstep = (!F8 && p.b_mn) ? 128ull : 2ull;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            if (F8)
              mma_e4m3_ss(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb | k) != 0 ? 1u : 0u);
            else
              mma_bf16_ss(d_tmem, ad + astep * k, bd + bstep * k, idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit(empty(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(tfull(acc));
      }
      // No MMA may still read shared memory or write TMEM when the CTA releases them.
      mma_commit(drain);
      mbar_wait_slow(drain, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes this warp may read
    const int part = (warp - 2) >> 2;
    EpiStore es{&tmO, base + STAGES * STAGE_BYTES + 1024 + (warp - 2) * 2 * EPI_BOX_BYTES, 0, 0, &tmR,
                bar0 + 256u + 16u * (warp - 2), p.err};
    int it = 0;
    for (int u = blockIdx.x; part < p.epi_split && u < p.num_units; u += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = (it >> 1) & 1;
      const bool ok = mbar_wait(tfull(acc), use, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const Unit w = decode_unit(p, u);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      int lo, hi;
      epilogue_part<MODE>(p, unit_width<MODE>(w), part, lo, hi);
      if (lo < hi)
        epilogue_tile<MODE, F8>(p, tacc, w.tm * BM, unit_col0<MODE>(w), unit_width<MODE>(w), quad * 32 + lane, lo, hi,
                                es);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
    }
    if (es.n > 0 && lane == 0) cp_bulk_wait_all();  // this warp's output stores are complete
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Accumulator columns an epilogue part reads: 32-column chunks c of [lo, hi) with c0 + c < N
// (SwiGLU: each also the up chunk `width` columns later).  Returns the count; col(i) the i-th.
template <int MODE>
struct PartCols {
  int lo, width, n_gate;
  __device__ __forceinline__ PartCols(const GemmParams& p, int c0, int width_, int lo_, int hi) : lo(lo_), width(width_) {
    const int end = min(hi, p.N - c0);
    n_gate = end > lo ? (end - lo + 31) / 32 : 0;
  }
  __device__ __forceinline__ int count() const { return MODE == kEpiSwiglu ? 2 * n_gate : n_gate; }
  __device__ __forceinline__ int col(int i) const {
    return MODE == kEpiSwiglu && i >= n_gate ? width + lo + 32 * (i - n_gate) : lo + 32 * i;
  }
};

// K-split tail, a unit with kpart > 0: this warp's columns of the partial sum (the columns its
// epilogue part would store) go to slot kpart - 1, then one arrival on the tile's counter.
template <int MODE>
__device__ __forceinline__ void kpart_store(const GemmParams& p, const Unit& w, uint32_t tacc, int c0, int width,
                                            int rank, int quad, int part, int lo, int hi) {
  const int lane = threadIdx.x & 31;
  float4* dst = p.kws + (static_cast<size_t>(w.tail * (w.ks - 1) + w.kpart - 1) * 8 + rank * 4 + quad) * kKsWarpF4 + lane;
  const PartCols<MODE> pc(p, c0, width, lo, hi);
#pragma unroll 1
  for (int i = 0; i < pc.count(); ++i) {
    const int col = pc.col(i);
    float v[32];
    tmem_ld32(tacc + col, v);
#pragma unroll
    for (int g = 0; g < 8; ++g)
      __stcg(dst + (col >> 5) * 256 + 32 * g, make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) red_release_gpu_add(p.kflags + ((w.tail * 2 + rank) * 4 + quad) * 2 + part, 1);
}

// Adds NP (1 or 2) partial slots to this warp's accumulator columns, one 32-column chunk at a
// time with the chunk's loads of both slots issued before the first add (the partials come from
// L2, and their latency, not their bytes, paces the fold).
template <int MODE, int NP>
__device__ __forceinline__ void fold_chunks(const float4* base, uint32_t tacc, const PartCols<MODE>& pc) {
#pragma unroll 1
  for (int i = 0; i < pc.count(); ++i) {
    const int col = pc.col(i);
    const float4* src = base + (col >> 5) * 256;
    float4 t[NP][8];
#pragma unroll
    for (int q = 0; q < NP; ++q)
#pragma unroll
      for (int g = 0; g < 8; ++g) t[q][g] = __ldcg(src + static_cast<size_t>(q) * kKsSlotF4 + 32 * g);
    float v[32];
    tmem_ld32(tacc + col, v);
#pragma unroll
    for (int q = 0; q < NP; ++q)
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        v[4 * g] += t[q][g].x;
        v[4 * g + 1] += t[q][g].y;
        v[4 * g + 2] += t[q][g].z;
        v[4 * g + 3] += t[q][g].w;
      }
    tmem_st32(tacc + col, v);
  }
}

// K-split tail, the unit with kpart 0: waits (bounded) until the other ks - 1 units have stored
// this warp's partials and adds them, in K order, to its accumulator columns in TMEM; on timeout
// sets the error word and leaves the accumulator as it is.
template <int MODE>
__device__ __forceinline__ void kpart_fold(const GemmParams& p, const Unit& w, uint32_t tacc, int c0, int width,
                                           int rank, int quad, int part, int lo, int hi) {
  const int lane = threadIdx.x & 31;
  const int* flag = p.kflags + ((w.tail * 2 + rank) * 4 + quad) * 2 + part;
  bool ok = ld_acquire_gpu(flag) >= w.ks - 1;
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (!(ok = ld_acquire_gpu(flag) >= w.ks - 1)) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(p.err, 0, kErrTimeout);
        break;
      }
    }
  }
  if (!__all_sync(0xffffffffu, ok)) return;
  const float4* base = p.kws + (static_cast<size_t>(w.tail * (w.ks - 1)) * 8 + rank * 4 + quad) * kKsWarpF4 + lane;
  const PartCols<MODE> pc(p, c0, width, lo, hi);
  // the partials are added to the fp32 accumulator in K order: ((acc + part 1) + part 2) + part 3
  if (w.ks == 2) {
    fold_chunks<MODE, 1>(base, tacc, pc);
  } else {
    fold_chunks<MODE, 2>(base, tacc, pc);
    if (w.ks == 4) fold_chunks<MODE, 1>(base + 2 * kKsSlotF4, tacc, pc);
  }
}

// Residual epilogue: the row segment this warp's lane will add, pulled into L2 while the unit's
// main loop still runs (the residual is typically cold in DRAM; its latency, one chunk at a time,
// otherwise paces the epilogue of short-K GEMMs).
template <int MODE>
__device__ __forceinline__ void prefetch_resid(const GemmParams& p, const Unit& w, int m0, int part, int r_in_tile) {
  if constexpr (MODE == kEpiResid) {
    const int width = unit_width<MODE>(w), c0 = unit_col0<MODE>(w);
    int lo, hi;
    epilogue_part<MODE>(p, width, part, lo, hi);
    const int row = m0 + r_in_tile, end = min(hi, p.N - c0);
    if (row >= p.M || end <= lo) return;
    const char* src = reinterpret_cast<const char*>(p.resid + static_cast<size_t>(row) * p.ldr + c0 + lo);
    for (int off = 0; off < (end - lo) * 2; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + off));
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
// The same GEMM with 256 x 256 tiles on a cluster of two CTAs (cta_group::2).  Each CTA stages
// its own 128 rows of A and half of the tile's B rows (N / 2; for SwiGLU the even CTA holds the
// gate rows and the odd one the up rows), so a CTA moves 32 KB per K block instead of 48 KB and
// fits P_STAGES stages.  The even CTA's thread issues the M = 256 MMAs, which write each CTA's
// 128 accumulator rows into that CTA's tensor memory; its commits arrive on the barriers of both
// CTAs.  Both CTAs' TMA copies complete on the even CTA's `full` barriers, and both CTAs'
// active epilogue warps release an accumulator on the even CTA's `tempty` barrier (count 8 * epi_split).
constexpr int P_STAGES = 6;
constexpr int P_B_BYTES = 128 * BK * 2;  // up to 128 B rows per CTA
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES;
constexpr size_t P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + 1024 + EPI_STAGE_BYTES;
static_assert(SMEM_BYTES <= 232448 && P_SMEM_BYTES <= 232448, "GEMM tiles exceed the shared memory of a CTA");

template <int MODE, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmR, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + P_STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + P_STAGES * P_STAGE_BYTES);
  // bars: full[P_STAGES] | empty[P_STAGES] | tmem_full[2] | tmem_empty[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (P_STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * P_STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * P_STAGES + 2 + a); };
  const uint32_t drain = bar0 + 8u * (2 * P_STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 8 * p.epi_split);  // both CTAs' active epilogue warps
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 2 * EPI_WARPS; ++i) mbar_init(bar0 + 256u + 8u * i, 1);  // residual boxes
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    tma_prefetch(&tmB64);
    if (p.tma_out) tma_prefetch(&tmO);
    if (p.tma_out && MODE == kEpiResid) tma_prefetch(&tmR);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised and the tensor memory is allocated before either uses them
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  // the setup above overlaps the end of the previous kernel; the producer waits for it only after
  // issuing the weight loads that do not depend on it
  if (warp != 0) pdl_wait();
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  constexpr int KB = F8 ? 128 : BK;
  const int num_kb = (p.K + KB - 1) / KB;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      // B (a weight) of the first unit's first stages, before the wait for the previous kernel
      int pre = 0;
      if (p.b_static && pair < p.num_units && !(!F8 && MODE == kEpiStore && p.b_mn)) {
        const Unit w = decode_unit(p, pair);
        const int width = unit_width<MODE>(w);
        const int c0 = unit_col0<MODE>(w);
        const int b_rows = MODE == kEpiSwiglu ? width : width / 2;
        const int b_row0 = MODE == kEpiSwiglu ? c0 + (rank ? p.b_row_step : 0) : c0 + static_cast<int>(rank) * b_rows;
        const CUtensorMap* mb = b_rows == 128 ? &tmB : &tmB64;
        const uint32_t pair_bytes = 2u * (A_BYTES + b_rows * 128);
        const int kb0 = unit_kb0(w, num_kb);
        pre = min(P_STAGES, unit_kb1(w, num_kb) - kb0);
        for (int s = 0; s < pre; ++s) {  // fresh stages: nothing to wait for
          const uint32_t fb = map_to_rank(full(s), 0);
          if (leader) mbar_arrive_expect_tx(full(s), pair_bytes);
          tma_load_2d_pair(smem_u32(sB + s * P_B_BYTES), mb, fb, (kb0 + s) * KB, b_row0);
        }
      }
      pdl_wait();
      for (int u = pair; ok && u < p.num_units; u += npairs) {
        const Unit w = decode_unit(p, u);
        const int m0 = w.tm * (2 * BM) + static_cast<int>(rank) * BM;
        const int width = unit_width<MODE>(w);
        const int c0 = unit_col0<MODE>(w);
        // this CTA's B rows: SwiGLU gate (even CTA) or up (odd CTA) rows [c0, c0 + width);
        // otherwise half of [c0, c0 + width)
        const int b_rows = MODE == kEpiSwiglu ? width : width / 2;
        const int b_row0 = MODE == kEpiSwiglu ? c0 + (rank ? p.b_row_step : 0) : c0 + static_cast<int>(rank) * b_rows;
        const CUtensorMap* mb = b_rows == 128 ? &tmB : &tmB64;
        const uint32_t pair_bytes = 2u * (A_BYTES + b_rows * 128);
        const int kb1 = unit_kb1(w, num_kb);
        for (int kb = unit_kb0(w, num_kb); kb < kb1; ++kb) {
          const bool early = issued < pre;  // this stage's B and expected bytes are already issued
          if (!early && !mbar_wait(empty(stage), phase ^ 1u, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_to_rank(full(stage), 0);
          if (leader && !early) mbar_arrive_expect_tx(full(stage), pair_bytes);
          const uint32_t a_dst = smem_u32(sA + stage * A_BYTES), b_dst = smem_u32(sB + stage * P_B_BYTES);
          if (!F8 && p.a_mn) {  // A stored [K, M]: two [64 K x 64 M] blocks
            tma_load_2d_pair(a_dst, &tmA, fb, m0, kb * KB);
            tma_load_2d_pair(a_dst + 8192, &tmA, fb, m0 + 64, kb * KB);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb, kb * KB, m0);
          }
          if (early) {
          } else if (!F8 && MODE == kEpiStore && p.b_mn) {  // B stored [K, N]: b_rows / 64 blocks of [64 K x 64 N]
            for (int a = 0; a < b_rows / 64; ++a) tma_load_2d_pair(b_dst + a * 8192, &tmB, fb, b_row0 + 64 * a, kb * KB);
          } else {
            tma_load_2d_pair(b_dst, mb, fb, kb * KB, b_row0);
          }
          ++issued;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // the pair's copies in flight complete on these barriers
        for (int s = 0; s < P_STAGES; ++s)
          if (s < stage || issued >= P_STAGES)
            mbar_wait_slow(full(s), s < stage ? phase : (phase ^ 1u), nullptr, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = pair; ok && u < p.num_units; u += npairs, ++it) {
        const Unit w = decode_unit(p, u);
        const int width = unit_width<MODE>(w);
        const int n_mma = MODE == kEpiSwiglu ? 2 * width : width;
        const uint32_t idesc = F8 ? idesc_e4m3(2 * BM, n_mma)
                                  : (idesc_bf16(2 * BM, n_mma) | (p.a_mn ? 1u << 15 : 0u) | (p.b_mn ? 1u << 16 : 0u));
        const int acc = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(tempty(acc), use ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int kb0 = unit_kb0(w, num_kb), kb1 = unit_kb1(w, num_kb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full(stage), phase, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_s = smem_u32(sA + stage * A_BYTES), b_s = smem_u32(sB + stage * P_B_BYTES);
          const uint64_t ad = (!F8 && p.a_mn) ? sw128_desc_mn(a_s, 8192) : sw128_desc(a_s);
          const uint64_t bd = (!F8 && p.b_mn) ? sw128_desc_mn(b_s, 8192) : sw128_desc(b_s);
          const uint64_t astep = (!F8 && p.a_mn) ? 128ull : 2ull, bstep = (!F8 && p.b_mn) ? 128ull : 2ull;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            if (F8)
              mma_e4m3_pair(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb != kb0 || k) ? 1u : 0u);
            else
              mma_bf16_pair(d_tmem, ad + astep * k, bd + bstep * k, idesc, (kb != kb0 || k) ? 1u : 0u);
          mma_commit_pair(empty(stage));
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit_pair(tfull(acc));
      }
      // No MMA may still read either CTA's shared memory or write tensor memory at the exit.
      mma_commit_pair(drain);
      mbar_wait_slow(drain, 0, nullptr, nullptr, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else {
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
    EpiStore es{&tmO, base + P_STAGES * P_STAGE_BYTES + 1024 + (warp - 2) * 2 * EPI_BOX_BYTES, 0, 0, &tmR,
                bar0 + 256u + 16u * (warp - 2), p.err};
    int it = 0;
    for (int u = pair; part < p.epi_split && u < p.num_units; u += npairs, ++it) {
      const int acc = it & 1;
      const uint32_t use = (it >> 1) & 1;
      const Unit w = decode_unit(p, u);
      if (w.kpart == 0) prefetch_resid<MODE>(p, w, w.tm * (2 * BM) + static_cast<int>(rank) * BM, part, quad * 32 + lane);
      const bool ok = mbar_wait(tfull(acc), use, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      int lo, hi;
      epilogue_part<MODE>(p, unit_width<MODE>(w), part, lo, hi);
      if (w.kpart > 0) {
        kpart_store<MODE>(p, w, tacc, unit_col0<MODE>(w), unit_width<MODE>(w), static_cast<int>(rank), quad, part, lo,
                          hi);
      } else {
        if (w.ks > 1)
          kpart_fold<MODE>(p, w, tacc, unit_col0<MODE>(w), unit_width<MODE>(w), static_cast<int>(rank), quad, part, lo,
                           hi);
        if (lo < hi)
          epilogue_tile<MODE, F8>(p, tacc, w.tm * (2 * BM) + static_cast<int>(rank) * BM, unit_col0<MODE>(w),
                                  unit_width<MODE>(w), quad * 32 + lane, lo, hi, es);
        __syncwarp();
        if (w.ks > 1 && lane == 0)  // every partial of this launch has arrived and been read
          p.kflags[((w.tail * 2 + static_cast<int>(rank)) * 4 + quad) * 2 + part] = 0;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty(acc), 0));
    }
    if (es.n > 0 && lane == 0) cp_bulk_wait_all();  // this warp's output stores are complete
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, copies and epilogue reads are over in both CTAs
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int MODE, bool F8>
cudaError_t launch_mode(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB64, const CUtensorMap& tmO,
                        const CUtensorMap& tmR, const GemmParams& p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<MODE, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<MODE, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(P_SMEM_BYTES));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (!p.pair && p.ksplit > 1) return cudaErrorInvalidValue;  // K ranges only in the pair kernel
  if (p.ksplit > 1 && (p.kws == nullptr || p.kflags == nullptr || p.err == nullptr)) return cudaErrorInvalidValue;
  if (p.pair) {
    const int pairs = gemm_pair_slots();
    const int grid = 2 * (p.num_units < pairs ? p.num_units : pairs);
    return launch_pdl(gemm_pair_kernel<MODE, F8>, dim3(grid), dim3(GEMM_THREADS), P_SMEM_BYTES, stream, tmA, tmB, tmB64,
                      tmO, tmR, p);
  }
  const int grid = p.num_units < num_sms() ? p.num_units : num_sms();
  return launch_pdl(gemm_kernel<MODE, F8>, dim3(grid), dim3(GEMM_THREADS), SMEM_BYTES, stream, tmA, tmB, tmB64, tmO, tmR,
                    p);
}

template <bool F8>
cudaError_t launch_kind(int mode, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB64,
                        const CUtensorMap& tmO, const CUtensorMap& tmR, const GemmParams& p, cudaStream_t stream) {
  switch (mode) {
    case kEpiStore: return launch_mode<kEpiStore, F8>(tmA, tmB, tmB64, tmO, tmR, p, stream);
    case kEpiResid: return launch_mode<kEpiResid, F8>(tmA, tmB, tmB64, tmO, tmR, p, stream);
    case kEpiQkv: return launch_mode<kEpiQkv, F8>(tmA, tmB, tmB64, tmO, tmR, p, stream);
    case kEpiSwiglu: return launch_mode<kEpiSwiglu, F8>(tmA, tmB, tmB64, tmO, tmR, p, stream);
    case kEpiGelu: return launch_mode<kEpiGelu, F8>(tmA, tmB, tmB64, tmO, tmR, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_pair_slots() {
  static int n = 0;
  if (n == 0) {
    int slots = 0;
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<kEpiStore, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(P_SMEM_BYTES));
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
      cfg.blockDim = dim3(192, 1, 1);
      cfg.dynamicSmemBytes = P_SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&slots, gemm_pair_kernel<kEpiStore, false>, &cfg);
    }
    if (e != cudaSuccess || slots <= 0) {
      cudaGetLastError();  // clear a failed query; fall back to one cluster per two SMs
      slots = num_sms() / 2;
    }
    n = slots < num_sms() / 2 ? slots : num_sms() / 2;
    if (n < 1) n = 1;
  }
  return n;
}

size_t gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_gemm(int mode, bool fp8, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB64,
                        const CUtensorMap& tmO, const CUtensorMap& tmR, const GemmParams& p, cudaStream_t stream) {
  if (p.num_units <= 0) return cudaSuccess;
  if (p.tma_out && (p.out8 != nullptr || p.out32 != nullptr || (mode == kEpiQkv && p.batch != 1)))
    return cudaErrorInvalidValue;
  return fp8 ? launch_kind<true>(mode, tmA, tmB, tmB64, tmO, tmR, p, stream)
             : launch_kind<false>(mode, tmA, tmB, tmB64, tmO, tmR, p, stream);
}

}  // namespace mt
