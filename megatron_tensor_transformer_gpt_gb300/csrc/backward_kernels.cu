// Bandwidth-bound kernels of the layer's backward pass (the matrix products run on the tcgen05
// GEMM; the attention's own backward is in attention_bwd.cu).  The chain rule through the forward:
// norms, RoPE, SwiGLU / GeLU(tanh).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf(float g) { return 1.0f / (1.0f + expf(-g)); }

// Gradient through the activation: du from da = dL/da and the fc1 output u.
//   SwiGLU: d gate = da up silu'(gate), d up = da silu(gate), silu'(g) = s (1 + g (1 - s)), s = sigmoid(g)
//   GeLU(tanh): du = da gelu'(u)
__global__ void act_bwd_kernel(const bf16* __restrict__ u, const bf16* __restrict__ da, bf16* __restrict__ du, size_t T,
                               int f, int swiglu) {
  const int f8 = f >> 3;
  const size_t n8 = T * f8;
  for (size_t v = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; v < n8;
       v += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = v / f8;
    const int c = static_cast<int>(v - t * f8) * 8;
    float ga[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(da + t * f + c), ga);
    if (swiglu) {
      float g[8], up[8], dg[8], dup[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * 2 * f + c), g);
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * 2 * f + f + c), up);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float sg = sigmoidf(g[e]);
        dg[e] = ga[e] * up[e] * sg * (1.0f + g[e] * (1.0f - sg));
        dup[e] = ga[e] * g[e] * sg;
      }
      *reinterpret_cast<uint4*>(du + t * 2 * f + c) = pack_bf16x8(dg);
      *reinterpret_cast<uint4*>(du + t * 2 * f + f + c) = pack_bf16x8(dup);
    } else {
      float x[8], r[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * f + c), x);
      const float k0 = 0.7978845608028654f, k1 = 0.044715f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float th = tanhf(k0 * (x[e] + k1 * x[e] * x[e] * x[e]));
        const float d = 0.5f * (1.0f + th) + 0.5f * x[e] * (1.0f - th * th) * k0 * (1.0f + 3.0f * k1 * x[e] * x[e]);
        r[e] = ga[e] * d;
      }
      *reinterpret_cast<uint4*>(du + t * f + c) = pack_bf16x8(r);
    }
  }
}

// Norm backward of one row (CTA per row): with xhat, r = 1/sigma recomputed from the norm input
// x and gx = dy * gamma,
//   RMSNorm:   dx = r (gx - xhat mean(gx xhat))
//   LayerNorm: dx = r (gx - mean(gx) - xhat mean(gx xhat))
// out = add + dx (the residual branch's gradient, may be null); d gamma = sum over rows of dy * xhat
// and d beta = sum of dy (LayerNorm), gathered as per-CTA partial rows.
constexpr int kNormBwdRows = 16;  // rows per CTA: one partial row of d gamma (and d beta) per CTA

// Sum of (a, b) over the CTA; every thread gets both totals.
__device__ __forceinline__ float2 cta_sum2(float a, float b, float2* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  a = warp_sum_f(a);
  b = warp_sum_f(b);
  __syncthreads();
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  for (int i = 0; i < nw; ++i) {
    t.x += red[i].x;
    t.y += red[i].y;
  }
  return t;
}

// One CTA per kNormBwdRows rows; each thread holds VPT 8-column vectors of a row in registers (x
// and dy read once, 16 bytes at a time); the next row's x and dy, and the current row's `add`, are
// loaded while the current row is reduced, so the rows' load latencies overlap.  partial[blockIdx.x, :] = sum over the CTA's rows of
// dy * xhat (and, LayerNorm, partial[gridDim.x + blockIdx.x, :] = sum of dy), folded over the CTAs
// by the column-sum kernel into d gamma (d beta).
template <int VPT, bool LN>
__global__ void __launch_bounds__(1024) norm_bwd_kernel(const bf16* __restrict__ dy, const bf16* __restrict__ x,
                                                        const bf16* __restrict__ gamma, const bf16* __restrict__ add,
                                                        bf16* __restrict__ out, float* __restrict__ partial, int T,
                                                        int H, float eps) {
  __shared__ float2 red[32];
  const int nvec = H >> 3;
  const float inv_h = 1.0f / static_cast<float>(H);
  float gm[VPT][8], pg[VPT][8], pb[VPT][8];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    if (idx < nvec) {
      unpack_bf16x8(reinterpret_cast<const uint4*>(gamma)[idx], gm[i]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gm[i][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) pg[i][e] = pb[i][e] = 0.f;
  }
  const int r_end = min(T, static_cast<int>(blockIdx.x + 1) * kNormBwdRows);
  // raw 16-byte vectors of x and dy of a row (zero past the row's end)
  uint4 rx[VPT], rg[VPT];
  auto fetch = [&](int row) {
    const size_t base = static_cast<size_t>(row) * nvec;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = i * blockDim.x + threadIdx.x;
      const bool in = idx < nvec;
      rx[i] = in ? reinterpret_cast<const uint4*>(x)[base + idx] : make_uint4(0u, 0u, 0u, 0u);
      rg[i] = in ? reinterpret_cast<const uint4*>(dy)[base + idx] : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (static_cast<int>(blockIdx.x) * kNormBwdRows < r_end) fetch(blockIdx.x * kNormBwdRows);
  for (int row = blockIdx.x * kNormBwdRows; row < r_end; ++row) {
    const size_t base = static_cast<size_t>(row) * nvec;
    float xv[VPT][8], gv[VPT][8];
    uint4 rad[VPT];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = i * blockDim.x + threadIdx.x;
      unpack_bf16x8(rx[i], xv[i]);
      unpack_bf16x8(rg[i], gv[i]);
      rad[i] = (idx < nvec && add != nullptr) ? reinterpret_cast<const uint4*>(add)[base + idx] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s1 += xv[i][e];
        s2 += xv[i][e] * xv[i][e];
      }
    }
    if (row + 1 < r_end) fetch(row + 1);
    float mean = 0.f, var;
    if (LN) {  // two-pass variance from the registers
      mean = cta_sum2(s1, 0.f, red).x * inv_h;
      float sq = 0.f;
#pragma unroll
      for (int i = 0; i < VPT; ++i)
        if (i * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x) < nvec)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float dd = xv[i][e] - mean;
            sq += dd * dd;
          }
      var = cta_sum2(sq, 0.f, red).x * inv_h;
    } else {
      var = cta_sum2(s2, 0.f, red).x * inv_h;
    }
    const float r = rsqrtf(var + eps);
    float a1 = 0.f, a2 = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xh = (xv[i][e] - mean) * r, gx = gv[i][e] * gm[i][e];
        a1 += gx;
        a2 += gx * xh;
      }
    const float2 a = cta_sum2(a1, a2, red);
    const float m1 = LN ? a.x * inv_h : 0.f, m2 = a.y * inv_h;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = i * blockDim.x + threadIdx.x;
      if (idx >= nvec) continue;
      float ad[8], o[8];
      unpack_bf16x8(rad[i], ad);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xh = (xv[i][e] - mean) * r;
        o[e] = r * (gv[i][e] * gm[i][e] - xh * m2 - m1) + ad[e];
        pg[i][e] += gv[i][e] * xh;
        pb[i][e] += gv[i][e];
      }
      reinterpret_cast<uint4*>(out)[base + idx] = pack_bf16x8(o);
    }
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    if (idx >= nvec) continue;
    float4* pr = reinterpret_cast<float4*>(partial + static_cast<size_t>(blockIdx.x) * H + idx * 8);
    pr[0] = make_float4(pg[i][0], pg[i][1], pg[i][2], pg[i][3]);
    pr[1] = make_float4(pg[i][4], pg[i][5], pg[i][6], pg[i][7]);
    if (LN) {
      float4* pq = reinterpret_cast<float4*>(partial + static_cast<size_t>(gridDim.x + blockIdx.x) * H + idx * 8);
      pq[0] = make_float4(pb[i][0], pb[i][1], pb[i][2], pb[i][3]);
      pq[1] = make_float4(pb[i][4], pb[i][5], pb[i][6], pb[i][7]);
    }
  }
}

// Column sums of a [T, N] matrix (bf16 or fp32, pitch ld) in fp32, written as bf16; rows split
// over gridDim.y and folded with fp32 atomics into acc (zeroed by the caller), then converted.
template <typename In>
__global__ void colsum_kernel(const In* __restrict__ src, size_t ld, int T, int N, float* acc) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= N) return;
  const int per = (T + gridDim.y - 1) / gridDim.y;
  const int r0 = blockIdx.y * per, r1 = min(T, r0 + per);
  float s = 0.f;
  for (int r = r0; r < r1; ++r) {
    if constexpr (sizeof(In) == 2)
      s += __bfloat162float(src[static_cast<size_t>(r) * ld + c]);
    else
      s += src[static_cast<size_t>(r) * ld + c];
  }
  atomicAdd(acc + c, s);
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ a, bf16* __restrict__ b, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) b[i] = __float2bfloat16_rn(a[i]);
}

// Eight consecutive floats at src, summed over n buffers `stride` floats apart (in buffer order).
__device__ __forceinline__ void load8_sum(const float* src, int n, size_t stride, float* g) {
  *reinterpret_cast<float4*>(g) = *reinterpret_cast<const float4*>(src);
  *reinterpret_cast<float4*>(g + 4) = *reinterpret_cast<const float4*>(src + 4);
  for (int r = 1; r < n; ++r) {
    const float4 a = *reinterpret_cast<const float4*>(src + r * stride);
    const float4 c = *reinterpret_cast<const float4*>(src + r * stride + 4);
    g[0] += a.x;
    g[1] += a.y;
    g[2] += a.z;
    g[3] += a.w;
    g[4] += c.x;
    g[5] += c.y;
    g[6] += c.z;
    g[7] += c.w;
  }
}

// dqkv[t, :] from the per-head fp32 gradients of q, k (after RoPE) and v: the rotation's transpose
// (the opposite angle) on q and k, then [q heads | k groups | v groups] in the fused layout; dk and dv
// are summed over `parts` partial buffers first.
__global__ void rope_bwd_pack_kernel(const float* __restrict__ dq, const float* __restrict__ dk,
                                     const float* __restrict__ dv, int parts, size_t part_stride,
                                     const float2* __restrict__ rope, bf16* __restrict__ dqkv, int S, int B, int nh,
                                     int ng, int d) {
  const int t = blockIdx.x;  // token row s*B + b
  const int s = t / B, b = t - s * B;
  const int half = d / 2;
  const int ncols = (nh + 2 * ng) * d;
  // eight consecutive columns of one head per thread and step (d / 2 is a multiple of 8)
  for (int c = threadIdx.x * 8; c < ncols; c += blockDim.x * 8) {
    const int head = c / d, i = c - head * d;
    const float* src;
    if (head < nh) src = dq + ((static_cast<size_t>(b) * nh + head) * S + s) * d;
    else if (head < nh + ng) src = dk + ((static_cast<size_t>(b) * ng + head - nh) * S + s) * d;
    else src = dv + ((static_cast<size_t>(b) * ng + head - nh - ng) * S + s) * d;
    const int np = head < nh ? 1 : parts;  // dk and dv: the sum of the partial buffers
    float g[8];
    load8_sum(src + i, np, part_stride, g);
    if (rope != nullptr && head < nh + ng) {
      // forward: y1 = x1 c - x2 s, y2 = x2 c + x1 s  ->  dx1 = dy1 c + dy2 s, dx2 = dy2 c - dy1 s
      const bool first = i < half;
      const int p = first ? i : i - half;
      float o[8];
      load8_sum(src + (first ? i + half : i - half), np, part_stride, o);
      const float4* cs4 = reinterpret_cast<const float4*>(rope + static_cast<size_t>(s) * half + p);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 cs = cs4[k];  // (cos, sin) of columns p + 2k and p + 2k + 1
        const float sg = first ? 1.f : -1.f;
        g[2 * k] = g[2 * k] * cs.x + sg * o[2 * k] * cs.y;
        g[2 * k + 1] = g[2 * k + 1] * cs.z + sg * o[2 * k + 1] * cs.w;
      }
    }
    *reinterpret_cast<uint4*>(dqkv + static_cast<size_t>(t) * ncols + c) = pack_bf16x8(g);
  }
}

// dst[C, R] = src[R, C]^T (bf16; pitches in elements; R and C multiples of 8) through a 64 x 64 tile in
// shared memory, every global load and store a 16-byte vector and coalesced (a warp moves 128
// contiguous bytes of four rows).  Tile row r keeps its eight 16-byte chunks with chunk ch at
// ch ^ (r / 8), so that the transposed reads (2-byte elements of one column from eight rows 8g ..
// 8g + 7, g differing across a warp) fall in distinct banks.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const bf16* __restrict__ src, size_t sp,
                                                             bf16* __restrict__ dst, size_t dp, int R, int C) {
  __shared__ uint4 tile[64 * 8];
  const int tr = blockIdx.y * 64, tc = blockIdx.x * 64;  // tile origin in src (row, column)
  const int t = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = t / 8 + 32 * k, ch = t % 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (tr + r < R && tc + 8 * ch < C) v = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(tr + r) * sp + tc + 8 * ch);
    tile[r * 8 + ((ch ^ (r >> 3)) & 7)] = v;
  }
  __syncthreads();
  const uint16_t* ts = reinterpret_cast<const uint16_t*>(tile);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int c = t / 8 + 32 * k, g = t % 8;  // dst row tc + c holds src rows tr + 8g .. tr + 8g + 7 here
    if (tc + c >= C || tr + 8 * g >= R) continue;
    const int phys = (((c >> 3) ^ g) & 7) * 8 + (c & 7);  // element c of a row of group g
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = static_cast<uint32_t>(ts[(8 * g + 2 * q) * 64 + phys]) |
             (static_cast<uint32_t>(ts[(8 * g + 2 * q + 1) * 64 + phys]) << 16);
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(tc + c) * dp + tr + 8 * g) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The attention backward's V operand in bf16 (its dP = dO V^T product pairs it with the bf16 dO) from
// the forward's head-major fp16 V: fp16 -> fp32 is exact, then one round to nearest even.  n8
// vectors of eight elements.
__global__ void f16_to_bf16_kernel(const __half* __restrict__ src, bf16* __restrict__ dst, size_t n8) {
  for (size_t v = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; v < n8;
       v += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[v];
    const __half2* h = reinterpret_cast<const __half2*>(&u);
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __half22float2(h[e]);
      f[2 * e] = x.x;
      f[2 * e + 1] = x.y;
    }
    reinterpret_cast<uint4*>(dst)[v] = pack_bf16x8(f);
  }
}

}  // namespace

// Blocks of 256 threads for T x f / 8 vectors: one pass, at most 32 blocks per SM.
static unsigned act_grid(size_t T, int f) {
  const size_t n8 = T * static_cast<size_t>(f / 8);
  const size_t blocks = (n8 + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms()) * 32;
  return static_cast<unsigned>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_act_bwd(const bf16* u, const bf16* da, bf16* du, size_t T, int f, bool swiglu, cudaStream_t st) {
  if (f % 8) return cudaErrorInvalidValue;
  act_bwd_kernel<<<act_grid(T, f), 256, 0, st>>>(u, da, du, T, f, swiglu ? 1 : 0);
  return cudaGetLastError();
}

int norm_bwd_blocks(int T) { return (T + kNormBwdRows - 1) / kNormBwdRows; }

cudaError_t launch_norm_bwd(const bf16* dy, const bf16* x, const bf16* gamma, const bf16* add, bf16* out,
                            float* partial, int T, int H, float eps, bool layer_norm, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (H % 8 != 0 || H > 8192) return cudaErrorInvalidValue;  // one 8-column vector per thread
  const int threads = (H / 8 + 31) / 32 * 32;
  const int blocks = norm_bwd_blocks(T);
  if (layer_norm) norm_bwd_kernel<1, true><<<blocks, threads, 0, st>>>(dy, x, gamma, add, out, partial, T, H, eps);
  else norm_bwd_kernel<1, false><<<blocks, threads, 0, st>>>(dy, x, gamma, add, out, partial, T, H, eps);
  return cudaGetLastError();
}

cudaError_t launch_colsum(const void* src, bool f32, size_t ld, int T, int N, float* acc, bf16* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(acc, 0, static_cast<size_t>(N) * sizeof(float), st);
  if (e != cudaSuccess) return e;
  const dim3 grid((N + 255) / 256, T >= 4096 ? 32 : (T + 127) / 128);
  if (f32) colsum_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(src), ld, T, N, acc);
  else colsum_kernel<bf16><<<grid, 256, 0, st>>>(static_cast<const bf16*>(src), ld, T, N, acc);
  f32_to_bf16_kernel<<<(N + 255) / 256, 256, 0, st>>>(acc, out, N);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const bf16* src, size_t sp, bf16* dst, size_t dp, int R, int C, cudaStream_t st) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (R % 8 || C % 8 || sp % 8 || dp % 8 || reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16)
    return cudaErrorInvalidValue;
  transpose_bf16_kernel<<<dim3((C + 63) / 64, (R + 63) / 64), 256, 0, st>>>(src, sp, dst, dp, R, C);
  return cudaGetLastError();
}

cudaError_t launch_f16_to_bf16(const __half* src, bf16* dst, size_t n, cudaStream_t st) {
  if (n % 8) return cudaErrorInvalidValue;
  f16_to_bf16_kernel<<<act_grid(n / 8, 8), 256, 0, st>>>(src, dst, n / 8);
  return cudaGetLastError();
}

cudaError_t launch_rope_bwd_pack(const float* dq, const float* dk, const float* dv, int parts, size_t part_stride,
                                 const float2* rope, bf16* dqkv, int S, int B, int nh, int ng, int d, cudaStream_t st) {
  if (parts < 1 || part_stride % 8 != 0) return cudaErrorInvalidValue;
  if (d % 16 != 0) return cudaErrorInvalidValue;  // eight-column vectors inside each half of a head
  const int threads = std::min(256, ((nh + 2 * ng) * d / 8 + 31) / 32 * 32);
  rope_bwd_pack_kernel<<<S * B, threads, 0, st>>>(dq, dk, dv, parts, part_stride, rope, dqkv, S, B, nh, ng, d);
  return cudaGetLastError();
}

}  // namespace mt
