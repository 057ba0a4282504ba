// Bandwidth-bound kernels of the layer's backward pass (the matrix products run on the tcgen05
// GEMM; the attention's own backward is in attention_bwd.cu).  The chain rule through the forward:
// norms, RoPE, SwiGLU / GeLU(tanh).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the CTA (at most 32 warps); every thread gets the total.
__device__ __forceinline__ float cta_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = warp_sum_f(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

__device__ __forceinline__ float sigmoidf(float g) { return 1.0f / (1.0f + expf(-g)); }

// SwiGLU / GeLU(tanh) forward from the stored fc1 output u: a = silu(u[:, :f]) u[:, f:] or gelu(u).
__global__ void act_fwd_kernel(const bf16* __restrict__ u, bf16* __restrict__ a, size_t T, int f, int swiglu) {
  // eight outputs (16 bytes) per thread and iteration; f is a multiple of 8
  const int f8 = f >> 3;
  const size_t n8 = T * f8;
  for (size_t v = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; v < n8;
       v += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = v / f8;
    const int c = static_cast<int>(v - t * f8) * 8;
    float r[8];
    if (swiglu) {
      float g[8], up[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * 2 * f + c), g);
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * 2 * f + f + c), up);
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = g[e] * sigmoidf(g[e]) * up[e];
    } else {
      float x[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(u + t * f + c), x);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        r[e] = 0.5f * x[e] * (1.0f + tanhf(0.7978845608028654f * (x[e] + 0.044715f * x[e] * x[e] * x[e])));
    }
    *reinterpret_cast<uint4*>(a + t * f + c) = pack_bf16x8(r);
  }
}

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
// out = add + dx (the residual branch's gradient, may be null); growth[t, :] = dy * xhat (summed
// over rows into d gamma afterwards).
__global__ void norm_bwd_kernel(const bf16* __restrict__ dy, const bf16* __restrict__ x, const bf16* __restrict__ gamma,
                                const bf16* __restrict__ add, bf16* __restrict__ out, float* __restrict__ grow, int H,
                                float eps, int layer_norm) {
  __shared__ float red[32];
  const size_t row = blockIdx.x;
  const bf16* xr = x + row * H;
  const bf16* dr = dy + row * H;
  float s1 = 0.f, s2 = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = __bfloat162float(xr[c]);
    s1 += v;
    s2 += v * v;
  }
  s1 = cta_sum(s1, red);
  s2 = cta_sum(s2, red);
  const float mean = layer_norm ? s1 / H : 0.f;
  const float var = layer_norm ? fmaxf(s2 / H - mean * mean, 0.f) : s2 / H;
  float var2 = var;
  if (layer_norm) {  // two-pass variance for accuracy
    float sq = 0.f;
    for (int c = threadIdx.x; c < H; c += blockDim.x) {
      const float dd = __bfloat162float(xr[c]) - mean;
      sq += dd * dd;
    }
    var2 = cta_sum(sq, red) / H;
  }
  const float r = rsqrtf(var2 + eps);
  float a1 = 0.f, a2 = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float xh = (__bfloat162float(xr[c]) - mean) * r;
    const float gx = __bfloat162float(dr[c]) * __bfloat162float(gamma[c]);
    a1 += gx;
    a2 += gx * xh;
  }
  a1 = cta_sum(a1, red) / H;
  a2 = cta_sum(a2, red) / H;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float xh = (__bfloat162float(xr[c]) - mean) * r;
    const float g = __bfloat162float(dr[c]);
    const float gx = g * __bfloat162float(gamma[c]);
    float dx = r * (gx - xh * a2 - (layer_norm ? a1 : 0.f));
    if (add != nullptr) dx += __bfloat162float(add[row * H + c]);
    out[row * H + c] = __float2bfloat16_rn(dx);
    grow[row * H + c] = g * xh;
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

// dqkv[t, :] from the per-head fp32 gradients of q, k (after RoPE) and v: the rotation's transpose
// (the opposite angle) on q and k, then [q heads | k groups | v groups] in the fused layout.
__global__ void rope_bwd_pack_kernel(const float* __restrict__ dq, const float* __restrict__ dk,
                                     const float* __restrict__ dv, const float2* __restrict__ rope,
                                     bf16* __restrict__ dqkv, int S, int B, int nh, int ng, int d) {
  const int t = blockIdx.x;  // token row s*B + b
  const int s = t / B, b = t - s * B;
  const int half = d / 2;
  const int ncols = (nh + 2 * ng) * d;
  for (int c = threadIdx.x; c < ncols; c += blockDim.x) {
    const int head = c / d, i = c - head * d;
    const float* src;
    if (head < nh) src = dq + ((static_cast<size_t>(b) * nh + head) * S + s) * d;
    else if (head < nh + ng) src = dk + ((static_cast<size_t>(b) * ng + head - nh) * S + s) * d;
    else src = dv + ((static_cast<size_t>(b) * ng + head - nh - ng) * S + s) * d;
    float g = src[i];
    if (rope != nullptr && head < nh + ng) {
      const int p = i < half ? i : i - half;
      const float2 cs = rope[static_cast<size_t>(s) * half + p];
      // forward: y1 = x1 c - x2 s, y2 = x2 c + x1 s  ->  dx1 = dy1 c + dy2 s, dx2 = dy2 c - dy1 s
      g = i < half ? src[i] * cs.x + src[i + half] * cs.y : src[i] * cs.x - src[i - half] * cs.y;
    }
    dqkv[static_cast<size_t>(t) * ncols + c] = __float2bfloat16_rn(g);
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

cudaError_t launch_act_fwd(const bf16* u, bf16* a, size_t T, int f, bool swiglu, cudaStream_t st) {
  if (f % 8) return cudaErrorInvalidValue;
  act_fwd_kernel<<<act_grid(T, f), 256, 0, st>>>(u, a, T, f, swiglu ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_act_bwd(const bf16* u, const bf16* da, bf16* du, size_t T, int f, bool swiglu, cudaStream_t st) {
  if (f % 8) return cudaErrorInvalidValue;
  act_bwd_kernel<<<act_grid(T, f), 256, 0, st>>>(u, da, du, T, f, swiglu ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(const bf16* dy, const bf16* x, const bf16* gamma, const bf16* add, bf16* out, float* grow,
                            int T, int H, float eps, bool layer_norm, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  norm_bwd_kernel<<<T, 256, 0, st>>>(dy, x, gamma, add, out, grow, H, eps, layer_norm ? 1 : 0);
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

cudaError_t launch_rope_bwd_pack(const float* dq, const float* dk, const float* dv, const float2* rope, bf16* dqkv,
                                 int S, int B, int nh, int ng, int d, cudaStream_t st) {
  rope_bwd_pack_kernel<<<S * B, 256, 0, st>>>(dq, dk, dv, rope, dqkv, S, B, nh, ng, d);
  return cudaGetLastError();
}

}  // namespace mt
