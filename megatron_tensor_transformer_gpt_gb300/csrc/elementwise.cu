// Bandwidth-bound pieces of the layer: the input / pre-MLP norms, the RoPE angle table, and the
// bounded-wait self test.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace mt {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 u;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
               : "l"(p));
  return u;
}

// Sum over the CTA (at most 32 warps); every thread gets the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();  // `red` may still be read by a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

// One CTA per row; thread i holds VPT 16-byte vectors (8 bf16 each) of the row in registers,
// statistics in fp32.
//   RMSNorm:   y = x / sqrt(mean(x^2) + eps) * g           (input_layernorm for LLaMA)
//   LayerNorm: y = (x - mean) / sqrt(var + eps) * g + b     (biased variance, two passes)
template <int VPT, bool LN>
__global__ void __launch_bounds__(1024) norm_kernel(const bf16* __restrict__ x, const bf16* __restrict__ gamma,
                                                    const bf16* __restrict__ beta, bf16* __restrict__ y, int H,
                                                    float eps) {
  __shared__ float red[32];
  const size_t row = blockIdx.x;
  const int nvec = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
  uint4 raw[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    raw[i] = idx < nvec ? ld_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float f[8];
    unpack_bf16x8(raw[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += LN ? f[e] : f[e] * f[e];
  }
  acc = block_sum(acc, red);
  const float inv_h = 1.0f / static_cast<float>(H);
  float mean = 0.f, rstd;
  if (LN) {
    mean = acc * inv_h;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (i * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x) < nvec) {
        float f[8];
        unpack_bf16x8(raw[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dd = f[e] - mean;
          sq += dd * dd;
        }
      }
    }
    sq = block_sum(sq, red);
    rstd = rsqrtf(sq * inv_h + eps);
  } else {
    rstd = rsqrtf(acc * inv_h + eps);
  }
  uint4* yr = reinterpret_cast<uint4*>(y + row * H);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const uint4* br = reinterpret_cast<const uint4*>(beta);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    if (idx < nvec) {
      float f[8], gf[8], bfv[8], o[8];
      unpack_bf16x8(raw[i], f);
      unpack_bf16x8(__ldg(gr + idx), gf);
      if (LN) unpack_bf16x8(__ldg(br + idx), bfv);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * gf[e] + (LN ? bfv[e] : 0.f);
      yr[idx] = pack_bf16x8(o);
    }
  }
}

template <bool LN>
cudaError_t launch_norm_ln(const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int H, float eps,
                           cudaStream_t stream) {
  const int nvec = H / 8;
  if (nvec >= 256) {  // two vectors per thread
    const int threads = ((nvec + 1) / 2 + 31) / 32 * 32;
    if (threads > 1024) return cudaErrorInvalidValue;
    norm_kernel<2, LN><<<rows, threads, 0, stream>>>(x, g, b, y, H, eps);
  } else {
    const int threads = (nvec + 31) / 32 * 32;
    norm_kernel<1, LN><<<rows, threads, 0, stream>>>(x, g, b, y, H, eps);
  }
  return cudaGetLastError();
}

// (cos, sin) of s * theta_i for s < seq, i < half.  The angle is formed and reduced modulo 2*pi
// in double precision, so the single-precision sine/cosine act on an argument in [-pi, pi].
__global__ void rope_table_kernel(float2* __restrict__ tab, const double* __restrict__ theta, int seq, int half) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= seq * half) return;
  const int s = idx / half, i = idx - s * half;
  const double a = static_cast<double>(s) * theta[i];
  const double turns = rint(a * 0.15915494309189535);  // a / (2 pi)
  const float r = static_cast<float>(fma(-turns, 6.283185307179586, a));
  float sn, cs;
  sincosf(r, &sn, &cs);
  tab[idx] = make_float2(cs, sn);
}

// A barrier nothing will ever complete: the bounded wait has to give up and report.
__global__ void wait_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_slow(smem_u32(&bar), 0, err, &abort_flag, limit_ns);
}


// Sequence-parallel epilogue of a row-parallel linear (one rank's slice of the reduce-scatter, fused
// with bias-dropout-add and the next norm).  One CTA per output row; thread i holds VPT 16-byte
// vectors.  h = resid + sum_i partial_i + bias is summed in fp32 and stored as bf16; the norm's
// statistics are taken over the stored bf16 values, as the unfused norm kernel would see them.
template <int VPT, bool LN>
__global__ void __launch_bounds__(1024) sp_add_norm_kernel(const SpParams p) {
  __shared__ float red[32];
  const size_t row = blockIdx.x;  // row within the slice
  const int nvec = p.H >> 3;
  const uint4* rr = reinterpret_cast<const uint4*>(p.resid + row * p.H);
  uint4 hv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    hv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < nvec) {
      float acc[8], f[8];
      unpack_bf16x8(ld_stream(rr + idx), acc);
      for (int k = 0; k < p.nparts; ++k) {
        unpack_bf16x8(ld_stream(reinterpret_cast<const uint4*>(p.parts[k] + (p.row0 + row) * p.H) + idx), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
      if (p.bias != nullptr) {
        unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.bias) + idx), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
      hv[i] = pack_bf16x8(acc);
      reinterpret_cast<uint4*>(p.h + row * p.H)[idx] = hv[i];
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float f[8];
    unpack_bf16x8(hv[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += LN ? f[e] : f[e] * f[e];
  }
  acc = block_sum(acc, red);
  const float inv_h = 1.0f / static_cast<float>(p.H);
  float mean = 0.f, rstd;
  if (LN) {
    mean = acc * inv_h;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (i * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x) < nvec) {
        float f[8];
        unpack_bf16x8(hv[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dd = f[e] - mean;
          sq += dd * dd;
        }
      }
    }
    sq = block_sum(sq, red);
    rstd = rsqrtf(sq * inv_h + p.eps);
  } else {
    rstd = rsqrtf(acc * inv_h + p.eps);
  }
  const uint4* gr = reinterpret_cast<const uint4*>(p.gamma);
  const uint4* br = reinterpret_cast<const uint4*>(p.beta);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = i * blockDim.x + threadIdx.x;
    if (idx < nvec) {
      float f[8], gf[8], bfv[8], o[8];
      unpack_bf16x8(hv[i], f);
      unpack_bf16x8(__ldg(gr + idx), gf);
      if (LN) unpack_bf16x8(__ldg(br + idx), bfv);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * gf[e] + (LN ? bfv[e] : 0.f);
      reinterpret_cast<uint4*>(p.hn + row * p.H)[idx] = pack_bf16x8(o);
    }
  }
}

template <bool LN>
cudaError_t launch_sp_ln(const SpParams& p, cudaStream_t stream) {
  const int nvec = p.H / 8;
  if (nvec >= 256) {
    const int threads = ((nvec + 1) / 2 + 31) / 32 * 32;
    if (threads > 1024) return cudaErrorInvalidValue;
    sp_add_norm_kernel<2, LN><<<p.rows, threads, 0, stream>>>(p);
  } else {
    sp_add_norm_kernel<1, LN><<<p.rows, (nvec + 31) / 32 * 32, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

// Per-token index of packed samples: token t of sample i (cu[i] <= t < cu[i+1]) has RoPE
// position t - cu[i] and v^T column 8*ceil(cu[i]/8) + 8*i + (t - cu[i]) (every sample starts on
// a 16-byte boundary of v^T, as the TMA loads need).  Inconsistent cu_seqlens are reported in
// *err and mapped to index 0, which keeps every later access in bounds.
__global__ void packed_index_kernel(const int* __restrict__ cu, int n, int T, int max_len, int vcols,
                                    int* __restrict__ pos, int* __restrict__ vcol, int* err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  bool ok = (t != 0 || (cu[0] == 0 && cu[n] == T));
  int lo = 0, hi = n - 1;  // largest i with cu[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int start = cu[lo], end = cu[lo + 1];
  const int p = t - start;
  const int v = 8 * ((start + 7) / 8) + 8 * lo + p;
  ok = ok && start <= t && t < end && p < max_len && start >= 0 && v < vcols;
  if (!ok) atomicCAS(err, 0, 1);  // MT_ERR_INVALID_ARG
  pos[t] = ok ? p : 0;
  vcol[t] = ok ? v : 0;
}

}  // namespace

cudaError_t launch_norm(bool layer_norm, const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int hidden,
                        float eps, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return layer_norm ? launch_norm_ln<true>(x, g, b, y, rows, hidden, eps, stream)
                    : launch_norm_ln<false>(x, g, b, y, rows, hidden, eps, stream);
}

cudaError_t launch_rope_table(float2* table, const double* theta, int seq, int half, cudaStream_t stream) {
  const int n = seq * half;
  if (n <= 0) return cudaSuccess;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(table, theta, seq, half);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_sp_add_norm(bool layer_norm, const SpParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  return layer_norm ? launch_sp_ln<true>(p, stream) : launch_sp_ln<false>(p, stream);
}

cudaError_t launch_packed_index(const int* cu, int num_seqs, int tokens, int max_seqlen, int vcols, int* pos, int* vcol,
                                int* err, cudaStream_t stream) {
  if (tokens <= 0) return cudaSuccess;
  packed_index_kernel<<<(tokens + 255) / 256, 256, 0, stream>>>(cu, num_seqs, tokens, max_seqlen, vcols, pos, vcol, err);
  return cudaGetLastError();
}

}  // namespace mt
