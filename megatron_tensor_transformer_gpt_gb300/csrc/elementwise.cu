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

// (cos, sin) of s * theta_i.  The angle is formed and reduced modulo 2*pi in double precision, so
// the single-precision sine/cosine act on an argument in [-pi, pi].
__device__ __forceinline__ float2 rope_entry(int s, double theta_i) {
  const double a = static_cast<double>(s) * theta_i;
  const double turns = rint(a * 0.15915494309189535);  // a / (2 pi)
  const float r = static_cast<float>(fma(-turns, 6.283185307179586, a));
  float sn, cs;
  sincosf(r, &sn, &cs);
  return make_float2(cs, sn);
}

// Norm of token rows, statistics in fp32:
//   RMSNorm:   y = x / sqrt(mean(x^2) + eps) * g           (input_layernorm for LLaMA)
//   LayerNorm: y = (x - mean) / sqrt(var + eps) * g + b     (biased variance, two passes)
// A row belongs to W warps of an NW-warp CTA (NW / W rows per CTA); lane l of the row's warp w
// holds the VPL 16-byte vectors (8 bf16 each) i * 32W + 32w + l, so every load and store of a warp
// covers 512 contiguous bytes, the whole row sits in registers between the reduction and the
// output, and all loads of a thread are in flight at once.  The warps of a row combine their sums
// through shared memory (one barrier per reduction); W = 1 reduces with shuffles only.  Measured
// on the Llama-3-8B (H = 4096), GPT-345M (1024) and 70B (8192) rows: two vectors per thread and
// many small CTAs beat whole rows per warp (which hold 16 vectors per thread and leave fewer loads
// in flight per SM) by 25-40%.
// OUT8: write E4M3 codes of y * (*q_scale) to y8 instead of bf16 y, and fold max |y| of the CTA's
// rows into *amax (one atomic per CTA).
// rope.tab != null: the warps of row r also write row rope.row0 + r of the RoPE table (when below
// rope.rows), so the table needs no launch of its own.
template <int VPL, int W, int NW, bool LN, bool OUT8>
__global__ void __launch_bounds__(NW * 32, VPL == 1 ? 2048 / (NW * 32) : 1536 / (NW * 32))
    norm_kernel(const bf16* __restrict__ x, const bf16* __restrict__ gamma, const bf16* __restrict__ beta,
                bf16* __restrict__ y, int rows, int H, float eps, uint8_t* __restrict__ y8, const float* q_scale,
                unsigned* amax, const RopeRows rope) {
  constexpr int kRows = NW / W;
  __shared__ float red1[NW], red2[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = warp % W;
  const int r = static_cast<int>(blockIdx.x) * kRows + warp / W;
  const bool valid = r < rows;
  pdl_wait();
  pdl_trigger();
  const size_t row = static_cast<size_t>(valid ? r : 0);
  const int nvec = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
  uint4 raw[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = (i * W + sub) * 32 + lane;
    raw[i] = valid && idx < nvec ? ld_stream(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    float f[8];
    unpack_bf16x8(raw[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += LN ? f[e] : f[e] * f[e];
  }
  acc = warp_sum(acc);
  if (W > 1) {
    if (lane == 0) red1[warp] = acc;
    __syncthreads();
    acc = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) acc += red1[warp - sub + j];
  }
  const float inv_h = 1.0f / static_cast<float>(H);
  float mean = 0.f, rstd;
  if (LN) {
    mean = acc * inv_h;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if ((i * W + sub) * 32 + lane < nvec) {
        float f[8];
        unpack_bf16x8(raw[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dd = f[e] - mean;
          sq += dd * dd;
        }
      }
    }
    sq = warp_sum(sq);
    if (W > 1) {
      if (lane == 0) red2[warp] = sq;
      __syncthreads();
      sq = 0.f;
#pragma unroll
      for (int j = 0; j < W; ++j) sq += red2[warp - sub + j];
    }
    rstd = rsqrtf(sq * inv_h + eps);
  } else {
    rstd = rsqrtf(acc * inv_h + eps);
  }
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const uint4* br = reinterpret_cast<const uint4*>(beta);
  const float qs = OUT8 ? __ldg(q_scale) : 1.f;
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = (i * W + sub) * 32 + lane;
    if (valid && idx < nvec) {
      float f[8], gf[8], bfv[8], o[8];
      unpack_bf16x8(raw[i], f);
      unpack_bf16x8(__ldg(gr + idx), gf);
      if (LN) unpack_bf16x8(__ldg(br + idx), bfv);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * gf[e] + (LN ? bfv[e] : 0.f);
      if (OUT8) {
#pragma unroll
        for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(o[e]));
        reinterpret_cast<uint2*>(y8 + row * H)[idx] = pack_e4m3x8(o, qs);
      } else {
        reinterpret_cast<uint4*>(y + row * H)[idx] = pack_bf16x8(o);
      }
    }
  }
  // the RoPE table rows last, so that their arithmetic does not delay the row's loads
  if (valid && rope.tab != nullptr) {
    const int s = rope.row0 + r;
    if (s < rope.rows)
      for (int i = sub * 32 + lane; i < rope.half; i += 32 * W)
        rope.tab[static_cast<size_t>(s) * rope.half + i] = rope_entry(s, rope.theta[i]);
  }
  if (OUT8) {
    mx = warp_max(mx);
    __syncthreads();
    if (lane == 0) red1[warp] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < NW; ++i) mx = fmaxf(mx, red1[i]);
      atomic_max_abs(amax, mx);
    }
  }
}

template <int VPL, int W, bool LN, bool OUT8>
cudaError_t launch_norm_v(const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int H, float eps,
                          uint8_t* y8, const float* q_scale, unsigned* amax, const RopeRows& rope,
                          cudaStream_t stream) {
  constexpr int NW = W > 8 ? W : 8;
  const int ctas = (rows + NW / W - 1) / (NW / W);
  return launch_pdl(norm_kernel<VPL, W, NW, LN, OUT8>, dim3(ctas), dim3(NW * 32), 0, stream, x, g, b, y, rows, H,
                    eps, y8, q_scale, amax, rope);
}

// Two vectors per thread (one below 64 vectors a row) and as many warps per row as that needs.
template <bool LN, bool OUT8>
cudaError_t launch_norm_ln(const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int H, float eps,
                           uint8_t* y8, const float* q_scale, unsigned* amax, const RopeRows& rope,
                           cudaStream_t stream) {
  const int nvec = H / 8;
  if (nvec > 1024) return cudaErrorInvalidValue;
  if (nvec > 512) return launch_norm_v<2, 16, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
  if (nvec > 256) return launch_norm_v<2, 8, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
  if (nvec > 128) return launch_norm_v<2, 4, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
  if (nvec > 64) return launch_norm_v<2, 2, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
  if (nvec > 32) return launch_norm_v<2, 1, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
  return launch_norm_v<1, 1, LN, OUT8>(x, g, b, y, rows, H, eps, y8, q_scale, amax, rope, stream);
}

// Largest |x| of n bf16 values into *amax (float bits; the caller zeroes it first).
__global__ void amax_bf16_kernel(const bf16* __restrict__ x, size_t n8, unsigned* amax) {
  float mx = 0.f;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float f[8];
    unpack_bf16x8(ld_stream(reinterpret_cast<const uint4*>(x) + i), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(f[e]));
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) atomic_max_abs(amax, mx);
}

// Per-tensor current scaling: scale = 448 / amax (1 if amax is 0), codes of x * scale; slot[1]
// receives the dequantisation factor 1 / scale.
__global__ void quantize_e4m3_kernel(const bf16* __restrict__ x, size_t n8, uint8_t* __restrict__ q, float* slot) {
  const float amax = __uint_as_float(*reinterpret_cast<const unsigned*>(slot));
  const float scale = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) slot[1] = __frcp_rn(scale);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float f[8];
    unpack_bf16x8(ld_stream(reinterpret_cast<const uint4*>(x) + i), f);
    reinterpret_cast<uint2*>(q)[i] = pack_e4m3x8(f, scale);
  }
}

// Delayed scaling after a forward: append each activation's amax of this call to its history,
// clear it, and set scale = 448 / max(history) (1 while the history is all zero), deq = 1/scale.
// state: scale[4] | deq[4] | amax bits[4] | pad[4] | history[4][len].  One warp per tensor.
__global__ void fp8_history_kernel(float* state, int len, int pos) {
  const int t = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (t >= 4) return;
  unsigned* amax_bits = reinterpret_cast<unsigned*>(state + 8);
  float* hist = state + 16 + static_cast<size_t>(t) * len;
  if (lane == 0) {
    hist[pos] = __uint_as_float(amax_bits[t]);
    amax_bits[t] = 0u;
  }
  __syncwarp();
  float mx = 0.f;
  for (int i = lane; i < len; i += 32) mx = fmaxf(mx, hist[i]);
  mx = warp_max(mx);
  if (lane == 0) {
    const float scale = mx > 0.f ? __fdiv_rn(448.0f, mx) : 1.0f;
    state[t] = scale;
    state[4 + t] = __frcp_rn(scale);
  }
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

// Per-token RoPE position of packed samples: token t of sample i (cu[i] <= t < cu[i+1]) has
// position t - cu[i].  Inconsistent cu_seqlens are reported in *err and mapped to position 0, which
// keeps every later access in bounds.
__global__ void packed_index_kernel(const int* __restrict__ cu, int n, int T, int max_len, int* __restrict__ pos,
                                    int* err) {
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
  ok = ok && start <= t && t < end && p < max_len && start >= 0;
  if (!ok) atomicCAS(err, 0, 1);  // MT_ERR_INVALID_ARG
  pos[t] = ok ? p : 0;
}

}  // namespace

cudaError_t launch_norm(bool layer_norm, const bf16* x, const bf16* g, const bf16* b, bf16* y, int rows, int hidden,
                        float eps, cudaStream_t stream, uint8_t* y8, const float* q_scale, unsigned* amax,
                        const RopeRows* rope) {
  if (rows <= 0) return cudaSuccess;
  if (hidden <= 0 || hidden > 8192 || hidden % 8) return cudaErrorInvalidValue;
  const RopeRows rr = rope != nullptr ? *rope : RopeRows{};
  if (y8 != nullptr)
    return layer_norm ? launch_norm_ln<true, true>(x, g, b, y, rows, hidden, eps, y8, q_scale, amax, rr, stream)
                      : launch_norm_ln<false, true>(x, g, b, y, rows, hidden, eps, y8, q_scale, amax, rr, stream);
  return layer_norm ? launch_norm_ln<true, false>(x, g, b, y, rows, hidden, eps, y8, q_scale, amax, rr, stream)
                    : launch_norm_ln<false, false>(x, g, b, y, rows, hidden, eps, y8, q_scale, amax, rr, stream);
}

cudaError_t launch_quantize_e4m3(const bf16* x, size_t n, uint8_t* q, float* slot, cudaStream_t stream) {
  const size_t n8 = n / 8;
  cudaError_t e = cudaMemsetAsync(slot, 0, 2 * sizeof(float), stream);
  if (e != cudaSuccess || n8 == 0) return e;
  const int blocks = static_cast<int>(n8 / 256 + 1 < 4 * 152 ? n8 / 256 + 1 : 4 * 152);
  amax_bf16_kernel<<<blocks, 256, 0, stream>>>(x, n8, reinterpret_cast<unsigned*>(slot));
  quantize_e4m3_kernel<<<blocks, 256, 0, stream>>>(x, n8, q, slot);
  return cudaGetLastError();
}

cudaError_t launch_fp8_history(float* state, int len, int pos, cudaStream_t stream) {
  fp8_history_kernel<<<1, 128, 0, stream>>>(state, len, pos);
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

cudaError_t launch_packed_index(const int* cu, int num_seqs, int tokens, int max_seqlen, int* pos, int* err,
                                cudaStream_t stream) {
  if (tokens <= 0) return cudaSuccess;
  packed_index_kernel<<<(tokens + 255) / 256, 256, 0, stream>>>(cu, num_seqs, tokens, max_seqlen, pos, err);
  return cudaGetLastError();
}

}  // namespace mt
