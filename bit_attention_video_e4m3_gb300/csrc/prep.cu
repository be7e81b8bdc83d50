// Stage 1 kernels: FP8 preparation of post-RoPE bf16 Q, K, V.
//
// TeleFuser "FP8 Sol-Attn" blog, section "FP8 Preparation for attention":
// one scale per (batch, head, 64-token block) for Q and K, s = max|block|/448;
// V scaled per (batch, head, channel) over all tokens and stored
// token-contiguous so the PV product reads it K-major.
// VC-Attention news article, section 2 "V-Smooth": V rows gathered by a token
// permutation, each 128-row block mean removed (kept as a 16-bit vector) and
// only the residual quantised.
//
// Three launches, all bandwidth-bound:
//   prep_qk      one CTA per (64-token block, head, batch, Q|K): block amax,
//                fp32 scale, E4M3 codes (K rows gathered by the permutation)
//   prep_v_stats one CTA per (128-row V block, head, batch): exact block mean
//                (fp64 sum, one rounding to bf16), residual channel max folded
//                into a per-(batch, head, channel) maximum with atomicMax
//   prep_v_quant same grid: residual codes with the final channel scale,
//                written transposed ([channel][token]) for the PV operand
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace fp8attn {

namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two fp32 values -> two E4M3 codes (RNE, satfinite), x.lo in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Correctly rounded fp64 -> bf16 (nearest even): truncate to fp32, mark any
// discarded bits in the lowest fp32 bit (round-to-odd), then round the fp32 to
// bf16.  Round-to-odd at 24 bits followed by rounding at 8 bits is exact.
__device__ __forceinline__ uint16_t f64_to_bf16_rne(double d) {
  float f = __double2float_rz(d);
  uint32_t bits = __float_as_uint(f);
  if (static_cast<double>(f) != d) bits |= 1u;
  __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(bits));
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// Q/K: grid (nQK, H, 2B); 128 threads.  Thread t covers 16-byte chunk (t & 15)
// of rows (t >> 4) + 8 i, i = 0..7, of the 64-row block.
__global__ void __launch_bounds__(128) prep_qk_kernel(const PrepParams p) {
  const int blk = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z >> 1, is_k = blockIdx.z & 1;
  const __nv_bfloat16* src = is_k ? p.k : p.q;
  uint8_t* dst = is_k ? p.k8 : p.q8;
  float* scales = is_k ? p.k_scale : p.q_scale;
  const int tid = threadIdx.x, chunk = tid & 15, rsub = tid >> 4;
  const int bh = b * p.H + h;

  uint4 vals[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = blk * kQKBlock + rsub + 8 * i;
    vals[i] = make_uint4(0, 0, 0, 0);
    if (t < p.T) {
      const int srow = (is_k && p.perm) ? __ldg(p.perm + (size_t)bh * p.T + t) : t;
      const uint4* ptr = reinterpret_cast<const uint4*>(
          src + (((size_t)b * p.T + srow) * p.H + h) * kHeadDim + chunk * 8);
      vals[i] = __ldg(ptr);
      const uint32_t w[4] = {vals[i].x, vals[i].y, vals[i].z, vals[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[e] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[e] >> 16)));
      }
    }
  }
  __shared__ float red[4];
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  const float a = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float inv = a > 0.f ? __fdiv_rn(kE4M3Max, a) : 0.f;
  if (tid == 0) scales[(size_t)bh * p.nQK + blk] = __fdiv_rn(a, kE4M3Max);

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = blk * kQKBlock + rsub + 8 * i;
    if (t < p.T) {
      const uint32_t w[4] = {vals[i].x, vals[i].y, vals[i].z, vals[i].w};
      uint32_t o[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float x0 = __fmul_rn(bf16_bits_to_float(w[2 * e] & 0xFFFFu), inv);
        const float x1 = __fmul_rn(bf16_bits_to_float(w[2 * e] >> 16), inv);
        const float x2 = __fmul_rn(bf16_bits_to_float(w[2 * e + 1] & 0xFFFFu), inv);
        const float x3 = __fmul_rn(bf16_bits_to_float(w[2 * e + 1] >> 16), inv);
        o[e] = static_cast<uint32_t>(e4m3x2(x0, x1)) | (static_cast<uint32_t>(e4m3x2(x2, x3)) << 16);
      }
      *reinterpret_cast<uint2*>(dst + (((size_t)b * p.T + t) * p.H + h) * kHeadDim + chunk * 8) =
          make_uint2(o[0], o[1]);
    }
  }
}

// ---------------------------------------------------------------------------
// V pass 1: grid (nV, H, B); 256 threads.  Thread t owns channel c = t & 127
// and rows 64 * (t >> 7) .. +63 of the 128-row block.
__global__ void __launch_bounds__(256) prep_v_stats_kernel(const PrepParams p) {
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
  const int t0 = j * kVBlock;
  const int cnt = min(kVBlock, p.T - t0);
  const uint16_t* v = reinterpret_cast<const uint16_t*>(p.v);

  float x[64];
  double sum = 0.0;
#pragma unroll
  for (int r = 0; r < 64; ++r) {
    const int rr = half * 64 + r;
    x[r] = 0.f;
    if (rr < cnt) {
      const int t = t0 + rr;
      const int srow = p.perm ? __ldg(p.perm + (size_t)bh * p.T + t) : t;
      x[r] = bf16_bits_to_float(__ldg(v + (((size_t)b * p.T + srow) * p.H + h) * kHeadDim + c));
      sum += static_cast<double>(x[r]);
    }
  }
  __shared__ double part[2][128];
  __shared__ float pmax[2][128];
  float mu = 0.f;
  uint16_t mu_bits = 0;
  if (p.vsmooth) {
    part[half][c] = sum;
    __syncthreads();
    const double total = part[0][c] + part[1][c];
    mu_bits = f64_to_bf16_rne(total / static_cast<double>(cnt));
    mu = bf16_bits_to_float(mu_bits);
  }
  if (half == 0)
    reinterpret_cast<uint16_t*>(p.v_mean)[((size_t)bh * p.nV + j) * kHeadDim + c] = mu_bits;
  float rmax = 0.f;
#pragma unroll
  for (int r = 0; r < 64; ++r)
    if (half * 64 + r < cnt) rmax = fmaxf(rmax, fabsf(__fsub_rn(x[r], mu)));
  pmax[half][c] = rmax;
  __syncthreads();
  if (half == 0) {
    const float m = fmaxf(pmax[0][c], pmax[1][c]);
    atomicMax(p.v_amax + (size_t)bh * kHeadDim + c, __float_as_uint(m));
  }
}

// ---------------------------------------------------------------------------
// V pass 2: same grid and thread mapping; writes 64 consecutive token codes of
// channel c per thread (token-contiguous layout) and, from block 0, the scale.
__global__ void __launch_bounds__(256) prep_v_quant_kernel(const PrepParams p) {
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
  const int t0 = j * kVBlock;
  const int cnt = min(kVBlock, p.T - t0);
  const uint16_t* v = reinterpret_cast<const uint16_t*>(p.v);

  const float mu = p.vsmooth ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(
                                   p.v_mean)[((size_t)bh * p.nV + j) * kHeadDim + c])
                             : 0.f;
  const float amax = __uint_as_float(p.v_amax[(size_t)bh * kHeadDim + c]);
  const float inv = amax > 0.f ? __fdiv_rn(kE4M3Max, amax) : 0.f;
  if (j == 0 && half == 0) p.v_scale[(size_t)bh * kHeadDim + c] = __fdiv_rn(amax, kE4M3Max);

  uint32_t words[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int rr = half * 64 + 4 * q + e;
      y[e] = 0.f;
      if (rr < cnt) {
        const int t = t0 + rr;
        const int srow = p.perm ? __ldg(p.perm + (size_t)bh * p.T + t) : t;
        const float xv =
            bf16_bits_to_float(__ldg(v + (((size_t)b * p.T + srow) * p.H + h) * kHeadDim + c));
        y[e] = __fmul_rn(__fsub_rn(xv, mu), inv);
      }
    }
    uint32_t w = static_cast<uint32_t>(e4m3x2(y[0], y[1])) |
                 (static_cast<uint32_t>(e4m3x2(y[2], y[3])) << 16);
    // pad tokens (rr >= cnt) must be code 0; +-0 inputs already give 0x00/0x80,
    // so clear them explicitly.
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (half * 64 + 4 * q + e >= cnt) w &= ~(0xFFu << (8 * e));
    words[q] = w;
  }
  uint4* out = reinterpret_cast<uint4*>(p.v8 + ((size_t)bh * kHeadDim + c) * p.Tpad + t0 + half * 64);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    out[q] = make_uint4(words[4 * q], words[4 * q + 1], words[4 * q + 2], words[4 * q + 3]);
}

}  // namespace

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  prep_qk_kernel<<<dim3(p.nQK, p.H, 2 * p.B), 128, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prep_v_stats_kernel<<<dim3(p.nV, p.H, p.B), 256, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prep_v_quant_kernel<<<dim3(p.nV, p.H, p.B), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8attn
