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
// Three launches, all HBM-bound.  Each warp loads its 16 token rows (lane l:
// the 8 bytes of channels 4l .. 4l+3 of each row, so one warp instruction reads
// one 256-byte row; rows gathered through the permutation where there is one)
// straight into registers, all 16 loads in flight at once, and computes from
// there; shared memory holds only the cross-warp reductions:
//   prep_qk      one CTA per (64-token block, head, batch, Q|K): block amax,
//                fp32 scale, E4M3 codes (K rows gathered by the permutation)
//   prep_v_stats one CTA per (128-row V block, head, batch): exact block mean
//                (fixed-point integer sum, one rounding to bf16), residual
//                channel max folded into a per-(batch, head, channel) maximum
//                with atomicMax
//   prep_v_quant same grid: residual codes with the final channel scale,
//                transposed through shared memory to [channel][token] rows
//                for the PV operand
// With sequence-mean smoothing (TeleFuser blog, section "Diffusion precision
// guards") three more launches come first, over K (and V) in token order:
//   prep_seq_max      per (b, h, channel) max|x| over T
//   prep_seq_sum      exact fixed-point sums anchored at that maximum
//   prep_seq_finalize the exact mean rounded once to fp32
// and prep_offset writes the output offset mean_T(V) - bias at the end.
#include <algorithm>
#include <type_traits>

#include <cuda_fp8.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8attn {

namespace {

constexpr float kE4M3Max = 448.0f;
constexpr float kFp4Top = 2688.0f;      // 6 x 448: NVFP4 two-level range
constexpr uint32_t kRowBytes = kHeadDim * 2;     // one bf16 token row

// dynamic shared memory of the V kernels (offsets from the 128-byte aligned base)
constexpr uint32_t kVRed = 0;                                  // float [8][128]
constexpr uint32_t kVSum = kVRed + 8 * 128 * 4;                // int64 [8][128]
constexpr uint32_t kVLow = kVSum + 8 * 128 * 8;                // float [8][128]
constexpr uint32_t kVTile = kVRed;                             // quant: codes [128][128], aliases the reductions
constexpr uint32_t kVBias = kVLow + 8 * 128 * 4;               // quant: float [8][128] bias partials
constexpr uint32_t kVSmem = kVBias + 8 * 128 * 4 + 128;        // + alignment slack

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
  return __uint_as_float((b & 0xFFFFu) << 16);
}

// Two fp32 values -> two E4M3 codes (RNE, satfinite), x.lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3)));
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

// The bf16 value nearest to a * 2^e (ties to even) for an integer |a| < 2^53,
// without fp64 arithmetic: a rounded to 24 bits toward zero, the lowest bit set
// when anything was dropped (rounding to odd), the exponent moved by e, then
// one rounding to bf16; rounding to odd with two or more spare bits followed
// by rounding to nearest gives the correctly rounded result.  False when the
// result would leave the normal fp32 range (the caller takes the fp64 route).
__device__ __forceinline__ bool ll_pow2_to_bf16(long long a, int e, uint16_t& out) {
  if (a == 0) {
    out = 0;
    return true;
  }
  const float f = __ll2float_rz(a);
  uint32_t bits = __float_as_uint(f);
  if (__float2ll_rz(f) != a) bits |= 1u;
  const int ef = static_cast<int>((bits >> 23) & 0xFFu) + e;
  if (ef < 1 || ef > 254) return false;
  bits = (bits & 0x807FFFFFu) | (static_cast<uint32_t>(ef) << 23);
  const __nv_bfloat16 hb = __float2bfloat16_rn(__uint_as_float(bits));
  out = *reinterpret_cast<const uint16_t*>(&hb);
  return true;
}

// Per-halfword operations on two bf16 values in one word (exact): signed
// maximum and minimum, and the unsigned maximum of 16-bit halves (the
// unsigned minimum is min_u16x2).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 2^sh as two exact fp32 factors (sh can exceed the fp32 exponent range)
__device__ __forceinline__ void pow2_pair(int sh, float& f1, float& f2) {
  const int sh1 = max(min(sh, 100), -100);
  f1 = ldexpf(1.f, sh1);
  f2 = ldexpf(1.f, sh - sh1);
}

// Exact accumulation of an integer y = x * 2^k with |y| < 2^45 in two int32
// halves, without a 64-bit conversion: t = y + 1.5*2^46 stays in one binade
// (ulp 2^23), so bits(t) - bits(1.5*2^46) is y rounded to a multiple of 2^23,
// counted in those multiples; r = y - (t - 1.5*2^46) is exact with |r| <= 2^22
// and r + 1.5*2^23 (ulp 1) carries r the same way.  y = hi * 2^23 + lo.
// kPre: the scale 2^k is applied as two exact factors (k > 127).
template <bool kPre>
__device__ __forceinline__ void split_add(float x, float up1, float up2, int& hi, int& lo) {
  constexpr float kC1 = 105553116266496.f;   // 1.5 * 2^46
  constexpr float kC0 = 12582912.f;          // 1.5 * 2^23
  const float xs = kPre ? x * up1 : x;
  const float t = __fmaf_rn(xs, up2, kC1);
  const float h = __fsub_rn(t, kC1);
  const float r = __fmaf_rn(xs, up2, -h);
  hi += static_cast<int>(__float_as_uint(t) - 0x56C00000u);
  lo += static_cast<int>(__float_as_uint(__fadd_rn(r, kC0)) - 0x4B400000u);
}

// Window scale 2^sh for split_add: up2 alone when sh fits fp32, else up1*up2.
__device__ __forceinline__ bool split_scale(int sh, float& up1, float& up2) {
  if (sh <= 127) {
    up1 = 1.f;
    up2 = ldexpf(1.f, sh);
    return false;
  }
  up1 = ldexpf(1.f, sh - 127);
  up2 = ldexpf(1.f, 127);
  return true;
}

// Exponent E of a positive fp32 value (2^E <= m < 2^(E+1)); 0 for m == 0.
__device__ __forceinline__ int exp_of(float m) {
  return m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127 : 0;
}

// The fp32 value nearest to S * 2^lsb_exp / T (ties to even), from exact
// integer arithmetic: 128-bit quotient and remainder give the kept bits, the
// round bit and the sticky bit.  Normal range.
__device__ float exact_mean_f32(long long S, int lsb_exp, int T) {
  if (S == 0) return 0.f;
  const bool neg = S < 0;
  const unsigned long long a = neg ? static_cast<unsigned long long>(-(S + 1)) + 1ull
                                   : static_cast<unsigned long long>(S);
  const unsigned __int128 n = static_cast<unsigned __int128>(a) << 64;
  const unsigned __int128 q = n / static_cast<unsigned>(T);
  const bool rem = (n % static_cast<unsigned>(T)) != 0;
  const unsigned long long qh = static_cast<unsigned long long>(q >> 64);
  const int msb = qh ? 127 - __clzll(qh) : 63 - __clzll(static_cast<unsigned long long>(q));
  int s = msb - 23;                     // q >= 2^64 / T, so s > 0 for T < 2^40
  unsigned long long mant = static_cast<unsigned long long>(q >> s);
  const unsigned __int128 low = q & ((static_cast<unsigned __int128>(1) << s) - 1);
  const unsigned __int128 half = static_cast<unsigned __int128>(1) << (s - 1);
  if (low > half || (low == half && (rem || (mant & 1ull)))) {
    if (++mant == (1ull << 24)) {
      mant >>= 1;
      ++s;
    }
  }
  const float r = ldexpf(static_cast<float>(mant), s + lsb_exp - 64);
  return neg ? -r : r;
}


// The 16 rows r0 .. r0 + 15 of (b, h) handled by the calling warp: u[r] = lane
// l's 8 bytes (bf16 channels 4l .. 4l+3) of row r0 + r, read from token
// perm[r0 + r] when a permutation is given, zero for rows at or past r0 + nr.
// A permutation entry outside [0, T) reads token 0 (no access leaves the
// tensor) and is reported in the status word.  Lanes 0..15 fetch the
// permutation entries and broadcast them; the 16 row loads are independent.
__device__ __forceinline__ void load_rows16(const PrepParams& p, const __nv_bfloat16* src, const int32_t* perm,
                                            int b, int h, int bh, int r0, int nr, uint2 (&u)[16]) {
  const int l = threadIdx.x & 31;
  int tok = r0 + (l & 15);
  if (perm && l < nr && l < 16) {
    tok = __ldg(perm + (size_t)bh * p.T + r0 + l);
    if (static_cast<unsigned>(tok) >= static_cast<unsigned>(p.T)) {
      if (p.status) atomicExch(p.status, kStatusBadPerm);
      tok = 0;
    }
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int srow = __shfl_sync(0xffffffffu, tok, r);
    u[r] = r < nr ? __ldg(reinterpret_cast<const uint2*>(src + (((size_t)b * p.T + srow) * p.H + h) * kHeadDim) + l)
                  : make_uint2(0u, 0u);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Q/K: grid (nQK, H, 2B); 128 threads.  Warp w covers rows 16 w .. 16 w + 15 of
// the 64-row block, lane l channels 4 l .. 4 l + 3 (8 bytes of each row).
__global__ void __launch_bounds__(128) prep_qk_kernel(const PrepParams p) {
  const int blk = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z >> 1, is_k = blockIdx.z & 1;
  const __nv_bfloat16* src = is_k ? p.k : p.q;
  uint8_t* dst = is_k ? p.k8 : p.q8;
  float* scales = is_k ? p.k_scale : p.q_scale;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int bh = b * p.H + h;
  const int t0 = blk * kQKBlock;
  const int nrows = min(kQKBlock, p.T - t0);
  __shared__ float red[4];
  const int nr = min(16, max(0, nrows - 16 * w));  // valid rows of this warp
  uint2 u[16];
  load_rows16(p, src, is_k ? p.perm : nullptr, b, h, bh, t0 + 16 * w, nr, u);
  // sequence-mean smoothing of K: x' = fl32(x - mean_T), the block scale and
  // the codes come from the centred values
  float cen[4] = {0.f, 0.f, 0.f, 0.f};
  if (is_k && p.smooth >= 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) cen[k] = p.chan_mean[(size_t)bh * kHeadDim + 4 * l + k];
  }
  auto row4 = [&](int r, float (&x)[4]) {
    x[0] = __fsub_rn(bf16_bits_to_float(u[r].x), cen[0]);
    x[1] = __fsub_rn(bf16_bits_to_float(u[r].x >> 16), cen[1]);
    x[2] = __fsub_rn(bf16_bits_to_float(u[r].y), cen[2]);
    x[3] = __fsub_rn(bf16_bits_to_float(u[r].y >> 16), cen[3]);
  };

  const bool centred = is_k && p.smooth >= 1;
  float amax = 0.f;
  if (!centred) {
    // bf16 magnitudes compare as their 16-bit patterns: two per operation
    uint32_t am = 0u;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < nr) am = max_u16x2(am, max_u16x2(u[r].x & 0x7FFF7FFFu, u[r].y & 0x7FFF7FFFu));
    amax = fmaxf(bf16_bits_to_float(am), bf16_bits_to_float(am >> 16));
  } else {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r < nr) {
        float x[4];
        row4(r, x);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
      }
    }
  }
  amax = warp_max(amax);
  if (l == 0) red[w] = amax;
  __syncthreads();
  const float a = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float inv = a > 0.f ? __fdiv_rn(kE4M3Max, a) : 0.f;
  if (threadIdx.x == 0) scales[(size_t)bh * p.nQK + blk] = __fdiv_rn(a, kE4M3Max);

  const float2 inv2 = make_float2(inv, inv);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if (r < nr) {
      const int rr = 16 * w + r;
      float x[4];
      if (centred) {
        row4(r, x);
      } else {
        x[0] = bf16_bits_to_float(u[r].x);
        x[1] = bf16_bits_to_float(u[r].x >> 16);
        x[2] = bf16_bits_to_float(u[r].y);
        x[3] = bf16_bits_to_float(u[r].y >> 16);
      }
      // codes of x * (448 / a), two channels per f32x2 product
      const float2 qa = __fmul2_rn(make_float2(x[0], x[1]), inv2);
      const float2 qb = __fmul2_rn(make_float2(x[2], x[3]), inv2);
      const uint32_t code = e4m3x2(qa.x, qa.y) | (e4m3x2(qb.x, qb.y) << 16);
      *reinterpret_cast<uint32_t*>(dst + (((size_t)b * p.T + t0 + rr) * p.H + h) * kHeadDim + 4 * l) = code;
    }
  }
}

// ---------------------------------------------------------------------------
// V kernels: grid (nV, H, B); 256 threads.  Warp w covers rows 16 w .. 16 w + 15
// of the 128-row block, lane l channels 4 l .. 4 l + 3; rows past T are skipped.

// V pass 1: block means (V-Smooth only) and the residual channel maxima.
//
// Exact block mean without per-element fp64 arithmetic: each channel's values
// are summed as integers in a fixed-point window anchored at the block
// maximum.  With 2^E <= max|x| < 2^(E+1), a bf16 value of exponent e >= E - 37
// is an integer multiple of 2^(E-44) below 2^45 (added as two exact int32
// halves by split_add), and 128 of them sum below 2^53, so the int64 sum is
// exact and converts to fp64 exactly; the mean is then rounded once to bf16.
// Centred fp32 values (24-bit significands, sequence-mean smoothing) use a
// 31-binade window in units of 2^(E-54).  Values below the window are added
// separately in fp32 and make the result merely close.
//
// The block (in registers) is read once for the statistics: per channel the signed
// maximum and minimum and the smallest magnitude.  The residual maximum needs
// no further read: x -> fl(x - mu) is monotonic, so max_t |fl(x_t - mu)| =
// max(|fl(x_max - mu)|, |fl(x_min - mu)|).  When no value of a warp's channels
// lies below its window (the smallest magnitude tells), the sum skips the
// per-value window test and runs on packed f32x2 arithmetic.
__global__ void __launch_bounds__(256, 4) prep_v_stats_kernel(const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~static_cast<uintptr_t>(127));
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int t0 = j * kVBlock;
  const int cnt = min(kVBlock, p.T - t0);
  const int nr = min(16, max(0, cnt - 16 * w));    // valid rows of this warp
  uint2 u[16];
  load_rows16(p, p.v, p.perm, b, h, bh, t0 + 16 * w, nr, u);
  float (*s_red)[128] = reinterpret_cast<float (*)[128]>(sm + kVRed);
  long long (*s_sum)[128] = reinterpret_cast<long long (*)[128]>(sm + kVSum);
  float (*s_low)[128] = reinterpret_cast<float (*)[128]>(sm + kVLow);
  // statistics of the read: per warp the signed max (s_red), signed min and
  // smallest magnitude (in the sum area, free until the sums); per channel the
  // block maximum magnitude and smallest magnitude (in the bias area, used only
  // by the quantisation kernel)
  float (*s_min)[128] = reinterpret_cast<float (*)[128]>(sm + kVSum);
  float (*s_amin)[128] = reinterpret_cast<float (*)[128]>(sm + kVSum + 8 * 128 * 4);
  float* s_bmax = reinterpret_cast<float*>(sm + kVBias);
  float* s_bmin = s_bmax + 128;

  // sequence-mean smoothing of V: V' = fl32(V - mean_T)
  const bool centred = p.smooth == 2;
  float cen[4] = {0.f, 0.f, 0.f, 0.f};
  if (centred) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      cen[k] = p.chan_mean[((size_t)p.B * p.H + bh) * kHeadDim + 4 * l + k];
  }
  auto row4 = [&](int r, float (&x)[4]) {
    x[0] = __fsub_rn(bf16_bits_to_float(u[r].x), cen[0]);
    x[1] = __fsub_rn(bf16_bits_to_float(u[r].x >> 16), cen[1]);
    x[2] = __fsub_rn(bf16_bits_to_float(u[r].y), cen[2]);
    x[3] = __fsub_rn(bf16_bits_to_float(u[r].y >> 16), cen[3]);
  };

  // ---- statistics over the valid rows
  float xmax[4], xmin[4], amin[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    xmax[k] = -INFINITY;
    xmin[k] = INFINITY;
    amin[k] = INFINITY;
  }
  if (!centred) {
    // bf16 values: two channels per operation on the packed words (the same
    // maxima and minima as on their fp32 values), the smallest magnitude as
    // the unsigned minimum of the magnitude bits
    if (nr > 0) {
      uint32_t mx0 = u[0].x, mx1 = u[0].y, mn0 = u[0].x, mn1 = u[0].y;
      uint32_t am0 = u[0].x & 0x7FFF7FFFu, am1 = u[0].y & 0x7FFF7FFFu;
#pragma unroll
      for (int r = 1; r < 16; ++r) {
        if (r >= nr) break;
        mx0 = max_bf16x2(mx0, u[r].x);
        mx1 = max_bf16x2(mx1, u[r].y);
        mn0 = min_bf16x2(mn0, u[r].x);
        mn1 = min_bf16x2(mn1, u[r].y);
        am0 = min_u16x2(am0, u[r].x & 0x7FFF7FFFu);
        am1 = min_u16x2(am1, u[r].y & 0x7FFF7FFFu);
      }
      const uint32_t mx[4] = {mx0, mx0 >> 16, mx1, mx1 >> 16}, mn[4] = {mn0, mn0 >> 16, mn1, mn1 >> 16};
      const uint32_t am[4] = {am0, am0 >> 16, am1, am1 >> 16};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xmax[k] = bf16_bits_to_float(mx[k]);
        xmin[k] = bf16_bits_to_float(mn[k]);
        amin[k] = bf16_bits_to_float(am[k]);
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r >= nr) break;
      float x[4];
      row4(r, x);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xmax[k] = fmaxf(xmax[k], x[k]);
        xmin[k] = fminf(xmin[k], x[k]);
        amin[k] = fminf(amin[k], fabsf(x[k]));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    s_red[w][4 * l + k] = xmax[k];
    s_min[w][4 * l + k] = xmin[k];
    s_amin[w][4 * l + k] = amin[k];
  }
  __syncthreads();
  // thread c < 128 owns channel c: the block's signed max / min (kept for the
  // residual maximum) and, for everyone, its maximum and smallest magnitude
  float cmax = -INFINITY, cmin = INFINITY;
  if (threadIdx.x < 128) {
    const int c = threadIdx.x;
    float am = INFINITY;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      cmax = fmaxf(cmax, s_red[ww][c]);
      cmin = fminf(cmin, s_min[ww][c]);
      am = fminf(am, s_amin[ww][c]);
    }
    s_bmax[c] = fmaxf(fabsf(cmax), fabsf(cmin));
    s_bmin[c] = am;
  }
  __syncthreads();                                  // the sum area is reused below

  float mu_c = 0.f;      // block mean of channel threadIdx.x (< 128)
  if (p.vsmooth) {
    // fixed-point window of the block sums: bf16 values (8-bit significands)
    // are exact multiples of 2^(E-44) within 37 binades of the block maximum
    // (integers below 2^45, summed by split_add), centred fp32 values (24-bit)
    // exact multiples of 2^(E-54) within 31 binades (int64 conversion)
    const int wlsb = centred ? 54 : 44, wspan = centred ? 31 : 37;
    int E[4];
    float up1[4], up2[4], floor_mag[4];
    bool inside = true;        // every value of this thread's channels lies in its window
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float m = s_bmax[4 * l + k];
      // anchor exponent E of the block maximum (the window is empty if m == 0)
      E[k] = m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127 : 0;
      // 2^(wlsb-E) as two exact factors (the shift reaches 187 for
      // subnormal blocks); every in-window product is an integer below 2^55
      pow2_pair(wlsb - E[k], up1[k], up2[k]);
      floor_mag[k] = ldexpf(1.f, E[k] - wspan);
      inside = inside && s_bmin[4 * l + k] >= floor_mag[k];
    }
    long long acc[4] = {0, 0, 0, 0};
    float low[4] = {0.f, 0.f, 0.f, 0.f};
    if (centred) {
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r >= nr) break;
        float x[4];
        row4(r, x);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (fabsf(x[k]) >= floor_mag[k]) acc[k] += __float2ll_rn((x[k] * up1[k]) * up2[k]);
          else low[k] += x[k];
        }
      }
    } else {
      float s1[4], s2[4];
      bool pre = false;
#pragma unroll
      for (int k = 0; k < 4; ++k) pre |= split_scale(wlsb - E[k], s1[k], s2[k]);
      int hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};   // 16 rows: |hi|, |lo| < 2^27
      if (__all_sync(0xffffffffu, inside && !pre)) {
        // every value is inside its window, so each split is exact without a
        // test (split_add, two channels per packed operation); the raw bit
        // patterns are summed and the constant offsets removed afterwards.
        // The zero rows past the block's end add exactly those offsets.
        constexpr float kC1 = 105553116266496.f;   // 1.5 * 2^46
        constexpr float kC0 = 12582912.f;          // 1.5 * 2^23
        const float2 c1 = make_float2(kC1, kC1), c0 = make_float2(kC0, kC0), mc1 = make_float2(-kC1, -kC1);
        const float2 sa = make_float2(s2[0], s2[1]), sb = make_float2(s2[2], s2[3]);
        unsigned th[4] = {0u, 0u, 0u, 0u}, tq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float2 xa = make_float2(bf16_bits_to_float(u[r].x), bf16_bits_to_float(u[r].x >> 16));
          const float2 xb = make_float2(bf16_bits_to_float(u[r].y), bf16_bits_to_float(u[r].y >> 16));
          const float2 ta = __ffma2_rn(xa, sa, c1), tb = __ffma2_rn(xb, sb, c1);
          const float2 ha = __fadd2_rn(ta, mc1), hb = __fadd2_rn(tb, mc1);
          const float2 ra = __ffma2_rn(xa, sa, make_float2(-ha.x, -ha.y));
          const float2 rb = __ffma2_rn(xb, sb, make_float2(-hb.x, -hb.y));
          const float2 qa = __fadd2_rn(ra, c0), qb = __fadd2_rn(rb, c0);
          th[0] += __float_as_uint(ta.x);
          th[1] += __float_as_uint(ta.y);
          th[2] += __float_as_uint(tb.x);
          th[3] += __float_as_uint(tb.y);
          tq[0] += __float_as_uint(qa.x);
          tq[1] += __float_as_uint(qa.y);
          tq[2] += __float_as_uint(qb.x);
          tq[3] += __float_as_uint(qb.y);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          hi[k] = static_cast<int>(th[k] - 16u * 0x56C00000u);
          lo[k] = static_cast<int>(tq[k] - 16u * 0x4B400000u);
        }
      } else {
        auto rows = [&](auto pre_tag) {
          constexpr bool kPre = decltype(pre_tag)::value;
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            if (r >= nr) break;
            float x[4];
            row4(r, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              int dl = 0;   // below the window t == 1.5*2^46: hi gains 0
              split_add<kPre>(x[k], s1[k], s2[k], hi[k], dl);
              if (fabsf(x[k]) >= floor_mag[k]) lo[k] += dl;
              else low[k] += x[k];
            }
          }
        };
        if (pre) rows(std::true_type{});
        else rows(std::false_type{});
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = (static_cast<long long>(hi[k]) << 23) + lo[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s_sum[w][4 * l + k] = acc[k];
      s_low[w][4 * l + k] = low[k];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
      const int c = threadIdx.x;
      long long a = s_sum[0][c];
      float lo = s_low[0][c];
#pragma unroll
      for (int ww = 1; ww < 8; ++ww) {
        a += s_sum[ww][c];
        lo += s_low[ww][c];
      }
      const float m = s_bmax[c];
      const int Ec = m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127 : 0;
      // a full block (cnt a power of two) with nothing below the window is an
      // exact integer times a power of two; otherwise the fp64 quotient
      uint16_t mu_bits;
      const bool pow2_cnt = (cnt & (cnt - 1)) == 0;
      if (!(lo == 0.f && pow2_cnt && ll_pow2_to_bf16(a, Ec - wlsb - (__ffs(cnt) - 1), mu_bits))) {
        const double total = ldexp(static_cast<double>(a), Ec - wlsb) + static_cast<double>(lo);
        mu_bits = f64_to_bf16_rne(total / static_cast<double>(cnt));
      }
      reinterpret_cast<uint16_t*>(p.v_mean)[((size_t)bh * p.nV + j) * kHeadDim + c] = mu_bits;
      mu_c = bf16_bits_to_float(mu_bits);
    }
  } else if (threadIdx.x < 128) {
    reinterpret_cast<uint16_t*>(p.v_mean)[((size_t)bh * p.nV + j) * kHeadDim + threadIdx.x] = 0;
  }

  // residual channel maximum: the ends of the monotonic map x -> fl(x - mu)
  if (threadIdx.x < 128) {
    // (the atomic only when it can raise the current value: the maxima of one
    // head settle after a few blocks)
    const float rm = fmaxf(fabsf(__fsub_rn(cmax, mu_c)), fabsf(__fsub_rn(cmin, mu_c)));
    uint32_t* dst = p.v_amax + (size_t)bh * kHeadDim + threadIdx.x;
    if (__float_as_uint(rm) > __ldcg(dst)) atomicMax(dst, __float_as_uint(rm));
  }
}

// ---------------------------------------------------------------------------
// V pass 2: residual codes with the final channel scale.  The 128 x 128 code
// block is transposed through shared memory (16-byte chunks, XOR-swizzled so
// both the scattered writes and the row reads are conflict-free) and leaves as
// 128-byte token rows per channel: the token-contiguous PV operand layout.
// NVFP4 residual of one 16-token block of one channel (thread-local): channel
// scales s_c = amax/2688, G = 2688/amax; block scale UE4M3(fl32(a G) * fl32(1/6));
// codes E2M1(R * fl32(G / sf)); returns the scale code and the 8 code bytes.
__device__ __forceinline__ uint32_t fp4_block(const float (&r)[16], float G, uint32_t (&packed)[2]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(r[i]));
  const float sfin = __fmul_rn(__fmul_rn(a, G), __uint_as_float(0x3E2AAAABu));   // fl32(1/6)
  const uint32_t sf = e4m3x2(sfin, 0.f) & 0xFFu;
  const float sfv = ue4m3_value(sf);
  const float rs = sfv > 0.f ? __fdiv_rn(G, sfv) : 0.f;
  packed[0] = packed[1] = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    packed[i >> 2] |= e2m1x2(__fmul_rn(r[2 * i], rs), __fmul_rn(r[2 * i + 1], rs)) << (8 * (i & 3));
  return sf;
}

template <bool FP4>
__global__ void __launch_bounds__(256, FP4 ? 3 : 4) prep_v_quant_kernel(const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~static_cast<uintptr_t>(127));
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int t0 = j * kVBlock;
  const int cnt = min(kVBlock, p.T - t0);
  const int nr = min(16, max(0, cnt - 16 * w));    // valid rows of this warp
  uint2 u[16];
  load_rows16(p, p.v, p.perm, b, h, bh, t0 + 16 * w, nr, u);
  uint4* tile = reinterpret_cast<uint4*>(sm + kVTile);   // [channel][16-token chunk ^ ((channel >> 2) & 7)]

  float mu[4], inv[4], sv[4], cen[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = 4 * l + k;
    cen[k] = p.smooth == 2 ? p.chan_mean[((size_t)p.B * p.H + bh) * kHeadDim + c] : 0.f;
    mu[k] = p.vsmooth ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(
                            p.v_mean)[((size_t)bh * p.nV + j) * kHeadDim + c])
                      : 0.f;
    const float amax = __uint_as_float(p.v_amax[(size_t)bh * kHeadDim + c]);
    const float top = FP4 ? kFp4Top : kE4M3Max;
    inv[k] = amax > 0.f ? __fdiv_rn(top, amax) : 0.f;
    sv[k] = __fdiv_rn(amax, top);
    if (j == 0 && w == 0) p.v_scale[(size_t)bh * kHeadDim + c] = sv[k];
  }
  float bias[4] = {0.f, 0.f, 0.f, 0.f};     // sum of (dequantised - exact) residuals

  if constexpr (FP4) {
    // warp w owns tokens 16w..16w+15 of the block: one 16-token scale block per channel
    uint2* tile4 = reinterpret_cast<uint2*>(sm + kVTile);        // [channel][8-byte slot ^ ((channel >> 2) & 7)]
    uint8_t* sft = sm + kVTile + 8192;                            // scale tile, tcgen05.cp order
    float res[4][16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      const bool ok = rr < nr;
      const float x[4] = {bf16_bits_to_float(u[rr].x), bf16_bits_to_float(u[rr].x >> 16),
                          bf16_bits_to_float(u[rr].y), bf16_bits_to_float(u[rr].y >> 16)};
#pragma unroll
      for (int k = 0; k < 4; ++k) res[k][rr] = ok ? __fsub_rn(__fsub_rn(x[k], cen[k]), mu[k]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = 4 * l + k;
      uint32_t packed[2];
      const uint32_t sf = fp4_block(res[k], inv[k], packed);
      tile4[c * 8 + (w ^ (l & 7))] = make_uint2(packed[0], packed[1]);
      // scale byte of (channel c, token block w): MMA k-step w / 4, byte w % 4 of
      // row c % 32, word c / 32 of that k-step's 32 x 16-byte block
      sft[(w >> 2) * 512 + (c & 31) * 16 + (c >> 5) * 4 + (w & 3)] = static_cast<uint8_t>(sf);
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int idx = threadIdx.x + 256 * it;                     // 128 channels x 4 chunks of 16 B
      const int c = idx >> 2, q = idx & 3, f = (c >> 2) & 7;
      const uint2 lo = tile4[c * 8 + ((2 * q) ^ f)], hi = tile4[c * 8 + ((2 * q + 1) ^ f)];
      *reinterpret_cast<uint4*>(p.v4 + ((size_t)bh * kHeadDim + c) * (p.Tpad / 2) + t0 / 2 + 16 * q) =
          make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    if (threadIdx.x < 64)
      reinterpret_cast<uint4*>(p.v4_sf + ((size_t)bh * p.nV + j) * 1024)[threadIdx.x] =
          reinterpret_cast<const uint4*>(sft)[threadIdx.x];
    return;
  } else {

  const bool centred = p.smooth == 2;
  uint32_t words[4][4];     // [channel k][4-token group]
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t b0[4] = {0u, 0u, 0u, 0u}, b1[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int rr = 4 * q + e;                    // row of this warp; rows >= nr are zero in u
      const uint2 u0 = u[rr], u1 = u[rr + 1];
      const float x0[4] = {bf16_bits_to_float(u0.x), bf16_bits_to_float(u0.x >> 16),
                           bf16_bits_to_float(u0.y), bf16_bits_to_float(u0.y >> 16)};
      const float x1[4] = {bf16_bits_to_float(u1.x), bf16_bits_to_float(u1.x >> 16),
                           bf16_bits_to_float(u1.y), bf16_bits_to_float(u1.y >> 16)};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // the two tokens of channel k as one f32x2: r = fl(fl(x - cen) - mu)
        // (x - 0 is x, so the centring is skipped without it), codes of r / s_v
        float2 r2 = make_float2(x0[k], x1[k]);
        if (centred) r2 = __fadd2_rn(r2, make_float2(-cen[k], -cen[k]));
        r2 = __fadd2_rn(r2, make_float2(-mu[k], -mu[k]));
        const float2 q2 = __fmul2_rn(r2, make_float2(inv[k], inv[k]));
        const float r0 = r2.x, r1 = r2.y;
        uint32_t pr = e4m3x2(q2.x, q2.y);
        if (p.v_bias) {
          // measured E4M3 bias of the residual: dequantised minus exact
          if (rr < nr)
            bias[k] += __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(
                                     static_cast<__nv_fp8_storage_t>(pr & 0xFFu), __NV_E4M3))), sv[k]) - r0;
          if (rr + 1 < nr)
            bias[k] += __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(
                                     static_cast<__nv_fp8_storage_t>(pr >> 8), __NV_E4M3))), sv[k]) - r1;
        }
        // pad tokens (rows >= cnt) are code 0
        if (rr >= nr) pr &= 0xFF00u;
        if (rr + 1 >= nr) pr &= 0x00FFu;
        (e == 0 ? b0[k] : b1[k]) = pr;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) words[k][q] = b0[k] | (b1[k] << 16);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = 4 * l + k;
    tile[c * 8 + (w ^ (l & 7))] = make_uint4(words[k][0], words[k][1], words[k][2], words[k][3]);
  }
  float (*s_bias)[128] = reinterpret_cast<float (*)[128]>(sm + kVBias);
  if (p.v_bias) {
#pragma unroll
    for (int k = 0; k < 4; ++k) s_bias[w][4 * l + k] = bias[k];
  }
  __syncthreads();
  if (p.v_bias && threadIdx.x < 128) {
    // the block's sum per channel, then one atomic per channel per CTA
    float sb = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) sb += s_bias[ww][threadIdx.x];
    atomicAdd(p.vbias_acc + (size_t)bh * kHeadDim + threadIdx.x, sb);
  }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int idx = threadIdx.x + 256 * it;
    const int c = idx >> 3, q = idx & 7;
    const uint4 val = tile[c * 8 + (q ^ ((c >> 2) & 7))];
    *reinterpret_cast<uint4*>(p.v8 + ((size_t)bh * kHeadDim + c) * p.Tpad + t0 + 16 * q) = val;
  }
  }
}

// The E2M1 conversion alone (one code per output byte, low nibble), for
// checking the 4-bit codec value by value; the same cvt as the kernels.
__global__ void e2m1_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ codes, size_t n) {
  const size_t pairs = (n + 1) / 2;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < pairs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = 2 * i;
    const uint32_t c = e2m1x2(x[e], e + 1 < n ? x[e + 1] : 0.f);
    codes[e] = static_cast<uint8_t>(c & 0xFu);
    if (e + 1 < n) codes[e + 1] = static_cast<uint8_t>((c >> 4) & 0xFu);
  }
}

// The conversion alone (two values per thread, grid-stride), for checking the
// codec value by value; the same cvt.rn.satfinite.e4m3x2.f32 as the kernels.
__global__ void e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ codes, size_t n) {
  const size_t pairs = (n + 1) / 2;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < pairs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = 2 * i;
    const float lo = x[e];
    const float hi = e + 1 < n ? x[e + 1] : 0.f;
    const uint32_t c = e4m3x2(lo, hi);
    codes[e] = static_cast<uint8_t>(c & 0xFFu);
    if (e + 1 < n) codes[e + 1] = static_cast<uint8_t>(c >> 8);
  }
}

cudaError_t launch_e2m1_encode(const float* x, uint8_t* codes, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const size_t pairs = (n + 1) / 2;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((pairs + 255) / 256, 152 * 32));
  e2m1_encode_kernel<<<blocks, 256, 0, stream>>>(x, codes, n);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const size_t pairs = (n + 1) / 2;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((pairs + 255) / 256, 152 * 32));
  e4m3_encode_kernel<<<blocks, 256, 0, stream>>>(x, codes, n);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Sequence statistics for the smoothing: grid (nV, H, 2B) (z & 1: 0 = K,
// 1 = V), 256 threads, rows read in token order (a mean over T does not
// depend on the order).  Warp w covers rows 16 w .. +15 of the 128-row block,
// lane l channels 4 l .. 4 l + 3.
__device__ __forceinline__ bool seq_kind_active(const PrepParams& p, int is_v) {
  return is_v ? p.smooth == 2 : p.smooth >= 1;
}

__global__ void __launch_bounds__(256) prep_seq_max_kernel(const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~static_cast<uintptr_t>(127));
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, is_v = blockIdx.z & 1;
  if (!seq_kind_active(p, is_v)) return;
  const int bh = b * p.H + h;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int t0 = j * kVBlock, cnt = min(kVBlock, p.T - t0);
  const int nr = min(16, max(0, cnt - 16 * w));
  uint2 u[16];
  load_rows16(p, is_v ? p.v : p.k, nullptr, b, h, bh, t0 + 16 * w, nr, u);
  float (*s_red)[128] = reinterpret_cast<float (*)[128]>(sm + kVRed);
  float am[4] = {0.f, 0.f, 0.f, 0.f};       // the zero rows past the end change no maximum
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    am[0] = fmaxf(am[0], fabsf(bf16_bits_to_float(u[r].x)));
    am[1] = fmaxf(am[1], fabsf(bf16_bits_to_float(u[r].x >> 16)));
    am[2] = fmaxf(am[2], fabsf(bf16_bits_to_float(u[r].y)));
    am[3] = fmaxf(am[3], fabsf(bf16_bits_to_float(u[r].y >> 16)));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) s_red[w][4 * l + k] = am[k];
  __syncthreads();
  if (threadIdx.x < 128) {
    float m = s_red[0][threadIdx.x];
#pragma unroll
    for (int ww = 1; ww < 8; ++ww) m = fmaxf(m, s_red[ww][threadIdx.x]);
    uint32_t* dst = p.chan_max + ((size_t)is_v * p.B * p.H + bh) * kHeadDim + threadIdx.x;
    if (__float_as_uint(m) > __ldcg(dst)) atomicMax(dst, __float_as_uint(m));
  }
}

// Exact sums: with 2^E <= max|x| < 2^(E+1) over the whole sequence, a bf16
// value of exponent e >= E - W is an integer multiple of 2^(E-7-W) below
// 2^(E+1), so T of them sum below T * 2^(W+8) <= 2^62 (W = 62 - 8 -
// ceil(log2 T)): int64 atomics add them exactly, in any order.
__global__ void __launch_bounds__(256) prep_seq_sum_kernel(const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~static_cast<uintptr_t>(127));
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, is_v = blockIdx.z & 1;
  if (!seq_kind_active(p, is_v)) return;
  const int bh = b * p.H + h;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int t0 = j * kVBlock, cnt = min(kVBlock, p.T - t0);
  const int nr = min(16, max(0, cnt - 16 * w));
  uint2 u[16];
  load_rows16(p, is_v ? p.v : p.k, nullptr, b, h, bh, t0 + 16 * w, nr, u);
  long long (*s_sum)[128] = reinterpret_cast<long long (*)[128]>(sm + kVSum);
  float (*s_low)[128] = reinterpret_cast<float (*)[128]>(sm + kVLow);
  const size_t base = ((size_t)is_v * p.B * p.H + bh) * kHeadDim;
  // in-window values are integer multiples y of 2^(E-7-W), |y| < 2^(W+8) <= 2^45
  float up1[4], up2[4], floor_mag[4];
  bool pre = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int E = exp_of(__uint_as_float(p.chan_max[base + 4 * l + k]));
    pre |= split_scale(7 + p.sum_window - E, up1[k], up2[k]);
    floor_mag[k] = ldexpf(1.f, E - p.sum_window);
  }
  int hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};   // 16 rows: |hi|, |lo| < 2^27
  float low[4] = {0.f, 0.f, 0.f, 0.f};
  // a zero row (past the end) adds nothing to hi, lo or low
  auto rows = [&](auto pre_tag) {
    constexpr bool kPre = decltype(pre_tag)::value;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float x[4] = {bf16_bits_to_float(u[r].x), bf16_bits_to_float(u[r].x >> 16),
                          bf16_bits_to_float(u[r].y), bf16_bits_to_float(u[r].y >> 16)};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool in = fabsf(x[k]) >= floor_mag[k];
        int dl = 0;   // below the window t == 1.5*2^46: hi gains 0
        split_add<kPre>(x[k], up1[k], up2[k], hi[k], dl);
        if (in) lo[k] += dl;
        else low[k] += x[k];
      }
    }
  };
  if (pre) rows(std::true_type{});
  else rows(std::false_type{});
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    s_sum[w][4 * l + k] = (static_cast<long long>(hi[k]) << 23) + lo[k];
    s_low[w][4 * l + k] = low[k];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    long long a = 0;
    float lo = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      a += s_sum[ww][threadIdx.x];
      lo += s_low[ww][threadIdx.x];
    }
    atomicAdd(p.chan_sum + base + threadIdx.x, static_cast<unsigned long long>(a));
    if (lo != 0.f) atomicAdd(p.chan_low + base + threadIdx.x, lo);
  }
}

// grid (B*H, 2), 128 threads: the exact mean, rounded once to fp32.
__global__ void __launch_bounds__(128) prep_seq_finalize_kernel(const PrepParams p) {
  const int bh = blockIdx.x, is_v = blockIdx.y;
  if (!seq_kind_active(p, is_v)) return;
  const size_t i = ((size_t)is_v * p.B * p.H + bh) * kHeadDim + threadIdx.x;
  const int E = exp_of(__uint_as_float(p.chan_max[i]));
  const long long S = static_cast<long long>(p.chan_sum[i]);
  const float low = p.chan_low[i];
  const int lsb = E - 7 - p.sum_window;
  float mean;
  if (low == 0.f) {
    mean = exact_mean_f32(S, lsb, p.T);
  } else {   // values below the window: close, not guaranteed correctly rounded
    mean = static_cast<float>((ldexp(static_cast<double>(S), lsb) + static_cast<double>(low)) /
                              static_cast<double>(p.T));
  }
  p.chan_mean[i] = mean;
}

// grid (B*H), 128 threads: offset added to every output row.
__global__ void __launch_bounds__(128) prep_offset_kernel(const PrepParams p) {
  const size_t i = (size_t)blockIdx.x * kHeadDim + threadIdx.x;
  float off = 0.f;
  if (p.smooth == 2) off = p.chan_mean[(size_t)p.B * p.H * kHeadDim + i];
  if (p.v_bias) off = __fsub_rn(off, __fdiv_rn(p.vbias_acc[i], static_cast<float>(p.T)));
  p.v_offset[i] = off;
}

size_t prep_v_smem_bytes() { return kVSmem; }

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  static PerDeviceOnce once;
  cudaError_t e = once.run([] {
    const int bytes = static_cast<int>(kVSmem);
    cudaError_t r = cudaFuncSetAttribute(prep_v_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(prep_v_quant_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(prep_v_quant_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(prep_seq_max_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(prep_seq_sum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return r;
  });
  if (e != cudaSuccess) return e;
  if (p.smooth >= 1) {
    prep_seq_max_kernel<<<dim3(p.nV, p.H, 2 * p.B), 256, kVSmem, stream>>>(p);
    prep_seq_sum_kernel<<<dim3(p.nV, p.H, 2 * p.B), 256, kVSmem, stream>>>(p);
    prep_seq_finalize_kernel<<<dim3(p.B * p.H, 2), 128, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  prep_qk_kernel<<<dim3(p.nQK, p.H, 2 * p.B), 128, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prep_v_stats_kernel<<<dim3(p.nV, p.H, p.B), 256, kVSmem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.v_fp4)
    prep_v_quant_kernel<true><<<dim3(p.nV, p.H, p.B), 256, kVSmem, stream>>>(p);
  else
    prep_v_quant_kernel<false><<<dim3(p.nV, p.H, p.B), 256, kVSmem, stream>>>(p);
  if (p.v_offset) prep_offset_kernel<<<p.B * p.H, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8attn
