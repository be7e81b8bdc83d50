// Stage 2: block-scaled FP8 attention mainloop on tcgen05 tensor cores.
//
// What it computes (per query row, over the visited 128-key tiles):
//   TeleFuser "FP8 Sol-Attn" blog, section "SM90 CuTe mainloop": E4M3 QK with
//   fp32 accumulation, Q/K block scales applied to the scores before an fp32
//   online softmax, P cast to E4M3 and multiplied with token-contiguous E4M3 V,
//   the V channel scale applied after all PV products, bf16 output.
//   VC-Attention news article, section 2 "V-Smooth" (third step): the block
//   mean comes back as the rank-one term r_ij mu_j^T, r_ij the row sum of the
//   tile's probabilities, sharing the accumulator's rescaling; section 3
//   "ExpCast": the P byte is round(8 z + 56 + beta), z the base-2 log score.
//   P-Cast Precision review, sections 3-5: static P scale S before the cast,
//   forward or reverse KV order.  FPSAttention article, section 2.2: a
//   per-query-tile list of key tiles (sliding-tile window).
//
// Design (one CTA = one 128-row query tile; 320 threads, 1 CTA per SM):
//   warp 8      TMA producer: Q once, then K and V tiles through a 4-stage ring
//   warp 9      TMEM allocator and single-thread MMA issuer (descriptors are
//               precomputed; QK_{t+1} is issued before PV_t so the tensor
//               core has the next score tile queued while the softmax runs)
//   warps 0-7   softmax: query row i is shared by warp (i/32) and warp 4+(i/32);
//               the first owns key columns 0-63, the second 64-127 (and output
//               channels 0-63 / 64-127).  The two halves of a row exchange
//               their partial row max through shared memory and a per-pair
//               mbarrier every tile.
// Tensor memory (512 columns):
//   S0 [0,128) S1 [128,256)   double-buffered 128x128 fp32 scores
//   O  [256,400)              128x144 fp32 accumulator: 128 output channels,
//                             column 128 = row sum l, 129-143 zero
//   P0 [416,448) P1 [448,480) E4M3 probabilities, 4 codes per column (TS operand)
//   Q  [480,512)              E4M3 query tile (TS operand)
// Per KV tile t:
//   S_t  = Qq Kq_t^T                     kind::f8f6f4 TS, M=128 N=128 K=4x32
//   P_t  = E4M3 codes (exp2+cvt or ExpCast), written to TMEM by the softmax
//   O   += P_t [Vq_t ; 1 ; 0]            kind::f8f6f4 TS, M=128 N=144 K=4x32:
//          the ones row appended to the V tile makes column 128 accumulate the
//          row sum of the DECODED codes, with the same rescaling as O
//   every 4 tiles (V-Smooth only): O += [r_hi r_lo ...] [mu~ ; mu~ ...]  kind::tf32,
//          M=128 N=128 K=8: the rank-one mean terms of four tiles in one MMA;
//          r_t = l after tile t minus l before it, split into two TF32 halves;
//          mu~ = mu / s_v per channel
// The row max is updated exactly at every tile.  When it moves, the softmax
// threads rescale their O columns (and l) in TMEM after PV_{t-1} completes.
#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8attn {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = 128 * 128;               // one 128x128 E4M3 tile
constexpr uint32_t kVStageBytes = kTileBytes + 2048;     // V tile + 16-row ones block

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffMeanA = kOffV + kStages * kVStageBytes;   // 128 x 8 TF32, no swizzle
constexpr uint32_t kOffMeanB = kOffMeanA + 4096;                 // 128 x 8 TF32, no swizzle
constexpr uint32_t kOffSacc = kOffMeanB + 4096;                  // 128 fp32 output channel scales
constexpr uint32_t kOffMax = kOffSacc + 512;                     // [2 slots][2 halves][128] fp32
constexpr uint32_t kOffBar = kOffMax + 2048;
constexpr int kNumBars = 2 + 4 * kStages + 4 * 2 + 4 + 1;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;            // abort flag, TMEM base
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                // + alignment slack

// TMEM column map
constexpr uint32_t kColS = 0, kColO = 256, kColL = 256 + 128, kColP = 416, kColQ = 480;

constexpr uint32_t kIdescQK = make_idesc(0, 128, 128);     // E4M3 x E4M3 -> F32, N=128
constexpr uint32_t kIdescPV = make_idesc(0, 128, 144);     // N=144: 128 channels + ones row
constexpr uint32_t kIdescMean = make_idesc(2, 128, 128);   // TF32 x TF32 -> F32

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return make_sdesc(saddr, 16, 1024, 2);
}
__device__ __forceinline__ uint64_t plain_desc(uint32_t saddr) {
  // no swizzle, K-major: 8 rows x 16 B core matrices; K-adjacent cores 128 B
  // apart (LBO), 8-row groups 256 B apart (SBO)
  return make_sdesc(saddr, 128, 256, 0);
}

// Offset of element (row, k) of a 128 x 8 TF32 operand in the no-swizzle layout.
__device__ __forceinline__ uint32_t plain_off(int row, int k) {
  return (row >> 3) * 256 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4;
}

struct TileList {
  const int32_t* col;
  int base, n, nV, reverse;
  int* status;
  __device__ __forceinline__ int at(int it) const {
    const int idx = reverse ? (n - 1 - it) : it;
    int j = col ? __ldg(col + base + idx) : idx;
    if (static_cast<unsigned>(j) >= static_cast<unsigned>(nV)) {
      atomicExch(status, kStatusBadTile);
      j = 0;
    }
    return j;
  }
};

__device__ __forceinline__ bool flush_mean(int it, int n, int vsmooth) {
  return vsmooth && it >= 1 && ((it & 3) == 0 || it == n);
}

__device__ __forceinline__ void split_tf32(float r, float& hi, float& lo) {
  hi = round_tf32(r);
  lo = round_tf32(r - hi);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;

  TileList tl;
  tl.col = p.col;
  tl.nV = p.nV;
  tl.reverse = p.reverse;
  tl.status = p.status;
  if (p.row_ptr) {
    tl.base = __ldg(p.row_ptr + qt);
    tl.n = __ldg(p.row_ptr + qt + 1) - tl.base;
    if (tl.n < 0) {
      atomicExch(p.status, kStatusBadTile);
      tl.n = 0;
    }
  } else {
    tl.base = 0;
    tl.n = p.nV;
  }
  const int n = tl.n;

  const uint32_t bar0 = sb + kOffBar;
  const uint32_t q_full = bar0, q_tmem = bar0 + 8;
  auto k_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (2 + kStages + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + 2 * kStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (2 + 3 * kStages + s); };
  auto s_full = [&](int s) { return bar0 + 8 * (2 + 4 * kStages + s); };
  auto s_empty = [&](int s) { return bar0 + 8 * (4 + 4 * kStages + s); };
  auto p_full = [&](int s) { return bar0 + 8 * (6 + 4 * kStages + s); };
  auto o_done = [&](int s) { return bar0 + 8 * (8 + 4 * kStages + s); };
  auto xchg = [&](int w) { return bar0 + 8 * (10 + 4 * kStages + w); };
  const uint32_t mma_drain = bar0 + 8 * (14 + 4 * kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 4);
  float* s_acc = reinterpret_cast<float*>(smem + kOffSacc);
  const uint64_t to = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_tmem, 256);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 256);
      mbar_init(p_full(s), 256);
      mbar_init(o_done(s), 1);
    }
    for (int w = 0; w < 4; ++w) mbar_init(xchg(w), 64);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  {
    // ones block of every V stage: row 0 = E4M3 1.0 (0x38) for all 128 keys,
    // rows 1..15 = 0 (2 KB per stage, 128 x 16 B)
    const int t = threadIdx.x;
    for (int q = t; q < kStages * 128; q += kThreads) {
      const int st = q >> 7, c = q & 127;
      const uint32_t w = c < 8 ? 0x38383838u : 0u;
      *reinterpret_cast<uint4*>(smem + kOffV + st * kVStageBytes + kTileBytes + c * 16) =
          make_uint4(w, w, w, w);
    }
    if (t < 128) {
      const float sv = __ldg(p.v_scale + (size_t)bh * kHeadDim + t);
      s_acc[t] = sv > 0.f ? sv : 1.f;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int nk = 0, nv = 0;          // K / V loads issued
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_4d(sb + kOffQ, &p.tm_q, q_full, 0, h, qt * kTile, b);
      for (int it = 0; it < n; ++it) {
        const int j = tl.at(it);
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(k_empty(st), ph ^ 1, abort_flag, to)) break;
        mbar_arrive_expect_tx(k_full(st), kTileBytes);
        tma_load_4d(sb + kOffK + st * kTileBytes, &p.tm_k, k_full(st), 0, h, j * kTile, b);
        nk = it + 1;
        if (!mbar_wait(v_empty(st), ph ^ 1, abort_flag, to)) break;
        mbar_arrive_expect_tx(v_full(st), kTileBytes);
        tma_load_3d(sb + kOffV + st * kVStageBytes, &p.tm_v, v_full(st), j * kTile, 0, bh);
        nv = it + 1;
      }
      // Drain: every issued load must land before the CTA exits, whatever the
      // abort flag says.  A consumed phase tests complete at once.
      mbar_wait_drain(q_full, 0, to);
      for (int s = 0; s < kStages; ++s) {
        if (nk > s) mbar_wait_drain(k_full(s), ((nk - 1 - s) / kStages) & 1, to);
        if (nv > s) mbar_wait_drain(v_full(s), ((nv - 1 - s) / kStages) & 1, to);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // stage descriptors differ only in the start-address field (16-byte units)
      const uint64_t kdesc0 = sw128_desc(sb + kOffK), vdesc0 = sw128_desc(sb + kOffV);
      auto kdesc = [&](int st) { return kdesc0 + static_cast<uint64_t>(st * (kTileBytes >> 4)); };
      auto vdesc = [&](int st) { return vdesc0 + static_cast<uint64_t>(st * (kVStageBytes >> 4)); };
      const uint64_t mean_a = plain_desc(sb + kOffMeanA), mean_b = plain_desc(sb + kOffMeanB);
      const uint32_t tq = tmem + kColQ, to_ = tmem + kColO;
      bool ok = mbar_wait(q_tmem, 0, abort_flag, to);
      tc_fence_after();
      auto issue_qk = [&](int it) -> bool {
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        const int s = it & 1;
        if (!mbar_wait(k_full(st), ph, abort_flag, to)) return false;
        if (!mbar_wait(s_empty(s), ((it >> 1) & 1) ^ 1, abort_flag, to)) return false;
        tc_fence_after();
        const uint32_t ts = tmem + kColS + s * 128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_ts(ts, tq + kk * 8, kdesc(st) + 2 * kk, kIdescQK, kk > 0);
        mma_commit(s_full(s));
        mma_commit(k_empty(st));
        return true;
      };
      if (ok && n > 0) ok = issue_qk(0);
      for (int it = 0; ok && it <= n; ++it) {
        if (it + 1 < n && !issue_qk(it + 1)) break;
        if (!mbar_wait(p_full(it & 1), (it >> 1) & 1, abort_flag, to)) break;
        tc_fence_after();
        if (flush_mean(it, n, p.vsmooth)) mma_tf32(to_, mean_a, mean_b, kIdescMean, 1);
        if (it < n) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(v_full(st), ph, abort_flag, to)) break;
          tc_fence_after();
          const uint32_t tp = tmem + kColP + (it & 1) * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_ts(to_, tp + kk * 8, vdesc(st) + 2 * kk, kIdescPV, (it > 0 || kk > 0) ? 1u : 0u);
          mma_commit(v_empty(st));
        }
        mma_commit(o_done(it & 1));
      }
      // Drain: all issued MMAs must finish before TMEM is released.
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0, to);
    }
  } else {
    // ------------------------------------------------------------ softmax (rows)
    const int wq = warp & 3, half = warp >> 2;
    const int i = wq * 32 + lane;                      // query row within the tile
    const int row = qt * kTile + i;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO + half * 64;
    const float sq = row < p.T ? __ldg(p.q_scale + (size_t)bh * p.nQK + row / kQKBlock) : 0.f;
    const float cq = sq * p.sm_scale_log2;           // raw score -> log2-domain logit (x k scale)
    const float* kscale = p.k_scale + (size_t)bh * p.nQK;
    const uint16_t* vmean = reinterpret_cast<const uint16_t*>(p.v_mean) + (size_t)bh * p.nV * kHeadDim;
    float* xmax = reinterpret_cast<float*>(smem + kOffMax);
    const float inv_sacc = __fdiv_rn(1.f, s_acc[i]);
    bool ok = true;

    // Q tile -> TMEM (TS operand of QK): this half copies 16 columns (64 codes) of row i
    ok = mbar_wait(q_full, 0, abort_flag, to);
    if (__all_sync(0xffffffffu, ok)) {
      uint32_t qw[16];
      const uint8_t* qrow = smem + kOffQ + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + (((4 * half + c) ^ (i & 7)) << 4));
        qw[4 * c] = v.x;
        qw[4 * c + 1] = v.y;
        qw[4 * c + 2] = v.z;
        qw[4 * c + 3] = v.w;
      }
      tmem_st16(tmem + lane_base + kColQ + 16 * half, qw);
      tmem_wait_st();
    } else {
      ok = false;
    }
    tc_fence_before();
    mbar_arrive(q_tmem);

    float m = -INFINITY;     // running row max, log2 domain
    float lprev = 0.f;       // l (TMEM column 128) as PV of the newest tile found it
    float rp0 = 0.f, rp1 = 0.f, rp2 = 0.f, rp3 = 0.f;   // pending tile row sums of this mean group
    float mp0 = 0.f, mp1 = 0.f, mp2 = 0.f, mp3 = 0.f;   // mu~ of channel i for the group's tiles

    for (int it = 0; ok && it <= n; ++it) {
      float alpha = 1.f;
      float mu_new = 0.f;      // mu~ of this iteration's tile; slotted after the flush below
      if (it < n) {
        const int j = tl.at(it);
        const int s = it & 1;
        float mu_raw = 0.f;
        if (p.vsmooth && half == 1)
          mu_raw = __uint_as_float(static_cast<uint32_t>(__ldg(vmean + (size_t)j * kHeadDim + i)) << 16);
        const int kb = 2 * j + half;
        const float c = cq * (kb < p.nQK ? __ldg(kscale + kb) : 0.f);
        const int valid = min(64, p.T - j * kTile - 64 * half);   // may be <= 0

        ok = mbar_wait(s_full(s), (it >> 1) & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64];
        const uint32_t tS = tmem + lane_base + kColS + s * 128 + half * 64;
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_empty(s));

        if (valid < 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e >= valid) sv[e] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; e += 2) mx = fmax3(mx, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        const float part = valid > 0 ? mx * c : -INFINITY;
        // exchange the half-row maxima of row i with the partner warp
        xmax[((it & 1) * 2 + half) * 128 + i] = part;
        mbar_arrive(xchg(wq));
        ok = mbar_wait(xchg(wq), it & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const float other = xmax[((it & 1) * 2 + (half ^ 1)) * 128 + i];
        const float m_new = fmaxf(m, fmaxf(part, other));
        alpha = (m == m_new) ? 1.f : ex2_approx(m - m_new);
        m = m_new;

        uint32_t pw[16];
        if (p.pcast == 0) {
          // exp2 + cvt: code = E4M3(S * 2^(y - m)), y = raw * c
          const float bb = p.log2_pscale - m_new;
          const float2 c2 = make_float2(c, c), b2 = make_float2(bb, bb);
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float2 f01 = ffma2(make_float2(__uint_as_float(sv[4 * w]), __uint_as_float(sv[4 * w + 1])), c2, b2);
            const float2 f23 = ffma2(make_float2(__uint_as_float(sv[4 * w + 2]), __uint_as_float(sv[4 * w + 3])), c2, b2);
            pw[w] = prmt(cvt_e4m3x2(ex2_approx(f01.x), ex2_approx(f01.y)),
                         cvt_e4m3x2(ex2_approx(f23.x), ex2_approx(f23.y)), 0x5410u);
          }
        } else {
          // ExpCast: u = sat((8 (y - m + log2 S) + 56 + beta) / 256), code = rne(256 u)
          const float bb8 = (8.f * (p.log2_pscale - m_new) + 56.f + p.beta) * (1.f / 256.f);
          const float a8 = c * (8.f / 256.f);
          const float2 k256 = make_float2(256.f, 256.f), kmag = make_float2(8388608.f, 8388608.f);
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float u0 = fma_sat(__uint_as_float(sv[4 * w]), a8, bb8);
            const float u1 = fma_sat(__uint_as_float(sv[4 * w + 1]), a8, bb8);
            const float u2 = fma_sat(__uint_as_float(sv[4 * w + 2]), a8, bb8);
            const float u3 = fma_sat(__uint_as_float(sv[4 * w + 3]), a8, bb8);
            const float2 t01 = ffma2(make_float2(u0, u1), k256, kmag);
            const float2 t23 = ffma2(make_float2(u2, u3), k256, kmag);
            const uint32_t lo = prmt(__float_as_uint(t01.x), __float_as_uint(t01.y), 0x5140u);
            const uint32_t hi = prmt(__float_as_uint(t23.x), __float_as_uint(t23.y), 0x5140u);
            pw[w] = prmt(lo, hi, 0x5410u);
          }
        }
        if (valid < 64) {
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const int nvk = valid - 4 * w;
            if (nvk <= 0) pw[w] = 0u;
            else if (nvk < 4) pw[w] &= (1u << (8 * nvk)) - 1u;
          }
        }
        // P buffer s was last read by PV_{it-2}
        if (it >= 2) {
          ok = mbar_wait(o_done(s), ((it - 2) >> 1) & 1, abort_flag, to);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st16(tmem + lane_base + kColP + s * 32 + half * 16, pw);
        tmem_wait_st();
        mu_new = round_tf32(mu_raw * inv_sacc);
      }

      // ---- work that needs PV_{it-1}: V-Smooth row sum, O rescale
      const bool rescale = it >= 1 && it < n && __any_sync(0xffffffffu, alpha != 1.f);
      if (it >= 1 && (p.vsmooth || rescale)) {
        ok = mbar_wait(o_done((it - 1) & 1), ((it - 1) >> 1) & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (p.vsmooth && half == 0) {
          const float lnow = __uint_as_float(tmem_ld1(tmem + lane_base + kColL));
          tmem_wait_ld();
          const float r = lnow - lprev;
          lprev = lnow;
          switch ((it - 1) & 3) {
            case 0: rp0 = r; break;
            case 1: rp1 = r; break;
            case 2: rp2 = r; break;
            default: rp3 = r; break;
          }
        }
      }
      if (it < n) {
        rp0 *= alpha; rp1 *= alpha; rp2 *= alpha; rp3 *= alpha;
        if (rescale) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tmem_ld32(tO + cc * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 r2 = __fmul2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                           make_float2(alpha, alpha));
              v[e] = __float_as_uint(r2.x);
              v[e + 1] = __float_as_uint(r2.y);
            }
            tmem_st32(tO + cc * 32, v);
          }
          if (half == 0) {
            const float lnow = __uint_as_float(tmem_ld1(tmem + lane_base + kColL));
            tmem_wait_ld();
            const float lsc = lnow * alpha;
            tmem_st1(tmem + lane_base + kColL, __float_as_uint(lsc));
            lprev = lsc;
          }
          tmem_wait_st();
        }
      }
      if (flush_mean(it, n, p.vsmooth)) {
        if (half == 0) {
          float h0, l0, h1, l1, h2, l2, h3, l3;
          split_tf32(rp0, h0, l0);
          split_tf32(rp1, h1, l1);
          split_tf32(rp2, h2, l2);
          split_tf32(rp3, h3, l3);
          *reinterpret_cast<float4*>(smem + kOffMeanA + plain_off(i, 0)) = make_float4(h0, l0, h1, l1);
          *reinterpret_cast<float4*>(smem + kOffMeanA + plain_off(i, 4)) = make_float4(h2, l2, h3, l3);
          rp0 = rp1 = rp2 = rp3 = 0.f;
        } else {
          *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 0)) = make_float4(mp0, mp0, mp1, mp1);
          *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 4)) = make_float4(mp2, mp2, mp3, mp3);
        }
        fence_proxy_async_smem();
      }
      if (it < n) {
        switch (it & 3) {
          case 0: mp0 = mu_new; break;
          case 1: mp1 = mu_new; break;
          case 2: mp2 = mu_new; break;
          default: mp3 = mu_new; break;
        }
      }
      tc_fence_before();
      mbar_arrive(p_full(it & 1));
    }

    // ---- epilogue: O * s_acc / l -> bf16
    if (ok) {
      ok = mbar_wait(o_done(n & 1), (n >> 1) & 1, abort_flag, to);
      ok = __all_sync(0xffffffffu, ok);
    }
    tc_fence_after();
    const bool have = ok && n > 0;
    float l = 0.f;
    if (have) {
      l = __uint_as_float(tmem_ld1(tmem + lane_base + kColL));
      tmem_wait_ld();
    }
    const float inv_l = (l > 0.f) ? __fdiv_rn(1.f, l) : 0.f;
    __nv_bfloat16* orow = p.out + (((size_t)b * p.T + row) * p.H + h) * kHeadDim + half * 64;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tO + cc * 32, v);
        tmem_wait_ld();
      }
      if (row < p.T) {
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float o0 = 0.f, o1 = 0.f;
          if (have && l > 0.f) {
            const int ch = half * 64 + cc * 32 + 2 * e;
            o0 = __uint_as_float(v[2 * e]) * s_acc[ch] * inv_l;
            o1 = __uint_as_float(v[2 * e + 1]) * s_acc[ch + 1] * inv_l;
          }
          __nv_bfloat162 hv = __floats2bfloat162_rn(o0, o1);
          packed[e] = *reinterpret_cast<uint32_t*>(&hv);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, kStatusTimeout);
}

size_t attn_smem_bytes() { return kSmemBytes; }

cudaError_t launch_attn(const AttnParams& p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_fwd_kernel<<<dim3(p.nQt, p.H, p.B), kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8attn
