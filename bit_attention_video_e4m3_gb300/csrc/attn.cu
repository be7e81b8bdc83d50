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
// Design (one CTA = one 128-row query tile; 192 threads):
//   warp 4      TMA producer: Q once, then K and V tiles through a 3-stage ring
//   warp 5      TMEM allocator and single-thread MMA issuer:
//                 QK_{t+1} is issued before PV_t so the tensor core always
//                 has the next score tile queued while the softmax runs
//   warps 0-3   softmax: thread i owns query row i (TMEM lane i)
// Tensor memory (512 columns): S0 | S1 (double-buffered 128x128 fp32 scores),
//   O (128x128 fp32 output accumulator), R0 | R1 (16 columns each: row sums).
// Per KV tile t:
//   S_t  = Qq Kq_t^T                     kind::f8f6f4, M=128 N=128 K=4x32
//   P_t  = E4M3 codes (exp2+cvt or ExpCast) written to shared memory in the
//          128-byte-swizzled K-major layout the MMA reads
//   O   += P_t Vq_t                      kind::f8f6f4, M=128 N=128 K=4x32
//   R_t  = P_t 1                         kind::f8f6f4, M=128 N=16: the row sum of
//          the DECODED codes, exact in fp32 and free of CUDA-core work
//   every 4 tiles (V-Smooth only): O += [r_hi r_lo ...] [mu~ ; mu~ ...]   kind::tf32,
//          M=128 N=128 K=8: the rank-one mean terms of four tiles in one MMA,
//          r split into two TF32 halves, mu~ = mu / s_v per channel
// The row max is updated exactly at every tile; O is rescaled in TMEM by the
// softmax thread when its row max moves (after PV_{t-1} has completed).
#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8attn {

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = 128 * 128;   // one 128x128 E4M3 tile

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kStages * kTileBytes;
constexpr uint32_t kOffOnes = kOffP + 2 * kTileBytes;      // 16 x 128 B E4M3, row 0 = 1.0
constexpr uint32_t kOffMeanA = kOffOnes + 2048;            // 128 x 8 TF32, no swizzle
constexpr uint32_t kOffMeanB = kOffMeanA + 4096;           // 128 x 8 TF32, no swizzle
constexpr uint32_t kOffSacc = kOffMeanB + 4096;            // 128 fp32 output channel scales
constexpr uint32_t kOffBar = kOffSacc + 512;
// barriers: q_full, k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2],
// s_empty[2], p_full[2], o_done[2], mma_drain
constexpr int kNumBars = 1 + 4 * kStages + 4 * 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;      // abort flag, TMEM base
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;          // + alignment slack

// TMEM column map
constexpr uint32_t kColS0 = 0, kColO = 256, kColR0 = 384;

constexpr uint32_t kIdescQK = make_idesc(0, 128, 128);     // E4M3 x E4M3 -> F32
constexpr uint32_t kIdescRS = make_idesc(0, 128, 16);
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
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (1 + kStages + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (1 + 2 * kStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (1 + 3 * kStages + s); };
  auto s_full = [&](int s) { return bar0 + 8 * (1 + 4 * kStages + s); };
  auto s_empty = [&](int s) { return bar0 + 8 * (3 + 4 * kStages + s); };
  auto p_full = [&](int s) { return bar0 + 8 * (5 + 4 * kStages + s); };
  auto o_done = [&](int s) { return bar0 + 8 * (7 + 4 * kStages + s); };
  const uint32_t mma_drain = bar0 + 8 * (9 + 4 * kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 4);
  float* s_acc = reinterpret_cast<float*>(smem + kOffSacc);
  const uint64_t to = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 128);
      mbar_init(p_full(s), 128);
      mbar_init(o_done(s), 1);
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  if (threadIdx.x < 128) {
    // ones block: row 0 = E4M3 1.0 (0x38) in all 128 key slots, rows 1..15 = 0
    const uint32_t w = threadIdx.x < 8 ? 0x38383838u : 0u;
    reinterpret_cast<uint4*>(smem + kOffOnes)[threadIdx.x] = make_uint4(w, w, w, w);
    const float sv = __ldg(p.v_scale + (size_t)bh * kHeadDim + threadIdx.x);
    s_acc[threadIdx.x] = sv > 0.f ? sv : 1.f;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
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
        tma_load_3d(sb + kOffV + st * kTileBytes, &p.tm_v, v_full(st), j * kTile, 0, bh);
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, abort_flag, to);
      tc_fence_after();
      auto issue_qk = [&](int it) -> bool {
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        const int s = it & 1;
        if (!mbar_wait(k_full(st), ph, abort_flag, to)) return false;
        if (!mbar_wait(s_empty(s), ((it >> 1) & 1) ^ 1, abort_flag, to)) return false;
        tc_fence_after();
        const uint32_t qa = sb + kOffQ, ka = sb + kOffK + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8(tmem + kColS0 + s * 128, sw128_desc(qa + kk * 32), sw128_desc(ka + kk * 32),
                 kIdescQK, kk > 0);
        mma_commit(s_full(s));
        mma_commit(k_empty(st));
        return true;
      };
      if (ok && n > 0) ok = issue_qk(0);
      for (int it = 0; ok && it <= n; ++it) {
        if (it + 1 < n && !issue_qk(it + 1)) break;
        if (!mbar_wait(p_full(it & 1), (it >> 1) & 1, abort_flag, to)) break;
        tc_fence_after();
        if (flush_mean(it, n, p.vsmooth))
          mma_tf32(tmem + kColO, plain_desc(sb + kOffMeanA), plain_desc(sb + kOffMeanB),
                   kIdescMean, 1);
        if (it < n) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(v_full(st), ph, abort_flag, to)) break;
          tc_fence_after();
          const uint32_t pa = sb + kOffP + (it & 1) * kTileBytes;
          const uint32_t va = sb + kOffV + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(tmem + kColO, sw128_desc(pa + kk * 32), sw128_desc(va + kk * 32), kIdescQK,
                   (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(tmem + kColR0 + (it & 1) * 16, sw128_desc(pa + kk * 32),
                   sw128_desc(sb + kOffOnes + kk * 32), kIdescRS, kk > 0);
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
    const int i = threadIdx.x;                       // query row within the tile
    const int row = qt * kTile + i;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    const float sq = row < p.T ? __ldg(p.q_scale + (size_t)bh * p.nQK + row / kQKBlock) : 0.f;
    const float cq = sq * p.sm_scale_log2;           // raw score -> log2-domain logit (x k scale)
    const float inv_sacc = __fdiv_rn(1.f, s_acc[i]);
    const float* kscale = p.k_scale + (size_t)bh * p.nQK;
    const uint16_t* vmean = reinterpret_cast<const uint16_t*>(p.v_mean) + (size_t)bh * p.nV * kHeadDim;
    const uint32_t p_row_off = (i >> 3) * 1024 + (i & 7) * 128;

    float m = -INFINITY;     // running row max, log2 domain
    float lacc = 0.f;        // row sum (frame of the latest max), without the newest tile's r
    float rp0 = 0.f, rp1 = 0.f, rp2 = 0.f, rp3 = 0.f;   // pending tile row sums of this mean group
    float mp0 = 0.f, mp1 = 0.f, mp2 = 0.f, mp3 = 0.f;   // mu~ of channel i for the group's tiles
    bool ok = true;

    for (int it = 0; it <= n; ++it) {
      float alpha = 1.f;
      float mu_new = 0.f;      // mu~ of this iteration's tile; slotted after the flush below
      if (it < n) {
        const int j = tl.at(it);
        const int s = it & 1;
        float mu_raw = 0.f;
        if (p.vsmooth) mu_raw = __uint_as_float(static_cast<uint32_t>(__ldg(vmean + (size_t)j * kHeadDim + i)) << 16);
        const float sk0 = __ldg(kscale + 2 * j);
        const float sk1 = (2 * j + 1 < p.nQK) ? __ldg(kscale + 2 * j + 1) : 0.f;
        const float c0 = cq * sk0, c1 = cq * sk1;
        const int kv_valid = min(kTile, p.T - j * kTile);

        ok = mbar_wait(s_full(s), (it >> 1) & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[128];
        const uint32_t tS = tmem + lane_base + kColS0 + s * 128;
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(sv + 0));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(sv + 64));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(sv + 96));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_empty(s));

        if (kv_valid < kTile) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= kv_valid) sv[c] = __float_as_uint(-INFINITY);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 2) mx0 = fmax3(mx0, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
#pragma unroll
        for (int c = 64; c < 128; c += 2) mx1 = fmax3(mx1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        float mt = mx0 * c0;
        if (kv_valid > 64) mt = fmaxf(mt, mx1 * c1);
        const float m_new = fmaxf(m, mt);
        alpha = (m == m_new) ? 1.f : ex2_approx(m - m_new);
        m = m_new;

        uint32_t pw[32];
        if (p.pcast == 0) {
          // exp2 + cvt: code = E4M3(S * 2^(y - m)), y = raw * c
          const float bb = p.log2_pscale - m_new;
#pragma unroll
          for (int w = 0; w < 32; ++w) {
            const float c = w < 16 ? c0 : c1;
            float f0, f1, f2, f3;
            fma2(__uint_as_float(sv[4 * w]), __uint_as_float(sv[4 * w + 1]), c, c, bb, bb, f0, f1);
            fma2(__uint_as_float(sv[4 * w + 2]), __uint_as_float(sv[4 * w + 3]), c, c, bb, bb, f2, f3);
            pw[w] = cvt_e4m3x2(ex2_approx(f0), ex2_approx(f1)) |
                    (cvt_e4m3x2(ex2_approx(f2), ex2_approx(f3)) << 16);
          }
        } else {
          // ExpCast: u = sat((8 (y - m + log2 S) + 56 + beta) / 256), code = rne(256 u)
          const float bb8 = (8.f * (p.log2_pscale - m_new) + 56.f + p.beta) * (1.f / 256.f);
          const float a0 = c0 * (8.f / 256.f), a1 = c1 * (8.f / 256.f);
#pragma unroll
          for (int w = 0; w < 32; ++w) {
            const float a = w < 16 ? a0 : a1;
            const float u0 = fma_sat(__uint_as_float(sv[4 * w]), a, bb8);
            const float u1 = fma_sat(__uint_as_float(sv[4 * w + 1]), a, bb8);
            const float u2 = fma_sat(__uint_as_float(sv[4 * w + 2]), a, bb8);
            const float u3 = fma_sat(__uint_as_float(sv[4 * w + 3]), a, bb8);
            float t0, t1, t2, t3;
            fma2(u0, u1, 256.f, 256.f, 8388608.f, 8388608.f, t0, t1);
            fma2(u2, u3, 256.f, 256.f, 8388608.f, 8388608.f, t2, t3);
            const uint32_t lo = prmt(__float_as_uint(t0), __float_as_uint(t1), 0x5140u);
            const uint32_t hi = prmt(__float_as_uint(t2), __float_as_uint(t3), 0x5140u);
            pw[w] = prmt(lo, hi, 0x5410u);
          }
        }
        if (kv_valid < kTile) {
#pragma unroll
          for (int w = 0; w < 32; ++w) {
            const int nv = kv_valid - 4 * w;
            if (nv <= 0) pw[w] = 0u;
            else if (nv < 4) pw[w] &= (1u << (8 * nv)) - 1u;
          }
        }
        // P tile row i -> shared memory, 128-byte swizzle: chunk c at (c ^ (i & 7))
        uint8_t* prow = smem + kOffP + s * kTileBytes + p_row_off;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (i & 7)) << 4)) =
              make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
        fence_proxy_async_smem();
        mu_new = round_tf32(mu_raw * inv_sacc);
      }

      // ---- work that needs PV_{it-1}: its row sum, then the O rescale
      if (it >= 1) {
        ok = mbar_wait(o_done((it - 1) & 1), ((it - 1) >> 1) & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float r = __uint_as_float(tmem_ld1(tmem + lane_base + kColR0 + ((it - 1) & 1) * 16));
        tmem_wait_ld();
        lacc += r;
        switch ((it - 1) & 3) {
          case 0: rp0 = r; break;
          case 1: rp1 = r; break;
          case 2: rp2 = r; break;
          default: rp3 = r; break;
        }
      }
      if (it < n) {
        lacc *= alpha;
        rp0 *= alpha; rp1 *= alpha; rp2 *= alpha; rp3 *= alpha;
        if (it >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld32(tO + cc * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(tO + cc * 32, v);
          }
          tmem_wait_st();
        }
      }
      if (flush_mean(it, n, p.vsmooth)) {
        float h0, l0, h1, l1, h2, l2, h3, l3;
        split_tf32(rp0, h0, l0);
        split_tf32(rp1, h1, l1);
        split_tf32(rp2, h2, l2);
        split_tf32(rp3, h3, l3);
        *reinterpret_cast<float4*>(smem + kOffMeanA + plain_off(i, 0)) = make_float4(h0, l0, h1, l1);
        *reinterpret_cast<float4*>(smem + kOffMeanA + plain_off(i, 4)) = make_float4(h2, l2, h3, l3);
        *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 0)) = make_float4(mp0, mp0, mp1, mp1);
        *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 4)) = make_float4(mp2, mp2, mp3, mp3);
        fence_proxy_async_smem();
        rp0 = rp1 = rp2 = rp3 = 0.f;
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
    const float inv_l = (lacc > 0.f) ? __fdiv_rn(1.f, lacc) : 0.f;
    __nv_bfloat16* orow = p.out + (((size_t)b * p.T + row) * p.H + h) * kHeadDim;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
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
          if (have && lacc > 0.f) {
            o0 = __uint_as_float(v[2 * e]) * s_acc[cc * 32 + 2 * e] * inv_l;
            o1 = __uint_as_float(v[2 * e + 1]) * s_acc[cc * 32 + 2 * e + 1] * inv_l;
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
  if (warp == 5) {
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
