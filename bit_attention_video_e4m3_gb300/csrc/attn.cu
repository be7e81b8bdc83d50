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
// Design (one CTA = one 128-row query tile; 352 threads, 1 CTA per SM):
//   warp 8      TMA producer: Q once, then K_t and V_t in tile order through
//               two 4-stage rings (suspending waits on the ring stages)
//   warp 9      TMEM allocator and QK issuer: each QK as soon as its key tile
//               has landed and its score buffer is free, so score tiles run
//               ahead of the softmax
//   warp 10     PV issuer: each PV as soon as its probabilities are written.
//               Issuing warps run warp-wide loops with uniform control flow and
//               one elected lane issues each MMA (operands stay in uniform
//               registers); QK and PV have their own warps because a
//               tcgen05.mma stalls its warp while the tensor pipe is busy.
//   warps 0-3   softmax group 0: the even-numbered KV tiles of the visiting order
//   warps 4-7   softmax group 1: the odd-numbered tiles
//               In both groups thread (warp & 3) * 32 + lane owns query row i
//               (TMEM lane i) and all 128 key columns of its tile.  There is
//               ONE running row max: the group on tile t takes m_{t-1} from the
//               other group through shared memory.  The score barrier of tile t
//               counts the QK commit and the other group's 128 arrivals after it
//               stored m_{t-1}, so one wait covers both (a separate hand-off
//               barrier cost ~3 % more); the two groups overlap everything except
//               that hand-off.
// Tensor memory (512 columns):
//   S0 [0,128) S1 [128,256)   fp32 scores of the even / odd tiles
//   O  [256,400)              128x144 fp32 accumulator: output channels 0-127,
//                             column 128 = row sum l (all tiles),
//                             columns 129 / 130 = V-Smooth: the row sums of the
//                             even / odd tiles, accumulated (each in its own
//                             tile's frame; never rescaled, never written by
//                             the CUDA cores); 131-143 zero
//   A  [400,408) [408,416)    V-Smooth mean-term operands of the even / odd tiles
//                             (TF32, one element per column)
//   P0 [416,448) P1 [448,480) E4M3 probabilities, 4 codes per column (TS operand)
//   Q  [480,512)              E4M3 query tile (TS operand)
// Per KV tile t:
//   S_t  = Qq Kq_t^T                     kind::f8f6f4 TS, M=128 N=128 K=4x32
//   P_t  = E4M3 codes (exp2+cvt or ExpCast), written to TMEM by the softmax
//   O   += P_t [Vq_t ; 1 ; 1 ; 0]        kind::f8f6f4 TS, M=128 N=144 K=4x32:
//          the ones rows appended to the V tile make column 128 and column
//          129 + (t mod 2) accumulate the row sum of the DECODED codes
//   V-Smooth: the rank-one mean term of tile t-2 goes with tile t, issued right
//          behind PV_t (same frame), so that nobody waits for it: the group on
//          tile t, having seen PV_{t-2} complete (its P buffer wait), reads its
//          column (129 or 130) while its P stores land, takes r_{t-2} as the
//          difference to its previous reading (the column is never cleared: a
//          PV in flight rewrites all 144 columns, adding zero to the other
//          tiles' columns, so a clear could be lost), scales it to the frame
//          of m_t by 2^(m_{t-2} - m_t), writes A = [r_hi r_lo r_hi 0..] to TMEM
//          and B = [mu~_hi ; mu~_hi ; mu~_lo ; 0..] (mu~ = mu_{t-2} / s_v per
//          channel, both split into TF32 halves) to shared memory, and posts
//          them with P_t; O += A B is one kind::tf32 TS MMA, M=128 N=128 K=8,
//          committed with PV_t.  After the last tile group 0 adds the last two
//          tiles' terms in one more step.
// The row max is updated exactly at every tile.  On full tiles it comes with
// the score loads (tcgen05.ld.red.max returns the maximum of the columns it
// loads: one value per 64-key scale block); ragged tiles take it over their
// valid keys.  When it moves, the group on tile t rescales O in TMEM after
// PV_{t-1} completes (the 128 channels and the row-sum columns in use).
//
// Last-wave split (SPLIT with tail_cta0 >= 0): a query tile of the last wave
// runs as parts of its visiting order in separate CTAs; a part first takes
// max-only steps over the tiles before its range (K, QK, row max and hand-off;
// no P, no PV), so its running max, and with it every P code, is that of the
// unsplit order.  The parts are merged by log-sum-exp like split-KV parts.
//
// 4-bit PV variant (FP4; VC-Attention news article, 4-bit V-Smooth
// configuration: E2M1 values with a scale per 16 elements): V arrives as
// packed E2M1 (64-byte swizzled rows) with UE4M3 scales per (channel, 16
// tokens); the softmax writes P = 2688 * 2^(x - m) as E2M1 with one UE4M3
// scale per 16 keys to shared memory and the scales to TMEM, and
// O += P V runs as kind::mxf4nvf4 (two MMAs of K = 64 per tile).  The row sum
// is the sum of the decoded P, kept per softmax group in registers and merged
// at the end; with V-Smooth the mean term of tile t goes with PV_t.  TMEM:
// S0 S1 as above, O [256,384), P scales [384,448) (group g, k-step kk at
// 384 + 32 g + 16 kk), V scales [448,480), Q [480,512).
#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8attn {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;      // TMEM allocator and QK issuer
constexpr int kPvWarp = 10;      // PV (and V-Smooth mean) issuer
constexpr uint32_t kTileBytes = 128 * 128;               // one 128x128 E4M3 tile
constexpr uint32_t kVStageBytes = kTileBytes + 2048;     // V tile + 16-row ones block

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kMeanBuf = 4096;                              // 128 x 8 TF32, no swizzle
constexpr uint32_t kOffMeanA = kOffV + kStages * kVStageBytes;   // 2 buffers (flush parity)
constexpr uint32_t kOffMeanB = kOffMeanA + 2 * kMeanBuf;         // 2 buffers
constexpr uint32_t kOffMuSt = kOffMeanB + 2 * kMeanBuf;          // V-Smooth: bf16 block mean per V stage (256 B)
constexpr uint32_t kOffSacc = kOffMuSt + kStages * 256;          // 128 fp32 output channel scales
constexpr uint32_t kOffSoff = kOffSacc + 512;                    // 128 fp32 output offsets
constexpr uint32_t kOffMrow = kOffSoff + 512;                    // [2][128] fp32 running row max of the last 2 tiles
constexpr uint32_t kOffPrevC = kOffMrow + 1024;                  // [128] fp32 V-Smooth: group 1's last column reading
constexpr uint32_t kOffBar = kOffPrevC + 512;
constexpr int kNumBars = 2 + 4 * kStages + 5 * 2 + 3;   // one slot left unused
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;            // control block (16 ints), TMEM base
constexpr uint32_t kSmemUsed = kOffMisc + 80;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                // + alignment slack

// TMEM column map
constexpr uint32_t kColS = 0, kColO = 256, kColL = 256 + 128, kColR = 256 + 129, kColA = 400,
                   kColP = 416, kColQ = 480;
constexpr int kMaxRing = 2;       // running maxima kept in shared memory (tiles)

constexpr uint32_t kIdescQK = make_idesc(0, 128, 128);     // E4M3 x E4M3 -> F32, N=128
constexpr uint32_t kIdescPV = make_idesc(0, 128, 144);     // N=144: channels + ones rows
constexpr uint32_t kIdescMean = make_idesc(2, 128, 128);   // TF32 x TF32 -> F32

// 4-bit PV variant: V stages of 8 KB packed E2M1 + 1 KB block scales, and two
// 8 KB P buffers, inside the region the 8-bit V ring occupies.
constexpr uint32_t kVStage4 = 8192 + 1024;
constexpr uint32_t kOffP4 = kOffV + kStages * kVStage4;          // 2 x (128 rows x 64 B) E2M1 P
constexpr uint32_t kOffLx = kOffP4 + 2 * 8192;                   // [2][128] row sums, [2][128] their max
static_assert(kOffLx + 2048 <= kOffMeanA, "4-bit buffers fit in the 8-bit V ring");
static_assert(kOffV % 1024 == 0 && kOffP4 % 1024 == 0, "64-byte swizzled operands need aligned bases");
// 4-column scale blocks at 16-column aligned TMEM addresses
constexpr uint32_t kColPSF = 384, kColVSF = 448;
constexpr uint32_t kIdescPV4 = make_idesc_fp4(128, 128);
constexpr float kLog2Fp4Top = 11.392317422778761f;               // log2(6 x 448)

__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
  return make_sdesc(saddr, 16, 512, 4);     // 64-byte swizzle: rows of 64 B, 8-row atoms of 512 B
}

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

template <bool SPARSE>
struct TileList {
  const int32_t* col;
  int base, n, nV, reverse;
  int off, n_all;       // this CTA's part of the visiting order: positions [off, off + n) of n_all
  int* status;
  __device__ __forceinline__ int at(int it) const {
    const int pos = off + it;
    const int idx = reverse ? (n_all - 1 - pos) : pos;
    if (!SPARSE) return idx;
    int j = __ldg(col + base + idx);
    if (static_cast<unsigned>(j) >= static_cast<unsigned>(nV)) {
      atomicExch(status, kStatusBadTile);
      j = 0;
    }
    return j;
  }
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Warp-uniform bounded wait for the softmax warps: one test, then a vote, so
// every lane takes the same path and the warp-collective TMEM operations that
// follow stay convergent.  Returns false (for the whole warp) when it gave up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* ctl,
                                          uint64_t limit_ns, uint32_t tag) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const bool ok = mbar_wait_slow(bar, parity, ctl, limit_ns, tag);
  return __all_sync(0xffffffffu, ok);
}

// max of 64 fp32 values (raw bits) as a 3-ary tree: depth 4 instead of a
// 16-deep chain, so the warp does not wait on one max after another
__device__ __forceinline__ float max64(const uint32_t* v) {
  float a[22];
#pragma unroll
  for (int k = 0; k < 21; ++k)
    a[k] = fmax3(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]), __uint_as_float(v[3 * k + 2]));
  a[21] = __uint_as_float(v[63]);
  float b[8];
#pragma unroll
  for (int k = 0; k < 7; ++k) b[k] = fmax3(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
  b[7] = a[21];
  return fmax3(fmax3(b[0], b[1], b[2]), fmax3(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

// E4M3 codes of 4 consecutive scores (raw fp32 bits), packed little-endian.
// PCAST 0: exp2 + cvt.  PCAST 1 / 2: ExpCast, 2 when the top clamp at code
// 126 can be reached (8 log2 S + 56 + beta >= 126.5, i.e. S above ~430).
template <int PCAST>
__device__ __forceinline__ uint32_t pcast4(const uint32_t* s, float c, float bb) {
  const float2 c2 = make_float2(c, c), b2 = make_float2(bb, bb);
  const float2 f01 = ffma2(make_float2(__uint_as_float(s[0]), __uint_as_float(s[1])), c2, b2);
  const float2 f23 = ffma2(make_float2(__uint_as_float(s[2]), __uint_as_float(s[3])), c2, b2);
  if (PCAST == 0) {
    // exp2 + cvt: code = E4M3(S * 2^(y - m)), y = raw * c, bb = log2 S - m
    return cvt_e4m3x4(ex2_approx(f01.x), ex2_approx(f01.y), ex2_approx(f23.x), ex2_approx(f23.y));
  } else {
    // ExpCast: code = clamp(rne(8 (y - m + log2 S) + 56 + beta), 0, 126).  The
    // affine map is computed scaled by 2^-24 (c = 8 c_raw 2^-24, bb = (8 (log2 S
    // - m) + 56 + beta) 2^-24, exact power-of-two scalings): rounding that to
    // f16 lands on the subnormal grid k 2^-24, so the f16 bit pattern is the
    // integer code k, rounded to nearest even, and the relu conversion sends
    // every negative value to code 0.  Codes sit in bytes 0 and 2 of each pair.
    uint32_t h01 = cvt_relu_f16x2(f01.x, f01.y);
    uint32_t h23 = cvt_relu_f16x2(f23.x, f23.y);
    if (PCAST == 2) {
      // 126 is the largest finite E4M3 code (127 is NaN)
      h01 = min_u16x2(h01, 0x007E007Eu);
      h23 = min_u16x2(h23, 0x007E007Eu);
    }
    return prmt(h01, h23, 0x6420u);
  }
}

}  // namespace

template <int PCAST, bool VSMOOTH, bool SPARSE, bool SPLIT, bool FP4>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the last-wave split launch takes its query tiles from the linear CTA index
  const bool tail = SPLIT && p.tail_cta0 >= 0;
  const int lin = tail ? p.tail_cta0 + static_cast<int>(blockIdx.x) : 0;
  const int qt = tail ? lin % p.nQt : static_cast<int>(blockIdx.x);
  const int h = tail ? (lin / p.nQt) % p.H : static_cast<int>(blockIdx.y);
  const int b = tail ? lin / p.nQt / p.H
                     : (SPLIT ? static_cast<int>(blockIdx.z) / p.n_splits : static_cast<int>(blockIdx.z));
  const int split = SPLIT ? (tail ? static_cast<int>(blockIdx.z) : static_cast<int>(blockIdx.z) - b * p.n_splits) : 0;
  const int bh = b * p.H + h;
  // the plain launch leaves the query tiles of the last wave to the split launch
  if (!SPLIT && qt + p.nQt * (h + p.H * b) >= p.cta_limit) return;

  TileList<SPARSE> tl;
  tl.col = p.col;
  tl.nV = p.nV;
  tl.reverse = p.reverse;
  tl.status = p.status;
  if (SPARSE) {
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
  // split-KV: part `split` of n_splits holds visiting positions [lo, hi)
  tl.n_all = tl.n;
  tl.off = 0;
  if (SPLIT && tail) {
    tl.off = p.part_lo[split];
    tl.n = p.part_lo[split + 1] - tl.off;
  } else if (SPLIT) {
    tl.off = static_cast<int>((static_cast<long long>(split) * tl.n_all) / p.n_splits);
    tl.n = static_cast<int>((static_cast<long long>(split + 1) * tl.n_all) / p.n_splits) - tl.off;
  }
  const int n = tl.n;
  // a last-wave part first takes max-only steps over the positions before it
  // (K loads and QKs, the running max, no P, no PV), so that it enters its
  // range with the running max of the unsplit order and casts the unsplit P
  // codes.  Its start is a multiple of 4: the K and V rings then keep the
  // stage of every tile, and the two softmax groups keep their tiles' parity.
  // Steps: g = npre + t, t < 0 for the max-only ones.
  const int npre = tail ? tl.off : 0;
  const int nsteps = npre + n;

  const uint32_t bar0 = sb + kOffBar;
  const uint32_t q_full = bar0, q_tmem = bar0 + 8;
  auto k_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (2 + kStages + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + 2 * kStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (2 + 3 * kStages + s); };
  auto s_full = [&](int g) { return bar0 + 8 * (2 + 4 * kStages + g); };
  auto s_empty = [&](int g) { return bar0 + 8 * (4 + 4 * kStages + g); };
  auto p_full = [&](int g) { return bar0 + 8 * (6 + 4 * kStages + g); };
  auto o_done = [&](int g) { return bar0 + 8 * (8 + 4 * kStages + g); };
  const uint32_t m_done = bar0 + 8 * (10 + 4 * kStages);    // V-Smooth: group 1 finished (its last column reading)
  const uint32_t mma_drain = bar0 + 8 * (12 + 4 * kStages);
  const uint32_t o_final = bar0 + 8 * (13 + 4 * kStages);   // committed once after the last MMA
  const uint32_t qk_drain = bar0 + 8 * (14 + 4 * kStages);

  // control block: [0] abort flag, [1] first timed-out wait, [4 + warp] where each warp gave up
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 64);
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
    for (int g = 0; g < 2; ++g) {
      mbar_init(s_full(g), 1 + 128);   // QK commit + the other group's running max
      mbar_init(s_empty(g), 128);
      mbar_init(p_full(g), 128);
      mbar_init(o_done(g), 1);
    }
    mbar_init(mma_drain, 1);
    mbar_init(o_final, 1);
    mbar_init(qk_drain, 1);
    mbar_init(m_done, 128);

    for (int c = 0; c < 16; ++c) abort_flag[c] = 0;
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
    // ones block of every V stage s: row 0 (-> l) and row 1 + (s mod 2) (->
    // column 129 + (t mod 2), since stage s holds the tiles t = s mod 4) =
    // E4M3 1.0 (0x38) for all 128 keys, other rows 0 (2 KB per stage, 128 x
    // 16 B chunks, 8 per row)
    const int t = threadIdx.x;
    for (int q = t; !FP4 && q < kStages * 128; q += kThreads) {
      const int st = q >> 7, c = q & 127, r = c >> 3;
      const uint32_t w = (r == 0 || r == 1 + (st & 1)) ? 0x38383838u : 0u;
      *reinterpret_cast<uint4*>(smem + kOffV + st * kVStageBytes + kTileBytes + c * 16) =
          make_uint4(w, w, w, w);
    }
    // V-Smooth B operands: K slots 4..7 stay zero
    for (int q = t; VSMOOTH && !FP4 && q < 2 * kMeanBuf / 16; q += kThreads)
      reinterpret_cast<uint4*>(smem + kOffMeanB)[q] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // K_t then V_t for every tile of the visiting order (K only on the
    // max-only steps of a last-wave part), each after a wait for its ring
    // stage to be released (K stages free up after their QK, V stages after
    // their PV).  The waits suspend the warp in the barrier test,
    // so it takes no issue slots from the softmax warps of its sub-partition
    // (polling both rings without suspending was measured 2.5 % slower).  A
    // wait on a V stage can delay the next K load, but K loads are issued up
    // to four tiles before their QK, which covers it.  The whole warp runs the
    // loop; one elected lane issues each copy.
    int nk = 0, nv = 0;          // K / V loads issued
    if (elect_one()) {
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_4d(sb + kOffQ, &p.tm_q, q_full, 0, h, qt * kTile, b);
    }
    __syncwarp();
    for (int g = 0; g < nsteps; ++g) {
      const int st = g % kStages;              // = t mod 4 (npre is a multiple of 4)
      const int t = g - npre;
      const int j = tl.at(t);
      if (!warp_wait(k_empty(st), ((g / kStages) & 1) ^ 1, abort_flag, to, (3u << 24) | (1u << 16) | g)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(k_full(st), kTileBytes);
        tma_load_4d(sb + kOffK + st * kTileBytes, &p.tm_k, k_full(st), 0, h, j * kTile, b);
      }
      __syncwarp();
      ++nk;
      if (SPLIT && t < 0) continue;            // max-only step: no V
      if (!warp_wait(v_empty(st), ((t / kStages) & 1) ^ 1, abort_flag, to, (3u << 24) | (2u << 16) | t)) break;
      if (elect_one()) {
        if (FP4) {
          const uint32_t vst = sb + kOffV + st * kVStage4;
          mbar_arrive_expect_tx(v_full(st), kVStage4);
          tma_load_3d(vst, &p.tm_v, v_full(st), j * (kTile / 2), 0, bh);
          bulk_g2s(vst + 8192, p.v4_sf + ((size_t)bh * p.nV + j) * 1024, 1024, v_full(st));
        } else if (VSMOOTH && t >= 2) {
          // with V_t, the block mean of tile t-2 (its mean term goes with PV_t)
          mbar_arrive_expect_tx(v_full(st), kTileBytes + 256);
          tma_load_3d(sb + kOffV + st * kVStageBytes, &p.tm_v, v_full(st), j * kTile, 0, bh);
          bulk_g2s(sb + kOffMuSt + st * 256, p.v_mean + ((size_t)bh * p.nV + tl.at(t - 2)) * kHeadDim, 256, v_full(st));
        } else {
          mbar_arrive_expect_tx(v_full(st), kTileBytes);
          tma_load_3d(sb + kOffV + st * kVStageBytes, &p.tm_v, v_full(st), j * kTile, 0, bh);
        }
      }
      __syncwarp();
      ++nv;
    }
    // Drain: every issued load must land before the CTA exits, whatever the
    // abort flag says.  A consumed phase tests complete at once.
    mbar_wait_drain(q_full, 0, to);
    for (int s = 0; s < kStages; ++s) {
      if (nk > s) mbar_wait_drain(k_full(s), ((nk - 1 - s) / kStages) & 1, to);
      if (nv > s) mbar_wait_drain(v_full(s), ((nv - 1 - s) / kStages) & 1, to);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ QK issuer
    // QK_j is issued as soon as K_j has landed and the score buffer of its
    // group is free (the group has loaded S_{j-2}), so score tiles run ahead
    // of the softmax.  QKs and PVs come from two warps: a tcgen05.mma stalls
    // its issuing warp while the tensor pipe is busy, and a QK issued ahead
    // must not hold back the PV that the softmax is waiting for.
    // Warp-wide loop; one elected lane issues.  Stage descriptors differ only
    // in the start-address field (16-byte units).
    const uint64_t kdesc0 = sw128_desc(sb + kOffK);
    const uint32_t tq = tmem + kColQ;
    bool ok = warp_wait(q_tmem, 0, abort_flag, to, (2u << 24) | (1u << 16));
    tc_fence_after();
    for (int qk = 0; ok && qk < nsteps; ++qk) {
      const int st = qk % kStages;
      const int g = qk & 1;
      if (!warp_wait(k_full(st), (qk / kStages) & 1, abort_flag, to, (2u << 24) | (2u << 16) | qk)) break;
      if (!warp_wait(s_empty(g), ((qk >> 1) & 1) ^ 1, abort_flag, to, (2u << 24) | (3u << 16) | qk)) break;
      tc_fence_after();
      const uint32_t ts = tmem + kColS + g * 128;
      const uint64_t kd = kdesc0 + static_cast<uint64_t>(st * (kTileBytes >> 4));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8_ts(ts, tq + kk * 8, kd + 2 * kk, kIdescQK, kk > 0);
        mma_commit(s_full(g));
        mma_commit(k_empty(st));
      }
      __syncwarp();
    }
    // all issued QKs must finish before TMEM is released
    if (elect_one()) mma_commit(qk_drain);
    __syncwarp();
    mbar_wait_drain(qk_drain, 0, to);
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // PV_j as soon as its group has written P_j (and V_j has landed).  With
    // V-Smooth the mean term of tile t-2, posted with P_t, goes right after
    // PV_t, and one extra step after the last tile (posted by group 0) adds
    // those of the last two.
    // PVs are issued strictly in order, which keeps every barrier within one
    // phase of its waiters: a group's next p_full needs o_done of its previous
    // tile, and PV_{j+1} (hence o_done of the other group) is issued only
    // after the group that rescales on o_done_j has posted p_full_{j+1}.
    const uint64_t vdesc0 = sw128_desc(sb + kOffV);
    const uint64_t mean_a0 = plain_desc(sb + kOffMeanA), mean_b0 = plain_desc(sb + kOffMeanB);
    const uint32_t to_ = tmem + kColO;
    // V-Smooth's extra step: group 0's next step after the last tile (even)
    const int pv_final = (VSMOOTH && !FP4 && n >= 1) ? n + (n & 1) : -1;
    const int steps = n + (pv_final >= 0 ? 1 : 0);
    for (int step = 0; step < steps; ++step) {
      const int pv = step < n ? step : pv_final;
      if (!warp_wait(p_full(pv & 1), (pv >> 1) & 1, abort_flag, to, (2u << 24) | (4u << 16) | pv)) break;
      const int st = pv % kStages;
      if (pv < n && !warp_wait(v_full(st), (pv / kStages) & 1, abort_flag, to, (2u << 24) | (5u << 16) | pv)) break;
      tc_fence_after();
      const uint64_t moff = static_cast<uint64_t>((pv & 1) * (kMeanBuf >> 4));
      const uint32_t tp = tmem + kColP + (pv & 1) * 32;
      const uint64_t vd = vdesc0 + static_cast<uint64_t>(st * (kVStageBytes >> 4));
      if (FP4) {
        if (elect_one()) {
          // this tile's V block scales into TMEM (a later copy overwrites them only
          // after these MMAs: tcgen05 copies and MMAs of one thread run in order)
          const uint32_t vst = sb + kOffV + st * kVStage4;
          tmem_cp_warpx4(tmem + kColVSF, make_sdesc(vst + 8192, 16, 128, 0));
          tmem_cp_warpx4(tmem + kColVSF + 16, make_sdesc(vst + 8192 + 512, 16, 128, 0));
          if (VSMOOTH) mma_tf32(to_, mean_a0 + moff, mean_b0 + moff, kIdescMean, pv > 0 ? 1u : 0u);
          const uint64_t pd = sw64_desc(sb + kOffP4 + (pv & 1) * 8192), vd4 = sw64_desc(vst);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_fp4_ss(to_, pd + 2 * kk, vd4 + 2 * kk, kIdescPV4, tmem + kColPSF + (pv & 1) * 32 + 16 * kk,
                       tmem + kColVSF + 16 * kk, (pv > 0 || VSMOOTH || kk > 0) ? 1u : 0u);
          mma_commit(v_empty(st));
          mma_commit(o_done(pv & 1));
        }
        __syncwarp();
        continue;
      }
      auto mean_mma = [&](uint32_t bsel) {
        mma_tf32_ts(to_, tmem + kColA + 8 * bsel, mean_b0 + static_cast<uint64_t>(bsel * (kMeanBuf >> 4)),
                    kIdescMean, 1);
      };
      if (elect_one()) {
        // after the last tile: the terms of the last two (A columns 400-407, B buffer 0)
        if (VSMOOTH && pv == pv_final) mean_mma(0);
        if (pv < n) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_ts(to_, tp + kk * 8, vd + 2 * kk, kIdescPV, (pv > 0 || kk > 0) ? 1u : 0u);
          mma_commit(v_empty(st));
          // the mean term of tile pv-2 (posted with P_pv, same frame)
          if (VSMOOTH && pv >= 2) mean_mma(static_cast<uint32_t>(pv & 1));
          mma_commit(o_done(pv & 1));
        }
      }
      __syncwarp();
    }
    // the epilogue waits on this single-use barrier (no phase aliasing).  Every
    // QK has completed before its scores were read, which precedes the PV of
    // the same tile, so this commit covers the last MMA of the CTA.  Then all
    // issued PVs must finish before TMEM is released.
    if (elect_one()) {
      mma_commit(o_final);
      mma_commit(mma_drain);
    }
    __syncwarp();
    mbar_wait_drain(mma_drain, 0, to);
  } else {
    // ------------------------------------------------------------ softmax groups
    const int wq = warp & 3, grp = warp >> 2;
    const int i = wq * 32 + lane;                      // query row within the tile
    const int row = qt * kTile + i;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    const uint32_t tS = tmem + lane_base + kColS + grp * 128;
    const uint32_t tP = tmem + lane_base + kColP + grp * 32;
    const float sq = row < p.T ? __ldg(p.q_scale + (size_t)bh * p.nQK + row / kQKBlock) : 0.f;
    // output channel scale of channel i and (group 0) its output offset
    // (sequence-mean smoothing of V / bias correction): loaded after the
    // CTA-wide barrier and used after the Q tile has gone to TMEM, so that
    // their latency overlaps that of the Q tile
    const float sv_i = __ldg(p.v_scale + (size_t)bh * kHeadDim + i);
    const float off_i = (grp == 0 && p.v_offset) ? __ldg(p.v_offset + (size_t)bh * kHeadDim + i) : 0.f;
    // raw score -> log2-domain logit, without the key-block scale
    const float cq = sq * p.sm_scale_log2;
    // ExpCast consumes 8 * logit * 2^-24 (see pcast4); per tile its offset is
    // (8 (log2 S - m) + 56 + beta) 2^-24 = kExpCastBase - m * 8 * 2^-24
    constexpr float kTiny = 5.9604644775390625e-8f;      // 2^-24
    constexpr float kCodeScale = PCAST == 0 ? 1.f : 8.f * kTiny;
    const float kExpCastBase = (8.f * p.log2_pscale + 56.f + p.beta) * kTiny;
    const float* kscale = p.k_scale + (size_t)bh * p.nQK;
    const uint16_t* vmean = reinterpret_cast<const uint16_t*>(p.v_mean) + (size_t)bh * p.nV * kHeadDim;
    float* mrow = reinterpret_cast<float*>(smem + kOffMrow);
    bool ok = true;

    // Q tile -> TMEM (TS operand of QK): group g copies codes 64g..64g+63 of row i
    ok = mbar_wait(q_full, 0, abort_flag, to, (1u << 24) | (grp << 20) | (6u << 16));
    if (__all_sync(0xffffffffu, ok)) {
      uint32_t qw[16];
      const uint8_t* qrow = smem + kOffQ + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + (((4 * grp + c) ^ (i & 7)) << 4));
        qw[4 * c] = v.x;
        qw[4 * c + 1] = v.y;
        qw[4 * c + 2] = v.z;
        qw[4 * c + 3] = v.w;
      }
      tmem_st16(tmem + lane_base + kColQ + 16 * grp, qw);
      tmem_wait_st();
    } else {
      ok = false;
    }
    tc_fence_before();
    mbar_arrive(q_tmem);
    // tile 0 has no previous running max: group 1 stands in for its hand-off
    if (grp == 1) mbar_arrive(s_full(0));
    // group 0 puts the output scales and offsets in shared memory for the epilogue
    const float sacc_i = sv_i > 0.f ? sv_i : 1.f;
    if (grp == 0) {
      s_acc[i] = sacc_i;
      reinterpret_cast<float*>(smem + kOffSoff)[i] = off_i;
    }
    const float inv_sacc = __fdiv_rn(1.f, sacc_i);
    float m_last = -INFINITY;        // running max at this group's latest tile

    // key-block scales of this group's first tile (then prefetched one tile ahead)
    float skn0 = 0.f, skn1 = 0.f;
    int jn = 0;
    if (grp < nsteps) {
      jn = tl.at(grp - npre);
      skn0 = __ldg(kscale + 2 * jn);
      skn1 = (2 * jn + 1 < p.nQK) ? __ldg(kscale + 2 * jn + 1) : 0.f;
    }

    // 4-bit PV: this group's running row sum of decoded P and the max it is framed in
    float l_run = 0.f, m_mine = -INFINITY;
    // V-Smooth: this group's column (129 + grp) at its last reading, and zero
    // K slots 4..7 of its A operand
    float prev_c = 0.f;
    if (VSMOOTH && !FP4) {
      const uint32_t z16[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (grp == 0) tmem_st16(tmem + lane_base + kColA, z16);
      tmem_wait_st();
    }

    auto tf32_split = [](float x, uint32_t* a) {          // V-Smooth: x -> [x_hi x_lo x_hi]
      const float xh = round_tf32(x);
      a[0] = __float_as_uint(xh);
      a[1] = __float_as_uint(round_tf32(x - xh));
      a[2] = a[0];
    };
    auto tf32_split_mu = [&](uint16_t mu_bits, float* b) {   // mu -> [mu~_hi mu~_hi mu~_lo]
      const float mu = __uint_as_float(static_cast<uint32_t>(mu_bits) << 16) * inv_sacc;
      const float mh = round_tf32(mu);
      b[0] = mh;
      b[1] = mh;
      b[2] = round_tf32(mu - mh);
    };
    for (int g = grp; ok && g < nsteps; g += 2) {
      const int t = g - npre;                   // < 0: a max-only step of a last-wave part
      float alpha = 1.f;
      uint16_t mu4 = 0;       // 4-bit PV with V-Smooth: the mean of this tile (latency hidden by the S wait)
      if (FP4 && VSMOOTH && t < n) mu4 = __ldg(vmean + (size_t)tl.at(t) * kHeadDim + i);
      // V-Smooth: the mean term of tile t-2 goes with this tile
      const bool vs_term = VSMOOTH && !FP4 && t >= 2;
      const float m_prev_own = m_last;            // this group's running max at tile t-2
      uint32_t col_raw = 0u;                      // V-Smooth column reading (loaded below)
      float vs_scale = 1.f;                       // V-Smooth: 2^(m_{t-2} - m_t)
      if (t < n) {
        const int j = jn;
        const float c0 = cq * skn0, c1 = cq * skn1;
        const int kv_valid = min(kTile, p.T - j * kTile);

        if (!warp_wait(s_full(grp), (g >> 1) & 1, abort_flag, to, (1u << 24) | (grp << 20) | (1u << 16) | g)) { ok = false; break; }
        tc_fence_after();
        // the key scales of this group's next tile, issued after the wait so that
        // they stay off the path from the previous tile's p_full to this one
        if (t + 2 < n) {
          jn = tl.at(t + 2);
          skn0 = __ldg(kscale + 2 * jn);
          skn1 = (2 * jn + 1 < p.nQK) ? __ldg(kscale + 2 * jn + 1) : 0.f;
        }
        uint32_t sv[128];
        float mt;
        float bmx[8];          // 4-bit PV: maximum raw score of each 16-key scale block
        if constexpr (FP4) {
          // eight loads of 16 columns, each returning its scale block's maximum
#pragma unroll
          for (int q = 0; q < 8; ++q) bmx[q] = tmem_ld16_max(tS + 16 * q, sv + 16 * q);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(s_empty(grp));
          mt = fmaxf(fmax3(bmx[0], bmx[1], fmaxf(bmx[2], bmx[3])) * c0,
                     fmax3(bmx[4], bmx[5], fmaxf(bmx[6], bmx[7])) * c1);
          if (kv_valid < kTile) {
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e >= kv_valid) sv[e] = __float_as_uint(-INFINITY);
            mt = max64(sv) * c0;
            if (kv_valid > 64) mt = fmaxf(mt, max64(sv + 64) * c1);
          }
        } else {
          // the score row in two loads that also return the maximum of their 64
          // columns (a reducing TMEM load: the max costs no instructions); a
          // ragged tile recomputes it over its valid keys only
          const float m0 = tmem_ld64_max(tS, sv);
          const float m1 = tmem_ld64_max(tS + 64, sv + 64);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(s_empty(grp));
          mt = fmaxf(m0 * c0, m1 * c1);
          if (kv_valid < kTile) {
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e >= kv_valid) sv[e] = __float_as_uint(-INFINITY);
            mt = max64(sv) * c0;
            if (kv_valid > 64) mt = fmaxf(mt, max64(sv + 64) * c1);
          }
        }
        // running max: m_{t-1} comes from the other group, which published it
        // before the s_full phase of tile t could complete.  mrow keeps the
        // maxima of the last two tiles: the slot of tile u is read by the other
        // group at tile u + 1 (and by the final V-Smooth step for the last
        // tile of group 1) and rewritten only at tile u + 2, after the other
        // group's hand-off for tile u + 1
        const float mprev = g >= 1 ? mrow[((g - 1) & (kMaxRing - 1)) * 128 + i] : -INFINITY;
        const float m_new = fmaxf(mprev, mt);
        mrow[(g & (kMaxRing - 1)) * 128 + i] = m_new;
        if (t + 1 < n) mbar_arrive(s_full(grp ^ 1));   // hand-off to tile t+1 of the other group
        m_last = m_new;
        if (SPLIT && t < 0) continue;             // max-only step
        alpha = (mprev == m_new) ? 1.f : ex2_approx(mprev - m_new);
        // V-Smooth: the factor that moves the row sums of tile t-2 to this frame
        if (vs_term) vs_scale = ex2_approx(m_prev_own - m_new);

        const float bb = PCAST == 0 ? p.log2_pscale - m_new
                                    : fmaf(m_new, -8.f * kTiny, kExpCastBase);
        // the P buffer of this group was last read by PV_{t-2}: the 4-bit path
        // waits for it here, the 8-bit path after computing its codes
        auto p_buffer_free = [&]() {
          return t < 2 || warp_wait(o_done(grp), ((t - 2) >> 1) & 1, abort_flag, to,
                                    (1u << 24) | (grp << 20) | (3u << 16) | t);
        };
        if constexpr (FP4) {
          // P = 2688 * 2^(x - m) as E2M1 with one UE4M3 scale per 16 keys:
          // sf = UE4M3(max * fl32(1/6)), code = E2M1(p * fl32(1/sf)); codes to the
          // shared P buffer (64-byte swizzled row i), scales to TMEM (row i's
          // word in column slot + i / 32 of lane i).  All codes are computed
          // into registers first; the wait for the P buffer comes after them
          const float bb4 = kLog2Fp4Top - m_new;
          uint8_t* prow = smem + kOffP4 + grp * 8192 + i * 64;
          const int swz = (i >> 1) & 3;
          uint32_t sfw[2] = {0u, 0u};
          float rhat = 0.f;
          const bool ragged = kv_valid < kTile;        // uniform over the tile
          uint4 chunk[4];                              // the row's four 16-byte chunks
#pragma unroll
          for (int bp = 0; bp < 4; ++bp) {             // two 16-key blocks = one 16-byte chunk of the row
            const float ch = bp < 2 ? c0 : c1;
            uint32_t wd[4];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int blk = 2 * bp + hb;
              if (!ragged) {
                // full tile: the block's largest p is 2^(max_s * c + bb4) (c >= 0), and
                // p / sf = 2^(s * c + bb4 - log2 sf): one FFMA and one exp2 per key
                float sb16[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) sb16[e] = __uint_as_float(sv[16 * blk + e]);
                const float mx = bmx[blk];          // from the reducing load (full tiles only)
                const float a = ex2_approx(fmaf(mx, ch, bb4));
                const uint32_t sf = cvt_e4m3x2(__fmul_rn(a, __uint_as_float(0x3E2AAAABu)), 0.f) & 0xFFu;
                const float sfv = ue4m3_decode(sf);
                const float lsh = sfv > 0.f ? bb4 - __log2f(sfv) : -INFINITY;
                const float2 ch2 = make_float2(ch, ch), lsh2 = make_float2(lsh, lsh);
                float q[16];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  const float2 x2 = ffma2(make_float2(sb16[e], sb16[e + 1]), ch2, lsh2);
                  q[e] = ex2_approx(x2.x);
                  q[e + 1] = ex2_approx(x2.y);
                }
                wd[2 * hb] = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
                wd[2 * hb + 1] = e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
                const int s2 = e2m1x8_sum2(wd[2 * hb + 1], e2m1x8_sum2(wd[2 * hb], 0));
                rhat = fmaf(0.5f * static_cast<float>(s2), sfv, rhat);
                sfw[blk >> 2] |= sf << (8 * (blk & 3));
                continue;
              }
              float pr[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) pr[e] = ex2_approx(fmaf(__uint_as_float(sv[16 * blk + e]), ch, bb4));
              {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (16 * blk + e >= kv_valid) pr[e] = 0.f;
              }
              float a8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) a8[e] = fmaxf(pr[2 * e], pr[2 * e + 1]);
              const float a = fmaxf(fmax3(a8[0], a8[1], a8[2]), fmax3(fmax3(a8[3], a8[4], a8[5]), a8[6], a8[7]));
              const uint32_t sf = cvt_e4m3x2(__fmul_rn(a, __uint_as_float(0x3E2AAAABu)), 0.f) & 0xFFu;
              const float sfv = ue4m3_decode(sf);
              const float rs = sfv > 0.f ? __frcp_rn(sfv) : 0.f;
              wd[2 * hb] = e2m1x8(__fmul_rn(pr[0], rs), __fmul_rn(pr[1], rs), __fmul_rn(pr[2], rs), __fmul_rn(pr[3], rs),
                                  __fmul_rn(pr[4], rs), __fmul_rn(pr[5], rs), __fmul_rn(pr[6], rs), __fmul_rn(pr[7], rs));
              wd[2 * hb + 1] = e2m1x8(__fmul_rn(pr[8], rs), __fmul_rn(pr[9], rs), __fmul_rn(pr[10], rs),
                                      __fmul_rn(pr[11], rs), __fmul_rn(pr[12], rs), __fmul_rn(pr[13], rs),
                                      __fmul_rn(pr[14], rs), __fmul_rn(pr[15], rs));
              const int s2 = e2m1x8_sum2(wd[2 * hb + 1], e2m1x8_sum2(wd[2 * hb], 0));
              rhat = fmaf(0.5f * static_cast<float>(s2), sfv, rhat);
              sfw[blk >> 2] |= sf << (8 * (blk & 3));
            }
            chunk[bp] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          }
          if (!p_buffer_free()) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int bp = 0; bp < 4; ++bp) *reinterpret_cast<uint4*>(prow + ((bp ^ swz) << 4)) = chunk[bp];
          tmem_st1(tmem + lane_base + kColPSF + grp * 32 + wq, sfw[0]);
          tmem_st1(tmem + lane_base + kColPSF + grp * 32 + 16 + wq, sfw[1]);
          tmem_wait_st();
          l_run = (l_run > 0.f ? l_run * ex2_approx(m_mine - m_new) : 0.f) + rhat;
          m_mine = m_new;
          if (VSMOOTH) {
            // rank-one mean term of this tile, issued with PV_t (same frame)
            const float rh = round_tf32(rhat), rl = round_tf32(rhat - rh);
            const float mu = __uint_as_float(static_cast<uint32_t>(mu4) << 16) * inv_sacc;
            const float mh = round_tf32(mu), ml = round_tf32(mu - mh);
            uint8_t* ma = smem + kOffMeanA + (t & 1) * kMeanBuf;
            uint8_t* mb = smem + kOffMeanB + (t & 1) * kMeanBuf;
            *reinterpret_cast<float4*>(ma + plain_off(i, 0)) = make_float4(rh, rl, rh, 0.f);
            *reinterpret_cast<float4*>(ma + plain_off(i, 4)) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(mb + plain_off(i, 0)) = make_float4(mh, mh, ml, 0.f);
            *reinterpret_cast<float4*>(mb + plain_off(i, 4)) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          fence_proxy_async_smem();
        } else {
        // the codes of all 128 keys into registers first (the score registers
        // die as they are used), so that the wait for the P buffer overlaps
        // the cast, then the two 64-key halves to TMEM
        uint32_t pw[2][16];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float ch = (hf == 0 ? c0 : c1) * kCodeScale;
#pragma unroll
          for (int w = 0; w < 16; ++w) pw[hf][w] = pcast4<PCAST>(sv + 64 * hf + 4 * w, ch, bb);
          if (kv_valid < kTile) {
#pragma unroll
            for (int w = 0; w < 16; ++w) {
              const int nvk = kv_valid - 64 * hf - 4 * w;
              if (nvk <= 0) pw[hf][w] = 0u;
              else if (nvk < 4) pw[hf][w] &= (1u << (8 * nvk)) - 1u;
            }
          }
        }
        if (!p_buffer_free()) { ok = false; break; }
        tc_fence_after();
        // V-Smooth: the reading of this group's row-sum column for the term of
        // tile t-2 (PV_{t-2} has completed); the P stores below hide its latency
        if (vs_term) col_raw = tmem_ld1(tO + 129 + grp);
        tmem_st16(tP, pw[0]);
        tmem_st16(tP + 16, pw[1]);
        if (vs_term) {
          // ---- V-Smooth mean term of tile t-2, while the P stores land:
          // A = [r_hi r_lo r_hi 0] to TMEM, B = [mu~_hi ; mu~_hi ; mu~_lo ; 0]
          // (mu~ = mu / s_v) to shared memory, both posted with P_t.  The mean
          // came with V_t (V stage t mod 4), which has landed by now: the test
          // of its barrier passes at once
          if (!warp_wait(v_full(t % kStages), (t / kStages) & 1, abort_flag, to, (1u << 24) | (grp << 20) | (9u << 16) | t)) { ok = false; break; }
          const uint16_t mu_use = reinterpret_cast<const uint16_t*>(smem + kOffMuSt + (t % kStages) * 256)[i];
          tmem_wait_ld_dep(col_raw);
          const float c = __uint_as_float(col_raw);
          const float r = (c - prev_c) * vs_scale;
          prev_c = c;
          uint32_t a4[4];
          tf32_split(r, a4);
          a4[3] = 0u;
          tmem_st4(tmem + lane_base + kColA + 8 * grp, a4);
          float b4[4];
          tf32_split_mu(mu_use, b4);
          b4[3] = 0.f;
          *reinterpret_cast<float4*>(smem + kOffMeanB + grp * kMeanBuf + plain_off(i, 0)) =
              make_float4(b4[0], b4[1], b4[2], b4[3]);
          fence_proxy_async_smem();
        }
        }
      }

      // ---- O rescale (needs PV_{t-1}); the V-Smooth ring keeps its own frames
      const bool rescale = t >= 1 && t < n && __any_sync(0xffffffffu, alpha != 1.f);
      if (rescale) {
        if (!warp_wait(o_done(grp ^ 1), ((t - 1) >> 1) & 1, abort_flag, to, (1u << 24) | (grp << 20) | (4u << 16) | t)) { ok = false; break; }
        tc_fence_after();
        const float2 a2 = make_float2(alpha, alpha);
        // the 128 channels in four loads and the row sum l (the score row is
        // dead by now, so its registers hold them), one wait
        uint32_t vv[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tO + cc * 32, vv[cc]);
        uint32_t l1 = 0;
        if (!FP4) l1 = tmem_ld1(tO + 128);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 r2 = __fmul2_rn(make_float2(__uint_as_float(vv[cc][e]), __uint_as_float(vv[cc][e + 1])), a2);
            vv[cc][e] = __float_as_uint(r2.x);
            vv[cc][e + 1] = __float_as_uint(r2.y);
          }
          tmem_st32(tO + cc * 32, vv[cc]);
        }
        if (!FP4) tmem_st1(tO + 128, __float_as_uint(__uint_as_float(l1) * alpha));
        tmem_wait_st();
      }

      tmem_wait_st();                  // P (and the mean-term operand) stored
      tc_fence_before();
      mbar_arrive(p_full(grp));
    }
    // V-Smooth: group 0's extra step after the last tile (step n + (n & 1) of
    // the PV issuer): the mean terms of the last two tiles, with the post
    if (VSMOOTH && !FP4 && grp == 0 && n >= 1 && ok) {
      const int t = n + (n & 1);
      do {
        // after the last tile: tiles t0 (this group's last, even) and t1 (group
        // 1's last, odd), once PV_{n-1} has completed.  A parity wait is only
        // sound while its barrier is at most one phase behind the awaited one;
        // this group last waited for PV_{n-3} (n odd) or PV_{n-4} (n even), so
        // for n even PV_{n-2} comes first.
        if ((n & 1) == 0) {
          if (n >= 2 && !warp_wait(o_done(0), ((n - 2) >> 1) & 1, abort_flag, to, (1u << 24) | (7u << 16) | t)) { ok = false; break; }
          if (!warp_wait(o_done(1), ((n - 1) >> 1) & 1, abort_flag, to, (1u << 24) | (4u << 16) | t)) { ok = false; break; }
        } else {
          if (!warp_wait(o_done(0), ((n - 1) >> 1) & 1, abort_flag, to, (1u << 24) | (4u << 16) | t)) { ok = false; break; }
        }
        // group 1 is done: its last reading and running max are published
        if (!warp_wait(m_done, 0, abort_flag, to, (1u << 24) | (8u << 16) | t)) { ok = false; break; }
        tc_fence_after();
        const int t1 = (n & 1) ? n - 2 : n - 1;     // group 1's last tile (none if < 1)
        const float m0 = m_last;
        const float m1 = t1 >= 1 ? mrow[(t1 & (kMaxRing - 1)) * 128 + i] : -INFINITY;
        const float mref = fmaxf(m0, m1);          // = m_{n-1}
        const float c0 = __uint_as_float(tmem_ld1(tO + 129));
        const float c1 = __uint_as_float(tmem_ld1(tO + 130));
        tmem_wait_ld();
        uint32_t a8[8];
        float b8[8];
        const int t0 = (n & 1) ? n - 1 : n - 2;     // this group's last tile
        tf32_split((c0 - prev_c) * ex2_approx(m0 - mref), a8);
        tf32_split_mu(__ldg(vmean + (size_t)tl.at(t0) * kHeadDim + i), b8);
        if (t1 >= 1) {
          const float prev1 = reinterpret_cast<const float*>(smem + kOffPrevC)[i];
          tf32_split((c1 - prev1) * ex2_approx(m1 - mref), a8 + 3);
          tf32_split_mu(__ldg(vmean + (size_t)tl.at(t1) * kHeadDim + i), b8 + 3);
        } else {
          a8[3] = a8[4] = a8[5] = 0u;
          b8[3] = b8[4] = b8[5] = 0.f;
        }
        a8[6] = a8[7] = 0u;
        b8[6] = b8[7] = 0.f;
        tmem_st4(tmem + lane_base + kColA, *reinterpret_cast<uint32_t(*)[4]>(a8));
        tmem_st4(tmem + lane_base + kColA + 4, *reinterpret_cast<uint32_t(*)[4]>(a8 + 4));
        *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 0)) = make_float4(b8[0], b8[1], b8[2], b8[3]);
        *reinterpret_cast<float4*>(smem + kOffMeanB + plain_off(i, 4)) = make_float4(b8[4], b8[5], b8[6], b8[7]);
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(0));
      } while (0);
    }
    if (VSMOOTH && !FP4 && grp == 1 && n >= 1) {
      // for group 0's last step: this group's last column reading (its running
      // max of its last tile is in mrow)
      reinterpret_cast<float*>(smem + kOffPrevC)[i] = prev_c;
      mbar_arrive(m_done);
    }

    // ---- epilogue: group g writes output channels 64g..64g+63: O * s_acc / l -> bf16
    if (ok) {
      ok = mbar_wait(o_final, 0, abort_flag, to, (1u << 24) | (grp << 20) | (5u << 16) | n);
      ok = __all_sync(0xffffffffu, ok);
    }
    tc_fence_after();
    // the two softmax groups (warps 0-7): group 0's output scales and offsets
    // are visible to both
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const bool have = ok && n > 0;
    float l = 0.f;
    float m_fin4 = -INFINITY;
    if constexpr (FP4) {
      // merge the two groups' row sums in the frame of the final row max
      float* s_lx = reinterpret_cast<float*>(smem + kOffLx);
      s_lx[grp * 128 + i] = l_run;
      s_lx[256 + grp * 128 + i] = m_mine;
      asm volatile("bar.sync 1, 256;" ::: "memory");      // the two softmax groups (warps 0-7)
      const float l0 = s_lx[i], l1 = s_lx[128 + i], m0 = s_lx[256 + i], m1 = s_lx[384 + i];
      m_fin4 = fmaxf(m0, m1);
      l = (l0 > 0.f ? l0 * ex2_approx(m0 - m_fin4) : 0.f) + (l1 > 0.f ? l1 * ex2_approx(m1 - m_fin4) : 0.f);
      if (!have) l = 0.f;
    } else if (have) {
      l = __uint_as_float(tmem_ld1(tmem + lane_base + kColL));
      tmem_wait_ld();
    }
    const float inv_l = (l > 0.f) ? __fdiv_rn(1.f, l) : 0.f;
    const float* s_off = reinterpret_cast<const float*>(smem + kOffSoff);
    __nv_bfloat16* orow = p.out + (((size_t)b * p.T + row) * p.H + h) * kHeadDim + grp * 64;
    if (SPLIT) {
      // split-KV part: O_s = O * s_acc / l_s in fp32 plus (m_s, l_s); the final
      // running max is the larger of the two groups' latest (exchanged through
      // the idle V ring)
      float m_fin = -INFINITY;
      bool have_m = have;
      if (FP4) {
        m_fin = have ? m_fin4 : -INFINITY;
      } else {
        float* s_mx = reinterpret_cast<float*>(smem + kOffLx);
        s_mx[grp * 128 + i] = m_last;
        asm volatile("bar.sync 1, 256;" ::: "memory");      // the two softmax groups (warps 0-7)
        if (have_m) m_fin = fmaxf(s_mx[i], s_mx[128 + i]);
      }
      // partial rows: [part][B H][T], or [part][n_tail][128] for a last-wave launch
      const size_t prow = tail ? ((size_t)split * p.n_tail + blockIdx.x) * kTile + i
                               : ((size_t)split * p.B * p.H + bh) * p.T + row;
      float* po = p.part_o + prow * kHeadDim + grp * 64;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(tO + grp * 64 + cc * 32, v);
          tmem_wait_ld();
        }
        if (row < p.T) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (have_m && l > 0.f) {
              const int ch = grp * 64 + cc * 32 + 4 * q;
              o4 = make_float4(__uint_as_float(v[4 * q]) * s_acc[ch] * inv_l,
                               __uint_as_float(v[4 * q + 1]) * s_acc[ch + 1] * inv_l,
                               __uint_as_float(v[4 * q + 2]) * s_acc[ch + 2] * inv_l,
                               __uint_as_float(v[4 * q + 3]) * s_acc[ch + 3] * inv_l);
            }
            reinterpret_cast<float4*>(po + cc * 32)[q] = o4;
          }
        }
      }
      if (grp == 0 && row < p.T) p.part_ml[prow] = make_float2(m_fin, have_m ? l : 0.f);
    } else {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tO + grp * 64 + cc * 32, v);
        tmem_wait_ld();
      }
      if (row < p.T) {
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float o0 = 0.f, o1 = 0.f;
          if (have && l > 0.f) {
            const int ch = grp * 64 + cc * 32 + 2 * e;
            o0 = __uint_as_float(v[2 * e]) * s_acc[ch] * inv_l + s_off[ch];
            o1 = __uint_as_float(v[2 * e + 1]) * s_acc[ch + 1] * inv_l + s_off[ch + 1];
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
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && abort_flag[0]) {
    atomicExch(p.status, kStatusTimeout);
    // the first CTA to fail records where every warp was waiting (status word + 1..)
    int* diag = p.status + 1;
    if (atomicCAS(diag, 0, abort_flag[1] ? abort_flag[1] : 1) == 0) {
      diag[1] = static_cast<int>(blockIdx.x | (blockIdx.y << 16) | (blockIdx.z << 28));
      for (int w = 0; w < kThreads / 32; ++w) diag[2 + w] = abort_flag[4 + w];
    }
  }
}

size_t attn_smem_bytes() { return kSmemBytes; }

// Split-KV merge (log-sum-exp): one warp per output row, 4 channels per lane.
// With M the largest m_s over parts with l_s > 0 and w_s = l_s 2^(m_s - M)
// (m in the kernel's log2 logit units): O = sum_s w_s O_s / sum_s w_s, plus the
// output offset; a row with no key in any part stays 0.
__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ AttnParams p) {
  // launched as a programmatic dependent of the attention grid: its launch
  // overlaps that grid's tail, and this wait returns once the grid has
  // completed and its partial results are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const bool tail = p.tail_cta0 >= 0;
  const size_t stride = tail ? (size_t)p.n_tail * kTile : (size_t)p.B * p.H * p.T;   // rows per part
  const size_t g = (size_t)blockIdx.x * 8 + w;
  if (g >= stride) return;
  int bh, row;
  if (tail) {
    // row i of the k-th query tile of the last-wave launch
    const int k = static_cast<int>(g / kTile), lin = p.tail_cta0 + k;
    const int qt = lin % p.nQt;
    bh = lin / p.nQt;
    row = qt * kTile + static_cast<int>(g - (size_t)k * kTile);
    if (row >= p.T) return;
  } else {
    bh = static_cast<int>(g / p.T);
    row = static_cast<int>(g - (size_t)bh * p.T);
  }
  const int b = bh / p.H, h = bh - b * p.H;
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) {
    const float2 ml = p.part_ml[s * stride + g];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const float2 ml = p.part_ml[s * stride + g];
    if (!(ml.y > 0.f)) continue;
    const float ws = ml.y * exp2f(ml.x - M);
    const float4 o = reinterpret_cast<const float4*>(p.part_o + (s * stride + g) * kHeadDim)[l];
    acc.x += ws * o.x;
    acc.y += ws * o.y;
    acc.z += ws * o.z;
    acc.w += ws * o.w;
    den += ws;
  }
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (den > 0.f) {
    const float inv = __fdiv_rn(1.f, den);
    float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.v_offset) off = reinterpret_cast<const float4*>(p.v_offset + (size_t)bh * kHeadDim)[l];
    r = make_float4(acc.x * inv + off.x, acc.y * inv + off.y, acc.z * inv + off.z, acc.w * inv + off.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(r.x, r.y), hi = __floats2bfloat162_rn(r.z, r.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(p.out + (((size_t)b * p.T + row) * p.H + h) * kHeadDim)[l] = packed;
}

namespace {
template <int PCAST, bool VSMOOTH, bool SPARSE, bool SPLIT, bool FP4>
cudaError_t launch_one(const AttnParams& p, cudaStream_t stream) {
  static PerDeviceOnce once;
  auto kern = attn_fwd_kernel<PCAST, VSMOOTH, SPARSE, SPLIT, FP4>;
  const cudaError_t e0 = once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
  });
  if (e0 != cudaSuccess) return e0;
  const bool tail = SPLIT && p.tail_cta0 >= 0;
  const dim3 grid = tail ? dim3(p.n_tail, 1, p.n_splits) : dim3(p.nQt, p.H, p.B * p.n_splits);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(p);
  if (SPLIT) {
    const size_t rows = tail ? (size_t)p.n_tail * kTile : (size_t)p.B * p.H * p.T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_merge_kernel, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

template <int PCAST, bool VSMOOTH, bool SPARSE, bool FP4 = false>
cudaError_t launch_variant(const AttnParams& p, cudaStream_t stream) {
  return p.n_splits > 1 ? launch_one<PCAST, VSMOOTH, SPARSE, true, FP4>(p, stream)
                        : launch_one<PCAST, VSMOOTH, SPARSE, false, FP4>(p, stream);
}
}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t stream) {
  const bool sparse = p.row_ptr != nullptr;
  if (p.fp4) {       // 4-bit PV: exp2 P cast only
    if (p.vsmooth) return sparse ? launch_variant<0, true, true, true>(p, stream) : launch_variant<0, true, false, true>(p, stream);
    return sparse ? launch_variant<0, false, true, true>(p, stream) : launch_variant<0, false, false, true>(p, stream);
  }
  if (p.pcast == 0) {
    if (p.vsmooth) return sparse ? launch_variant<0, true, true>(p, stream) : launch_variant<0, true, false>(p, stream);
    return sparse ? launch_variant<0, false, true>(p, stream) : launch_variant<0, false, false>(p, stream);
  }
  if (p.pcast == 2) {   // ExpCast whose top clamp can be reached
    if (p.vsmooth) return sparse ? launch_variant<2, true, true>(p, stream) : launch_variant<2, true, false>(p, stream);
    return sparse ? launch_variant<2, false, true>(p, stream) : launch_variant<2, false, false>(p, stream);
  }
  if (p.vsmooth) return sparse ? launch_variant<1, true, true>(p, stream) : launch_variant<1, true, false>(p, stream);
  return sparse ? launch_variant<1, false, true>(p, stream) : launch_variant<1, false, false>(p, stream);
}

}  // namespace fp8attn
