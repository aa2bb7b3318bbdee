// Per-shape planner: which kernel, tile, split and workspace a GEMM uses,
// and which roof should bound it.
//
// The course pages pick launch shapes by hand ("Project - tiled matrix
// multiply": 16 x 16 blocks in "Stage 0", TILE x TILE blocks and a TILE 16
// vs 32 comparison in "Stage 2") and classify kernels as memory- or
// compute-bound by comparing arithmetic intensity with the ridge point
// ("Bandwidths and peak rate - exercises", exercise 3).  The planner does
// both per call: it sizes the grid against the SM count read from the
// device and classifies the shape with the ridge point of the mode's roof.
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "common.cuh"

namespace gg {

namespace {

// Planning constants.  The measured figures used for reporting come from
// the bench; these only steer choices.
constexpr double kPlanHbmBytesPerSec = 6.8e12;    // GB300 STREAM-like copy, order of magnitude
constexpr double kPlanTf32DenseFlops = 1.1e15;    // GB300 dense TF32 tensor rate, nominal
constexpr int kFp32LanesPerSm = 128;

bool mode_known(int mode) {
  switch (mode) {
    case GEMM_MODE_AUTO: case GEMM_MODE_FP32_SIMT: case GEMM_MODE_TF32X3: case GEMM_MODE_TF32:
    case GEMM_MODE_NAIVE: case GEMM_MODE_COALESCED: case GEMM_MODE_TILED16:
    case GEMM_MODE_TILED32:
      return true;
    default:
      return false;
  }
}

// Estimated time of the SIMT kernel with `split` K slices.  The CTAs spread
// evenly over the SMs; the busiest SM runs u = ceil(tiles * split / SMs)
// CTA-slices (1/split of the K loop each), in pairs at the full per-SM rate
// (about 70% of the FP32 peak) and a leftover single CTA at about 60% of
// it.  A split adds a reduction that reads the slices and writes C once
// (at ~6 TB/s, plus a launch and one L2 round trip per 8 slices).
double simt_time_estimate(int64_t M, int64_t N, int64_t K, int64_t tiles, int split, int64_t sms,
                          double fp32_peak, const SimtConfig &c) {
  const double rate = 0.7 * fp32_peak / (double)sms;
  const double slice_flops = 2.0 * c.bm * c.bn * (double)K / split;
  const int64_t u = ceil_div(tiles * split, sms);
  double t = (double)(u / 2) * 2.0 * slice_flops / rate + (double)(u % 2) * slice_flops / (0.6 * rate);
  // the reduction: its traffic, its launch, and for a small C ~0.75 us per
  // 8 slices (eight chains in flight per thread; fitted on GB300 to the best
  // slice counts of 32 x 32 x 65536, 64 x 64 x 8192, 128 x 128 x 4096 and
  // 128 x 128 x 16384)
  if (split > 1)
    t += (split + 1.0) * (double)M * (double)N * 4.0 / 6.0e12 + 2e-6 +
         std::ceil(split / 8.0) * 0.75e-6;
  return t;
}

void plan_simt(int64_t M, int64_t N, int64_t K, bool vec, const DeviceProps &dp,
               double fp32_peak, gemm_plan_t *out) {
  const int64_t sms = dp.sm_count > 0 ? dp.sm_count : 152;
  const SimtConfig c = simt_config();
  const int64_t tiles = ceil_div(M, c.bm) * ceil_div(N, c.bn);
  // Slices of at least 64 along K, at most 256: a small output with a long
  // K needs many slices to occupy the SMs (GB300, 32 x 32 x 65536: 16
  // slices 238 us, 128 slices 39 us; 64 x 64 x 8192: 37.0 -> 14.7 us), and
  // the reduction's cost in the estimate keeps large outputs at few slices.
  int64_t max_split = K / 64;
  if (max_split > 256) max_split = 256;
  if (max_split < 1) max_split = 1;
  int split = 1;
  double best = simt_time_estimate(M, N, K, tiles, 1, sms, fp32_peak, c);
  for (int s = 2; s <= max_split; ++s) {
    const double t = simt_time_estimate(M, N, K, tiles, s, sms, fp32_peak, c);
    if (t < 0.97 * best) {
      best = t;
      split = s;
    }
  }
  // Tuning knob: GEMM_SIMT_SPLIT=n forces n K slices (0 or unset: the estimate).
  if (const char *env = std::getenv("GEMM_SIMT_SPLIT")) {
    const int forced = std::atoi(env);
    if (forced >= 1) split = forced;
  }
  out->kernel = GEMM_KERNEL_SIMT;
  out->bm = c.bm;
  out->bn = c.bn;
  out->bk = c.bk;
  out->stages = 4;
  // Tuning knob: GEMM_SIMT_CONFIG="bk,stages" picks another built K depth and
  // ring length (ignored if it names none).
  if (const char *cfg = std::getenv("GEMM_SIMT_CONFIG")) {
    int bk = 0, st = 0;
    if (std::sscanf(cfg, "%d,%d", &bk, &st) == 2 && simt_config_valid(bk, st)) {
      out->bk = bk;
      out->stages = st;
    }
  }
  out->threads = c.threads;
  out->vec = vec ? 1 : 0;
  if (split > 1) {
    // round the slice depth to whole BK tiles, then recount the slices
    int64_t kps = ceil_div(ceil_div(K, split), out->bk) * out->bk;
    split = (int)ceil_div(K, kps);
  }
  out->split_k = split;
  out->launches = split > 1 ? 2 : 1;
  out->ctas_per_sm = 2;
  out->grid_ctas = tiles * split;
  out->workspace_bytes = split > 1 ? (uint64_t)split * (uint64_t)M * (uint64_t)N * 4u : 0;
}

}  // namespace

// Small 3xTF32 products that run fastest as one CTA per 128 x 64 tile, both
// operands pre-split, no stream-K: the tiles fit one wave, N > 64 and K is
// moderate against the tile count (K <= 2048 and K <= 16 per tile; with
// fewer tiles or a longer K, spreading K over more SMs wins).  GB300 step
// times, this / the stream-K plan (us): 512^3 13.7 / 15.4, 640^3 16.4 /
// 17.5, 768^3 20.1 / 21.9, 1024^3 23.7 / 26.4, 1200 x 640 x 336 15.1 / 20.0;
// A with lda not a multiple of 4: 1023 x 1025 x 777 35.0 / 37.6, 1000 x
// 1000 x 1001 30.5 / 37.0, 1200 x 640 x 333 16.9 / 20.9, 1024^2 x 1024
// 25.3 / 29.7, 900 x 1100 x 2000 42.9 / 43.6; outside the rule 1024^2 x
// 4096 70.8 / 50.4, 2048 x 1024 x 1024 41.7 / 28.5, 384 x 384 x 1024
// 20.5 us against 14.3 on the CUDA cores.
static bool small_tc_product(int64_t M, int64_t N, int64_t K, int64_t sms) {
  const int64_t tiles64 = ceil_div(M, 128) * ceil_div(N, 64);
  return N > 64 && K <= 2048 && K <= 16 * tiles64 && tiles64 <= sms;
}

// Shapes the tensor-core path takes: the split pre-passes tile K in 32-deep
// rows of a grid's y dimension, and TMA tile coordinates are 32-bit.
static bool tc_shape_fits(int64_t M, int64_t N, int64_t K) {
  const int64_t lim = ((int64_t)1 << 31) - 512;
  return ceil_div(K, 32) <= 65535 && M < lim && N < lim && K < lim;
}

int make_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
              int mode, uintptr_t align_hint, int beta_nonzero, const DeviceProps &dp,
              gemm_plan_t *out, int ta, int tb) {
  if (!out || !mode_known(mode) || M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  // stored widths: A is M x K (K x M when ta), B is K x N (N x K when tb)
  const int64_t a_cols = ta ? M : K, b_cols = tb ? K : N;
  if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) ||
      ldc < (N > 1 ? N : 1))
    return GEMM_ERR_INVALID_ARG;
  gemm_plan_t p{};
  p.split_k = 1;
  p.stages = 1;
  p.flops = 2.0 * (double)M * (double)N * (double)K;
  p.bytes = 4.0 * ((double)M * K + (double)K * N + (double)M * N * (beta_nonzero ? 2.0 : 1.0));
  p.intensity = p.bytes > 0 ? p.flops / p.bytes : 0.0;
  const double fp32_peak = (double)(dp.sm_count > 0 ? dp.sm_count : 152) * kFp32LanesPerSm *
                           2.0 * (double)dp.clock_khz * 1e3;

  int resolved = mode;
  if (mode == GEMM_MODE_AUTO) {
    // Tensor cores (3xTF32) once the problem amortises the split pass and
    // the extra launches; the CUDA-core kernel for small problems, short K
    // (both paths are then bound by writing C and within a few percent) and
    // fewer than 128 rows (half of every 128-row tile would idle).  GB300
    // step times, CUDA cores / 3xTF32 (us): 512^3 16.5 / 15.6-19.1, 576^3
    // 20.6 / 19.8, 640^3 22.4 / 17.3, 1023 x 1025 x 777 55.4 / 29.3, 1024^3
    // 61.9 / 26.0, 2048 x 2048 x 512 100.5 / 32.0, 4096 x 64 x 4096
    // 100.5 / 33.3; 4096^2 x 64 71.8 / 75.8, 1024^2 x 128 14.4 / 15.9,
    // 64 x 4096 x 4096 53.3 / 65.2.  A tiny C (at most 256 x 256) with K up
    // to 16384 stays on the CUDA cores too: split K across ~70 slices there
    // fills the SMs where stream-K has only a few tiles to share (128 x 128 x
    // 16384 22.6 / 51.2, 256 x 256 x 4096 18.6 / 32.9, 128 x 512 x 8192
    // 28.8 / 42.9; 128 x 1024 x 8192 47.3 / 43.0, 256 x 256 x 65536
    // 172 / 123).
    const bool tiny_c = (double)M * (double)N <= 65536.0 && K <= 16384;
    // (from 1.2e8 multiply-adds for the small products above: 512^3 13.7
    // us against 14.4 on the CUDA cores, 768 x 768 x 256 10.6 / 14.4, 512 x
    // 2048 x 128 10.5 / 12.3; 256 x 1024 x 512 14.3 / 14.4)
    const int64_t sms0 = dp.sm_count > 0 ? dp.sm_count : 152;
    const double mnk = (double)M * N * K;
    const bool big = (mnk >= 2.0e8 || (mnk >= 1.2e8 && small_tc_product(M, N, K, sms0))) &&
                     K >= 128 && M >= 128 && !tiny_c;
    resolved = (tc_supported(dp) && big && tc_shape_fits(M, N, K)) ? GEMM_MODE_TF32X3
                                                         : GEMM_MODE_FP32_SIMT;
  }
  p.mode = resolved;

  if (M == 0 || N == 0) {
    p.kernel = GEMM_KERNEL_NONE;
    *out = p;
    return GEMM_OK;
  }
  if (K == 0) {
    p.kernel = GEMM_KERNEL_SCALE;
    p.launches = 1;
    p.threads = 256;
    p.grid_ctas = ceil_div(M * N, 256);
    p.bound = GEMM_BOUND_HBM;
    *out = p;
    return GEMM_OK;
  }

  const bool vec = (lda % 4 == 0) && (ldb % 4 == 0) && (ldc % 4 == 0) && ((align_hint & 15) == 0);
  // The teaching kernels take the course page's plain row-major operands only.
  const bool ladder = resolved == GEMM_MODE_NAIVE || resolved == GEMM_MODE_COALESCED ||
                      resolved == GEMM_MODE_TILED16 || resolved == GEMM_MODE_TILED32;
  if (ladder && (ta || tb)) return GEMM_ERR_UNSUPPORTED;
  switch (resolved) {
    case GEMM_MODE_NAIVE:
    case GEMM_MODE_COALESCED: {
      p.kernel = resolved == GEMM_MODE_NAIVE ? GEMM_KERNEL_NAIVE : GEMM_KERNEL_COALESCED;
      p.launches = 1;
      p.bm = p.bn = 16;
      p.threads = 256;
      const int64_t gy = resolved == GEMM_MODE_NAIVE ? ceil_div(N, 16) : ceil_div(M, 16);
      if (gy > 65535) return GEMM_ERR_UNSUPPORTED;
      p.grid_ctas = ceil_div(M, 16) * ceil_div(N, 16);
      break;
    }
    case GEMM_MODE_TILED16:
    case GEMM_MODE_TILED32: {
      const int t = resolved == GEMM_MODE_TILED16 ? 16 : 32;
      p.kernel = GEMM_KERNEL_TILED;
      p.launches = 1;
      p.bm = p.bn = p.bk = t;
      p.threads = t * t;
      if (ceil_div(M, t) > 65535) return GEMM_ERR_UNSUPPORTED;
      p.grid_ctas = ceil_div(M, t) * ceil_div(N, t);
      break;
    }
    case GEMM_MODE_FP32_SIMT:
      if (ceil_div(M, 64) > 65535) return GEMM_ERR_UNSUPPORTED;
      plan_simt(M, N, K, vec, dp, fp32_peak, &p);
      break;
    case GEMM_MODE_TF32X3:
    case GEMM_MODE_TF32: {
      if (!tc_supported(dp)) return GEMM_ERR_UNSUPPORTED;
      if (ceil_div(M, 128) > 65535 || !tc_shape_fits(M, N, K)) return GEMM_ERR_UNSUPPORTED;
      const bool x3 = resolved == GEMM_MODE_TF32X3;
      const int nprod = x3 ? 3 : 1;
      p.kernel = x3 ? GEMM_KERNEL_TC_TF32X3 : GEMM_KERNEL_TC_TF32;
      p.bm = 128;
      p.threads = 192;
      p.vec = vec ? 1 : 0;
      // A stored M x K and aligned for TMA (16-byte base, lda a multiple of
      // 4): the GEMM kernel reads FP32 A once and splits it on chip;
      // otherwise a pre-pass writes A_hi/A_lo (K-major) to the workspace.
      // B goes through the same pre-pass (transposed to K-major when stored
      // K x N) unless it is split on chip (b_tma below).
      const bool a_aligned = !ta && (lda % 4 == 0) && ((align_hint & 15) == 0);
      const int64_t sms = dp.sm_count > 0 ? dp.sm_count : 152;
      const int64_t tiles256 = ceil_div(M, 128) * ceil_div(N, 256);
      // 128 x 256 tiles once there are at least half a wave of them
      // (GB300, 3xTF32, N = K = 4096: M = 1024 150 us against 195 us with
      // 128 x 128 tiles, M = 2048 266 us against 336 us)
      // and for a long K, where the stream-K CTAs, at unrelated K positions,
      // stream their operands mostly from HBM and the larger tile moves
      // fewer bytes per product (1024 x 1024 x 16384: 154 us against 208 us;
      // at K = 8192 it is a wash: 1024 x 1024 x 8192 80 / 83 us, 512 x 2048
      // x 8192 130 / 116 us)
      // ... unless 256-column tiles would cover N with more than 1.25x the
      // columns 128-column tiles do (8192 x 384 x 8192: 512 columns of MMA
      // work for 384, 206 us against 185 us; 6144 x 640 x 2048 at 1.2x still
      // prefers the wide tile, 70.0 against 72.8 us).
      const bool wide = N > 128 && (tiles256 * 2 >= sms || K >= 16384) &&
                        4 * ceil_div(N, 256) * 256 <= 5 * ceil_div(N, 128) * 128;
      p.a_split_in_kernel = a_aligned ? 1 : 0;
      p.launches = 2;  // the split pass (A and B in one launch when both are split) and the GEMM
      bool no_stream_k = false;  // a configuration chosen to run one CTA per tile
      auto set = [&](int bn, int bk, int st, int cc, int bm = 128) {
        p.bm = bm; p.bn = bn; p.bk = bk; p.stages = st; p.b_concat = cc;
      };
      // 256 x 256 tiles (two 128-row accumulators sharing each B tile) halve
      // the operand bytes per MMA; they take pre-split operands.
      const int64_t tiles_m2 = ceil_div(M, 256) * ceil_div(N, 256);
      auto pre_split = [&]() { p.a_split_in_kernel = 0; };
      if (!x3) {
        // 1xTF32: one MMA per K step, so feeding operands is the limit.
        // Narrow B (HBM-bound on A): 128-row tiles with A split on chip, so A
        // is read once.  Wide: 256 x 256 tiles (GB300: 4096^3 kernel 176 us
        // against 241 us with 128 x 256 tiles, 8192^3 1.15 ms against
        // 1.87 ms) once there are half a wave of them; fewer go to 128 x 256
        // tiles (2048^3: 48.6 us against 60.1 us for 64 tiles of 256 x 256
        // shared out stream-K).  Otherwise 128 x 256 tiles, pre-split (the
        // on-chip split is the slower stage with a single MMA per K step:
        // 4096^3 380 us against 277 us).
        if (a_aligned && N <= 64) {
          set(64, 32, 4, 0);
        } else if (wide && 2 * tiles_m2 >= sms) {
          // BK = 16 with 6 stages is 1-3 % ahead of BK = 32 with 3 for K up
          // to ~6144 (4096^3 212-218 against 217-225 us, 8192 x 8192 x 2048
          // 382 against 392 us, 6144^3 equal), 10 % behind at 8192^3 (1468
          // against 1337 us)
          if (K >= 8192) set(256, 32, 3, 0, 256);
          else set(256, 16, 6, 0, 256);
          pre_split();
        } else {
          set(256, 16, 8, 0);
          pre_split();
        }
      } else if (!a_aligned && wide && tiles_m2 >= 4 * sms) {
        // A pre-split anyway and many tiles: 256 x 256 tiles (GB300, 8192^3:
        // kernel 3.03 ms against 3.31 ms for 128 x 256 tiles)
        set(256, 16, 3, 0, 256);
        pre_split();
      } else if (a_aligned) {
        // One CTA per SM leaves tensor memory for A_hi next to A_lo, so the
        // MMAs read only B from shared memory (GB300, interleaved runs: 4096^3
        // 469 vs 471 us, 6144^3 1.51 vs 1.53 ms; 128 x 128 tiles, where
        // shared memory is the limit: 1024 x 1024 x 8192 97 vs 117 us).  With
        // it the 128 x 256 tile also beats 256 x 256 tiles (pre-split A) at
        // every size measured: 8192^3 3.35 vs 3.54 ms, 6144^3 1.44 vs
        // 1.61 ms, 8192 x 4096 x 4096 902 vs 978 us.
        if (N <= 64) {
          // narrow: 2 CTAs per SM stream A; with few tiles (stream-K) one CTA
          // per SM with 6 stages halves the partial tiles (GB300, 1024 x 64 x
          // 8192: 38.2 -> 29.7 us, 2048 x 64 x 4096: 29.6 -> 25.7 us; equal
          // at 32-64 tiles, 204 against 271 us on 65536 x 64 x 4096)
          if (4 * ceil_div(M, 128) <= sms) set(64, 32, 6, 1);
          else set(64, 32, 3, 1);
        } else {
          if (wide) set(256, 16, 5, 0);
          else set(128, 32, 4, 1);
          p.a_hi_tmem = 1;
        }
      } else if (wide) {
        set(256, 16, 4, 0);
      } else {
        // Tiles filling at most half the SMs go stream-K (below); there one
        // CTA per SM with 6 stages beats two with 3 (the same bytes in
        // flight, half the partial tiles to sum): GB300, 1023 x 1025 x 777
        // (lda 777) 35.5 against 39.7 us.  More tiles keep two CTAs per SM,
        // so one CTA's epilogue overlaps the other's MMAs.
        const int64_t tiles128 = ceil_div(M, 128) * ceil_div(N, 128);
        if (2 * tiles128 <= sms) set(128, 16, 6, 1);
        else set(128, 16, 3, 1);
      }
      // small products: one CTA per 128 x 64 tile, no fix-up (small_tc_product).
      // Both operands pre-split, except for a shallow product with an
      // aligned A and at least 64 tiles: there A is split on chip (the
      // truncated split writes nothing back), 6 stages at one CTA per SM,
      // and the split pass only has B to do (GB300: 1200 x 640 x 336 15.3 ->
      // 13.5 us, 768^3 20.4 -> 19.0 us; 512^3, 32 tiles, 14.1 against 14.6
      // and 1024^3, K = 1024, 24.0 against 25.4 keep both pre-split).
      // With B split on chip as well (see b_tma below), an aligned A always
      // goes on chip too: the call is then one launch (GB300, step with the
      // pass(es) / one launch: B stored N x K 512^3 14.0 / 12.3 us, 640^3
      // 16.0 / 14.2, 1024^3 22.4 / 19.8; B stored K x N, transposed on chip,
      // 512^3 14.0 / 13.0, 768^3 19.2 / 16.9, 1024^3 23.9 / 20.8).
      const bool b_tma = (ldb % 4 == 0) && ((align_hint & 15) == 0);
      bool b_chip = tb || x3;
      if (const char *bs = std::getenv("GEMM_TC_BSPLIT")) b_chip = std::atoi(bs) != 0;  // tuning knob
      const bool b_aligned = b_chip && b_tma;
      if (x3 && small_tc_product(M, N, K, sms)) {
        if (a_aligned && (b_aligned || (K <= 768 && ceil_div(M, 128) * ceil_div(N, 64) >= 64))) {
          set(64, 32, 6, 1);
        } else {
          set(64, 32, 4, 1);
          pre_split();
        }
        p.a_hi_tmem = 0;
        no_stream_k = true;
      }
      // B aligned for TMA (16-byte base, ldb a multiple of 4) can be read as
      // stored and split on chip, so no pass handles B before the GEMM.
      // Stored N x K (K contiguous, the way the MMA reads it), the landed
      // tile is B_hi and B_lo is written beside it.  The split adds a read of
      // B and a write of B_lo to shared memory per stage, which the MMAs of
      // a long run of full tiles cannot spare: it is taken when the tiles
      // fit one wave without stream-K (decided below).  GB300, 3xTF32, step
      // time with the pass / on chip (us): 1200 x 640 x 336 13.0 / 10.5 (one
      // launch), 1024^3 23.2 / 22.5, 2048^3 68.5 / 65.8; 4096^3 (stream-K)
      // about equal with a kernel of 390-417 against 443 us, 8192^3
      // 3.30-3.42 against 3.47-3.67 ms.
      // Stored K x N, the converter warps also transpose it (an MMA reading
      // B N-contiguous, through the instruction descriptor's transpose bit,
      // left the kind::tf32 accumulator at zero on GB300); that pays for the
      // small-product tiles (128 x 64 x 32) with A split on chip as well, one
      // launch a call (GB300, with the pass / on chip: 512^3 14.0 / 13.1 us,
      // 1200 x 640 x 336 13.3 / 11.0, 768^3 18.9 / 16.9, 1024^3 23.9 /
      // 21.0), not for wider tiles (1536^3, 128 x 128 tiles, 34.9 / 39.3;
      // 2048^3 68.3 / 88.5) nor with A pre-split (512^3 14.0 / 14.6).
      const int ak = p.a_split_in_kernel ? (p.a_hi_tmem ? 2 : 1) : 0;
      p.b_split_in_kernel =
          (b_aligned && (tb || (p.bn == 64 && p.bk == 32 && ak != 0)) &&
           tc_config_valid(p.bm, p.bn, p.bk, p.stages, ak, p.b_concat, nprod, 1))
              ? 1
              : 0;
      bool b_forced = false;
      // Tuning knob: GEMM_TC_CONFIG="bn,bk,stages,a_split,b_concat" (128-row
      // tile), "bm,bn,bk,stages,a_split,b_concat" or
      // "bm,bn,bk,stages,a_split,b_concat,b_split" picks one of the built
      // configurations (ignored if it names none, or asks for an in-kernel
      // split of a misaligned operand, or of a B stored K x N in tiles other
      // than 64 x 32).  a_split: 0 pre-split, 1 on chip, 2 on chip with A_hi
      // kept in tensor memory; b_split: 1 on chip.
      if (const char *cfg = std::getenv("GEMM_TC_CONFIG")) {
        int v[7] = {0, 0, 0, 0, 0, 0, 0};
        const int n = std::sscanf(cfg, "%d,%d,%d,%d,%d,%d,%d", &v[0], &v[1], &v[2], &v[3],
                                  &v[4], &v[5], &v[6]);
        const int *c = n >= 6 ? v + 1 : v;
        const int bm = n >= 6 ? v[0] : 128;
        const int bsplit = n == 7 ? v[6] : 0;
        if (n >= 5 && tc_config_valid(bm, c[0], c[1], c[2], c[3], c[4], nprod, bsplit) &&
            (!c[3] || a_aligned) &&
            (!bsplit || (b_tma && (tb || (c[0] == 64 && c[1] == 32))))) {
          set(c[0], c[1], c[2], c[4], bm);
          p.a_split_in_kernel = c[3] != 0;
          p.a_hi_tmem = c[3] == 2;
          p.b_split_in_kernel = bsplit != 0;
          b_forced = n == 7;
        }
      }
      p.ctas_per_sm = tc_ctas_per_sm(p.bm, p.bn, p.bk, p.stages,
                                     p.a_split_in_kernel ? (p.a_hi_tmem ? 2 : 1) : 0, p.b_concat,
                                     nprod, p.b_split_in_kernel,
                                     dp.smem_per_sm > 0 ? dp.smem_per_sm : 233472);
      // Stream-K: when the tiles do not fill whole waves of resident CTAs,
      // launch one wave of persistent CTAs that take whole tiles in waves and
      // split the rest of the (tile, K block) work evenly (each at least 4 K
      // blocks); a fix-up kernel sums the parts of tiles shared between
      // CTAs, in CTA order.  Taken for HBM-bound shapes (idle SMs are lost
      // bandwidth), when the tiles fill at most half the SMs (one CTA per
      // tile is then bound by the latency of its own TMA loads, and more CTAs
      // per tile keep more loads in flight), and otherwise when a time model
      // says it pays.  Model: the tensor pipe of an SM at its dense rate,
      // CTAs sharing an SM sharing it; one CTA per tile takes
      // ceil(tiles / SMs) tile times (K blocks plus one epilogue), stream-K
      // spreads all K blocks over the SMs but drains up to two more partial
      // tiles per CTA, writes and re-reads one partial tile per part (about
      // G + shared tiles parts, ~6 TB/s, mostly through L2) and launches the
      // fix-up (~3 us).  GB300 step times, one CTA per tile / stream-K (us), 3xTF32:
      // 1023 x 1025 x 777 (lda 777) 54.7 / 43.5, (lda 780) 37.2 / 28.0,
      // 640^3 18.9 / 17.9, 1024^3 26.3 / 25.2, 256 x 4096 x 4096
      // 105.8 / 85.3, 128 x 128 x 16384 254 / 53, 1536^3 41.0 / 46.4,
      // 2048 x 2048 x 512 34.0 / 40.1, 2048^3 75.7 / 80.1, 3000^3 (lda 3003)
      // 258 / 284, 2560 x 2560 x 4096 256 / 192, 4096^3 513 / 460,
      // 2560 x 2560 x 1024 73.4 / 66.2, 6144 x 6144 x 2048 497 / 482,
      // 1024 x 4096 x 4096 143 / 169;
      // 1xTF32: 2048^3 74.5 / 64.7, 4096^3 244 / 249.
      {
        const int64_t tiles = ceil_div(M, p.bm) * ceil_div(N, p.bn);
        const int64_t slots = (int64_t)(p.ctas_per_sm > 0 ? p.ctas_per_sm : 1) * sms;
        const int64_t nkb = ceil_div(K, p.bk);
        const int64_t total = tiles * nkb;
        // at least 4 K blocks per CTA, and at most 64 CTAs per tile (the
        // fix-up sums up to 256 parts; a few tiles with a very long K, such
        // as 128 x 128 x 16384, then still spread over 64 SMs per tile)
        int64_t g = slots < total / 4 ? slots : total / 4;
        if (g > 64 * tiles) g = 64 * tiles;
        const char *sk = std::getenv("GEMM_TC_STREAMK");  // tuning knob: 0 off, 1 on
        const double roof = x3 ? kPlanTf32DenseFlops / 3.0 : kPlanTf32DenseFlops;
        const bool hbm_bound = p.intensity < roof / kPlanHbmBytesPerSec;
        const double t_kb = 2.0 * p.bm * p.bn * p.bk * nprod / (kPlanTf32DenseFlops / (double)sms);
        // draining one tile of accumulators to global memory (~32 GB/s an SM)
        const double t_epi = (double)p.bm * p.bn * 4.0 / 32.0e9;
        const int64_t waves_dp = ceil_div(tiles, sms);
        const double t_dp = (double)waves_dp * ((double)nkb * t_kb + t_epi);
        const int64_t shared = g > 0 && tiles > g ? tiles % g : tiles;
        const double t_sk = (double)ceil_div(total, sms) * t_kb +
                            (double)(tiles / (g > 0 ? g : 1) + 2) * t_epi +
                            2.0 * (double)(g + shared) * p.bm * p.bn * 4.0 / 6.0e12 + 3.0e-6;
        // (the half-a-wave shortcut is measured for 3xTF32; with a third of
        // the MMA work per tile, 1xTF32 follows the model: 1024^3 one CTA per
        // tile 25.6 us against 27.1 us, 1024 x 1024 x 4096 stream-K)
        bool want = (tiles % slots) != 0 && tiles < 8 * slots &&
                    (hbm_bound || (x3 && 2 * tiles <= sms) || t_sk < t_dp);
        if (no_stream_k) want = false;
        if (sk) want = std::atoi(sk) != 0;
        p.stream_k = (want && g >= 2) ? 1 : 0;
        p.grid_ctas = p.stream_k ? g : tiles;
        // B on chip only for one wave of whole tiles (see b_aligned above)
        if (!b_forced && (p.stream_k || tiles > slots) &&
            std::getenv("GEMM_TC_BSPLIT") == nullptr)
          p.b_split_in_kernel = 0;
        // no pass before the GEMM when both operands are split on chip
        if (p.a_split_in_kernel && p.b_split_in_kernel) p.launches = 1;
        if (p.stream_k) p.launches += 1;
      }
      p.workspace_bytes = tc_workspace_bytes(p, M, N, K);
      break;
    }
    default:
      return GEMM_ERR_INVALID_ARG;
  }

  // Governing roof: the ridge point of the mode's compute roof against HBM.
  double compute_roof = fp32_peak;
  int compute_bound = GEMM_BOUND_FP32;
  if (p.kernel == GEMM_KERNEL_TC_TF32X3) {
    compute_roof = kPlanTf32DenseFlops / 3.0;
    compute_bound = GEMM_BOUND_TF32X3;
  } else if (p.kernel == GEMM_KERNEL_TC_TF32) {
    compute_roof = kPlanTf32DenseFlops;
    compute_bound = GEMM_BOUND_TF32;
  }
  const double ridge = compute_roof / kPlanHbmBytesPerSec;
  p.bound = p.intensity < ridge ? GEMM_BOUND_HBM : compute_bound;
  *out = p;
  return GEMM_OK;
}

}  // namespace gg
