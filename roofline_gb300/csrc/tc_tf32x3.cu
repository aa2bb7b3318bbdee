// 3xTF32 GEMM on the tcgen05 tensor cores (sm_103a).
//
// The course page points at Tensor Cores as the last rung of the GEMM
// ladder and notes that letting cuBLAS use TF32 would beat the FP32 peak
// ("Project - tiled matrix multiply", sections "Stage 3 - the reference
// ceiling: cuBLAS" and "What comes next").  TF32 alone keeps only 11
// significant bits, so each FP32 operand x is split in two,
//     x_hi = tf32_trunc(x) (x's word with the low 13 mantissa bits cleared:
//                           exactly the TF32 value the MMA reads from x's
//                           own word, so an A tile can serve as A_hi as it
//                           lands),
//     x_lo = x - x_hi      (exact in FP32, |x_lo| < 2^-10 |x|; the MMA reads
//                           its leading 11 significant bits, which changes
//                           the product by less than 2^-20 of |x| |y|),
// and the product is formed from three TF32 MMAs accumulated in FP32:
//     A*B ~= A_hi*B_lo + A_lo*B_hi + A_hi*B_hi
// (the dropped A_lo*B_lo term is below 2^-20 of |A||B|).
//
// 1xTF32 mode issues only A_hi*B_hi, with x_hi rounded to nearest
// (tf32_rna), which halves its error against truncation.
//
// Kernel structure (192 threads per CTA; output tiles of BM = 128 or 256
// rows by BN columns; a 256-row tile is two 128-row halves, each with its
// own accumulator, sharing every B tile):
//   warp 0      TMA producer: one lane streams K-blocks of the operand tiles
//               into a STAGES-deep shared-memory ring (cp.async.bulk.tensor,
//               completion counted on per-stage mbarriers);
//   warp 1      allocates TMEM (the accumulators, plus the A_lo ring when A
//               is split on chip) and one lane issues tcgen05.mma
//               kind::tf32, committing each stage back to the producer when
//               its MMAs retire;
//   warps 2-5   (a) when A is split inside the kernel: compute each landed
//               FP32 A tile's lo part into a tensor-memory ring read by the
//               [a_tmem] form of the MMA (the landed tile itself is A_hi to
//               the MMA, or, when the CTA owns enough tensor memory, A_hi
//               goes to a second ring too), then release the stage to the
//               MMA warp; (b) epilogue: tcgen05.ld the accumulator rows,
//               apply C = alpha*acc + beta*C, store.
// A CTA walks a list of (tile, K-range) segments: whole tiles in waves, then
// an even share of the remaining tiles' K blocks (stream-K; see Walk), with
// the pipeline running across segment boundaries.
// Operands live in shared memory K-major with the TMA swizzle (64 B rows for
// BK = 16, 128 B rows for BK = 32), which is the layout the MMA's smem
// descriptors describe.  B stored K x N (N contiguous) is split by a pass
// that writes B_hi/B_lo transposed (N x K, K contiguous), or is read as it
// is and transposed and split on chip (BR = 2); B stored N x K is read as it
// is and split on chip like A (BR = 1).
//
// Every mbarrier wait is bounded by a %globaltimer deadline; on expiry the
// kernel records GEMM_ERR_DEVICE_TIMEOUT in a device status word, stops
// issuing work, waits (bounded) for the copies and MMAs it already issued,
// frees its TMEM and returns.
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "tc_common.cuh"

namespace gg {

using namespace tc;

namespace {

__device__ int g_tc_status;  // 0 = ok, else a GEMM_ERR_* code

// ------------------------------------------------------------------ the GEMM kernel

// BN: output columns per CTA.  BK: K depth of one stage (16 -> 64-byte
// swizzle, 32 -> 128-byte swizzle).  AK: A arrives raw (FP32) and the
// converter warps split it: the landed tile is A_hi to the MMA as it is (the
// MMA reads each word's leading 11 significant bits) and A_lo goes into a
// tensor-memory ring that the A_lo*B_hi MMA reads directly; otherwise A_hi
// and A_lo come pre-split from the workspace.  CONCAT: B_hi and B_lo sit
// next to each other in the stage, so A_hi*[B_hi | B_lo] is one MMA of width
// 2*BN into two accumulators that the epilogue adds.  BR: B arrives raw
// (FP32) too, so no pass splits B before the kernel.  BR = 1: B is stored
// N x K (K contiguous, as the MMA reads it); the landed tile is B_hi to the
// MMA as it is, and the converter warps write B_lo next to it (1xTF32:
// round B in place).  BR = 2: B is stored K x N; its BK x BN tile lands
// unswizzled in the B_hi buffer, the converter warps read it into
// registers, and after a barrier among themselves write it back K-major
// (B_hi, the raw values) with B_lo beside it.
template <int BM, int BN, int BK, int STAGES, int AK, bool CONCAT, int NPROD, int BR>
struct TcCfg {
  static_assert(NPROD == 3 || NPROD == 1, "3xTF32 or 1xTF32");
  static_assert(NPROD == 3 || !CONCAT, "1xTF32 has no B_lo to concatenate");
  static_assert(BM == 128 || (BM == 256 && AK != 2 && (AK || !CONCAT)),
                "a 256-row tile keeps A_hi in shared memory; concatenated B only with A split on chip");
  static_assert(AK >= 0 && AK <= 2 && (AK != 2 || NPROD == 3), "A_hi in TMEM is a 3xTF32 form");
  static_assert(BR >= 0 && BR <= 2 && (BR != 2 || NPROD == 3), "B transposed on chip is 3xTF32");
  static constexpr bool X3 = NPROD == 3;
  static constexpr int MH = BM / 128;  // 128-row halves, one accumulator each
  static constexpr int A_BYTES = BM * BK * 4;
  static constexpr int A_HALF_BYTES = 128 * BK * 4;
  static constexpr int B_BYTES = BN * BK * 4;
  static constexpr int A_SMEM = (AK || !X3) ? A_BYTES : 2 * A_BYTES;  // A (raw/hi) [+ A_lo]
  static constexpr int B_SMEM = X3 ? 2 * B_BYTES : B_BYTES;           // B_hi [+ B_lo]
  static constexpr int STAGE_BYTES = A_SMEM + B_SMEM;
  // bytes the TMA writes per stage (B_lo of a raw B is written on chip)
  static constexpr int TX_BYTES = A_SMEM + (BR ? B_BYTES : B_SMEM);
  static constexpr int ROW_BYTES = BK * 4;              // 64 or 128
  static constexpr uint32_t LAYOUT = ROW_BYTES == 128 ? 2u : 4u;
  static constexpr uint32_t SBO = 8 * ROW_BYTES;        // 8-row group stride
  static constexpr int ACC_HALF = CONCAT ? 2 * BN : BN;  // accumulator columns of one half
  static constexpr int ACC_COLS = MH * ACC_HALF;
  static constexpr int LO_COL0 = ACC_COLS;
  // A_lo ring: STAGES x BK columns for each 128-row half
  static constexpr int LO_RING = (AK && X3) ? STAGES * BK : 0;
  static constexpr int LO_COLS = MH * LO_RING;
  // AK == 2: the converters also put A_hi in a tensor-memory ring (the MMAs
  // read both A parts from TMEM; shared memory then carries only B)
  static constexpr bool HI_TMEM = AK == 2;
  static constexpr int HI_COL0 = LO_COL0 + LO_COLS;
  static constexpr int HI_COLS = HI_TMEM ? STAGES * BK : 0;
  // C_TMEM: with A pre-split the four epilogue warps have nothing to do while
  // the MMAs run, so for a whole tile with beta != 0 they copy C's old values
  // into tensor memory next to the accumulator; the epilogue then reads them
  // with it instead of from global memory after the last MMA.  Only where
  // the columns fit in 256 (two CTAs per SM keep their tensor memory).
  static constexpr int OLD_COL0 = HI_COL0 + HI_COLS;
  static constexpr bool C_TMEM = AK == 0 && OLD_COL0 + MH * BN <= 256;
  static constexpr int TMEM_NEED = OLD_COL0 + (C_TMEM ? MH * BN : 0);
  static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                   : TMEM_NEED <= 64  ? 64
                                   : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256
                                                      : 512;
  // epilogue staging: 32 rows x 16 floats per epilogue warp
  static constexpr int EPI_BYTES = 4 * 32 * 16 * 4;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + EPI_BYTES;
  static_assert(ROW_BYTES == 64 || ROW_BYTES == 128, "BK must be 16 or 32");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(!CONCAT || 2 * BN <= 256, "concatenated B must fit one MMA");
  static_assert(TMEM_NEED <= 512, "tensor memory");
};

// Epilogue store of one warp's 32 x 16 block: lane r holds v[0..15], row r,
// columns col0..col0+15, and dst points at row 0, column col0 of the block
// (row stride ld; rows and cols: how many of them lie inside the matrix).
// The block goes through the warp's 2 KB of shared memory (row r's 16-byte
// chunk k stored at chunk k ^ ((r >> 1) & 3), so both the row-per-lane
// writes and the reads below hit 32 distinct banks) and comes back out
// along rows: each store instruction covers 8 rows x 64 contiguous bytes
// (16-byte accesses) or 2 rows x 64 bytes (4-byte accesses, for an
// unaligned or clipped block), instead of 32 rows x 16 bytes.
// dst = alpha * v + beta * dst (beta == 0: dst is not read).
__device__ __forceinline__ void epi_store16(float4 *st, const float *v, float *dst, int64_t ld,
                                            int rows, int cols, bool vec, float alpha,
                                            float beta) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st[lane * 4 + (k ^ ((lane >> 1) & 3))] =
        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  __syncwarp();
  if (vec && cols >= 16) {
    float4 x[4], old[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 8 + (lane >> 2), k = lane & 3;
      x[it] = st[r * 4 + (k ^ ((r >> 1) & 3))];
      old[it] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (beta != 0.0f && r < rows)
        old[it] = *reinterpret_cast<const float4 *>(dst + (int64_t)r * ld + 4 * k);
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 8 + (lane >> 2), k = lane & 3;
      if (r < rows) {
        float4 o = make_float4(alpha * x[it].x, alpha * x[it].y, alpha * x[it].z, alpha * x[it].w);
        if (beta != 0.0f) {
          o.x = fmaf(beta, old[it].x, o.x);
          o.y = fmaf(beta, old[it].y, o.y);
          o.z = fmaf(beta, old[it].z, o.z);
          o.w = fmaf(beta, old[it].w, o.w);
        }
        *reinterpret_cast<float4 *>(dst + (int64_t)r * ld + 4 * k) = o;
      }
    }
  } else {
    // two passes of 16 rows: each issues its 8 reads of old values before
    // its first store, so a block costs two round trips to memory
    const float *sf = reinterpret_cast<const float *>(st);
    const int j = lane & 15;
    const int64_t ld2 = 2 * ld;
#pragma unroll 1
    for (int it0 = 0; it0 < 16; it0 += 8) {
      const int r0 = it0 * 2 + (lane >> 4);
      float *row0 = dst + (int64_t)r0 * ld + j;
      float old[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        old[u] = 0.0f;
        if (beta != 0.0f && r0 + 2 * u < rows && j < cols) old[u] = row0[u * ld2];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = r0 + 2 * u;
        if (r < rows && j < cols) {
          float o = alpha * sf[r * 16 + (((j >> 2) ^ ((r >> 1) & 3)) << 2) + (j & 3)];
          if (beta != 0.0f) o = fmaf(beta, old[u], o);
          row0[u * ld2] = o;
        }
      }
    }
  }
  __syncwarp();  // the buffer is rewritten by the next block
}

template <int BM, int BN, int BK, int STAGES, int AK, bool CONCAT, int NPROD, int BR>
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_tf32x3_kernel(const __grid_constant__ CUtensorMap tmA_hi,  // A fp32 when AK
                 const __grid_constant__ CUtensorMap tmA_lo,
                 const __grid_constant__ CUtensorMap tmB_hi,  // B fp32 as stored when BR
                 const __grid_constant__ CUtensorMap tmB_lo, TcParams p) {
  using Cfg = TcCfg<BM, BN, BK, STAGES, AK, CONCAT, NPROD, BR>;
  constexpr bool X3 = Cfg::X3;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t *conv = full + STAGES;    // A (AK) and B (BR) tiles split
  uint64_t *empty = conv + STAGES;   // stage free again
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 1;
  uint64_t *drain = acc_empty + 1;
  uint64_t *b_read = drain + 1;  // BR = 2: every converter thread has read the raw B tile
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(b_read + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  auto a_hi = [&](int s) { return smem + s * Cfg::STAGE_BYTES; };
  auto a_lo = [&](int s) { return smem + s * Cfg::STAGE_BYTES + Cfg::A_BYTES; };
  auto b_hi = [&](int s) { return smem + s * Cfg::STAGE_BYTES + Cfg::A_SMEM; };
  auto b_lo = [&](int s) { return smem + s * Cfg::STAGE_BYTES + Cfg::A_SMEM + Cfg::B_BYTES; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const uint64_t deadline = globaltimer() + p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], kConvThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kConvThreads);
    mbar_init(drain, 1);
    mbar_init(b_read, kConvThreads);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA_hi);
    prefetch_tmap(&tmB_hi);
    if (X3 && !BR) prefetch_tmap(&tmB_lo);
    if (!AK && X3) prefetch_tmap(&tmA_lo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // B_hi/B_lo (and A_hi/A_lo) come from the split kernels before this one
  grid_dependency_wait();
  // measurement aid: earliest start of any CTA (see gemm_set_profile_stamps)
  if (p.stamps != nullptr && threadIdx.x == 0) atomicMin(&p.stamps[0], globaltimer());

  bool ok = true;
  if (warp == 0) {
    // ---------------- TMA producer: every stage of every segment, in order
    int issued = 0;
    if (lane == 0 && !p.stall_producer) {
      Walk walk(p, blockIdx.x, G);
      Segment sg;
      while (ok && walk.next(p, sg)) {
        int64_t mt, nt;
        tile_coords(p, sg.tile, mt, nt);
        const int32_t m0 = (int32_t)(mt * BM);
        const int32_t n0 = (int32_t)(nt * BN);
        if (p.in_flag != nullptr) {
          // streaming: this tile's rows of A must have landed
          if (!flag_wait(p.in_flag + (mt * BM) / p.stream_rows, p.epoch, deadline, abort_flag)) {
            ok = false;
            break;
          }
          fence_async_global();
        }
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          const int s = issued % STAGES;
          const uint32_t ph = (uint32_t)(issued / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, deadline, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], Cfg::TX_BYTES);
          const int32_t kx = kb * BK;
          tma_load_2d(a_hi(s), &tmA_hi, &full[s], kx, m0);
          if (!AK && X3) tma_load_2d(a_lo(s), &tmA_lo, &full[s], kx, m0);
          if (BR == 2)
            tma_load_2d(b_hi(s), &tmB_hi, &full[s], n0, kx);  // BK rows of BN values
          else
            tma_load_2d(b_hi(s), &tmB_hi, &full[s], kx, n0);
          if (X3 && !BR) tma_load_2d(b_lo(s), &tmB_lo, &full[s], kx, n0);
          ++issued;
        }
      }
      if (!ok) *abort_flag = 1;
      // wait (bounded) for every load this lane issued, whatever happened
      const uint64_t drain_deadline = globaltimer() + 2000000000ull;
      volatile int never = 0;
      for (int it = issued - STAGES < 0 ? 0 : issued - STAGES; it < issued; ++it)
        mbar_wait(&full[it % STAGES], (uint32_t)(it / STAGES) & 1u, drain_deadline, &never);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(128, BN);
      constexpr uint32_t idesc2 = idesc_tf32(128, CONCAT ? 2 * BN : BN);
      bool any = false;
      int it = 0, si = 0;
      Walk walk(p, blockIdx.x, G);
      Segment sg;
      while (ok && walk.next(p, sg)) {
        if (si > 0) {
          // the epilogue must have drained the previous segment's accumulator
          if (!mbar_wait(acc_empty, (uint32_t)(si - 1) & 1u, deadline, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait((AK || BR) ? &conv[s] : &full[s], ph, deadline, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ah = smem_u32(a_hi(s)), al = smem_u32(a_lo(s));
          const uint32_t bh = smem_u32(b_hi(s)), bl = smem_u32(b_lo(s));
          const uint32_t lo_t0 = tmem_base + (uint32_t)(Cfg::LO_COL0 + s * BK);
          const uint32_t hi_t = tmem_base + (uint32_t)(Cfg::HI_COL0 + s * BK);
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint32_t off = kk * 32;  // 8 TF32 values = 32 bytes along K
            const uint64_t dbh = smem_desc(bh + off, Cfg::SBO, Cfg::LAYOUT);
            const uint32_t acc = (kb > sg.kb0 || kk > 0) ? 1u : 0u;
            // each 128-row half of the A tile feeds its own accumulator
#pragma unroll
            for (int h = 0; h < Cfg::MH; ++h) {
              const uint32_t ah_h = ah + h * Cfg::A_HALF_BYTES + off;
              const uint32_t al_h = al + h * Cfg::A_HALF_BYTES + off;
              const uint32_t d = tmem_base + (uint32_t)(h * Cfg::ACC_HALF);
              const uint32_t lo_t = lo_t0 + (uint32_t)(h * Cfg::LO_RING);
              const uint64_t dah = smem_desc(ah_h, Cfg::SBO, Cfg::LAYOUT);
              if (!X3) {
                mma_tf32(d, dah, dbh, idesc, acc);  // 1xTF32: A_hi * B_hi only
              } else if (CONCAT) {
                // columns [0, BN): A_hi*B_hi (+ A_lo*B_hi); [BN, 2BN): A_hi*B_lo
                if (Cfg::HI_TMEM)
                  mma_tf32_ts(d, hi_t + kk * 8, dbh, idesc2, acc);
                else
                  mma_tf32(d, dah, dbh, idesc2, acc);
                if (AK)
                  mma_tf32_ts(d, lo_t + kk * 8, dbh, idesc, 1u);
                else
                  mma_tf32(d, smem_desc(al_h, Cfg::SBO, Cfg::LAYOUT), dbh, idesc, 1u);
              } else {
                const uint64_t dbl = smem_desc(bl + off, Cfg::SBO, Cfg::LAYOUT);
                if (Cfg::HI_TMEM)  // small terms first
                  mma_tf32_ts(d, hi_t + kk * 8, dbl, idesc, acc);
                else
                  mma_tf32(d, dah, dbl, idesc, acc);
                if (AK)
                  mma_tf32_ts(d, lo_t + kk * 8, dbh, idesc, 1u);
                else
                  mma_tf32(d, smem_desc(al_h, Cfg::SBO, Cfg::LAYOUT), dbh, idesc, 1u);
                if (Cfg::HI_TMEM)
                  mma_tf32_ts(d, hi_t + kk * 8, dbh, idesc, 1u);
                else
                  mma_tf32(d, dah, dbh, idesc, 1u);
              }
            }
          }
          mma_commit(&empty[s]);
          any = true;
          ++it;
        }
        if (!ok) break;
        mma_commit(acc_full);
        ++si;
      }
      if (!ok) *abort_flag = 1;
      grid_launch_dependents();  // the fix-up may start launching
      if (any) {
        // every MMA issued so far must retire before TMEM is freed
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, globaltimer() + 2000000000ull, &never);
      }
    }
  } else {
    // ---------------- converters (AK) and epilogue, warps 2..5
    const int quarter = warp & 3;  // TMEM lanes this warp may touch
    const int row = quarter * 32 + lane;
    // this warp's epilogue staging buffer (after the barriers)
    float4 *epi = reinterpret_cast<float4 *>(reinterpret_cast<uint8_t *>(full) + 256) + quarter * 128;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
    int it = 0, si = 0;
    Walk walk(p, blockIdx.x, G);
    Segment sg;
    while (ok && walk.next(p, sg)) {
      if (p.beta != 0.0f && sg.kb0 == 0 && sg.kb1 == p.num_kb) {
        // A whole tile that reads C.  C_TMEM: lane r of this warp copies row
        // r of its 32 rows of the old C tile into tensor memory (columns
        // OLD_COL0 + h * BN ...; zeros outside the matrix).  Otherwise those
        // rows are requested into L2, so the epilogue's reads of the old
        // values hit L2 instead of waiting on DRAM after the last MMA.
        int64_t mt, nt;
        tile_coords(p, sg.tile, mt, nt);
        const int64_t left = p.N - nt * BN;
        const int ncols = left < BN ? (int)left : BN;
#pragma unroll 1
        for (int h = 0; h < Cfg::MH; ++h) {
          const int64_t r = mt * BM + h * 128 + quarter * 32 + lane;
          const float *row = p.C + r * p.ldc + nt * BN;
          if constexpr (Cfg::C_TMEM) {
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
              uint32_t v[32];
#pragma unroll
              for (int q = 0; q < 32; ++q)
                v[q] = (r < p.M && c + q < ncols) ? __float_as_uint(row[c + q]) : 0u;
              tmem_st<32>(lane_base + (uint32_t)(Cfg::OLD_COL0 + h * BN + c), v);
            }
          } else if (r < p.M) {
            for (int c = 0; c < ncols; c += 32) prefetch_l2(row + c);
            prefetch_l2(row + ncols - 1);
          }
        }
        if constexpr (Cfg::C_TMEM) tmem_st_wait();
      }
      if (AK || BR) {
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          // tcgen05.st below is warp-collective: the warp proceeds or stops as one
          if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, deadline, abort_flag))) {
            ok = false;
            break;
          }
          // BR = 2: the B tile landed as BK = 32 rows of BN = 64 values (row k
          // at k * 256 bytes).  Each converter thread takes one block of 4 k
          // x 4 n (n = 4 bjb.., k = 4 bc..) with four 128-bit loads, then
          // signals b_read and splits its rows of A while the others read.
          // A quarter warp (lanes l = ct & 7) reads 8 distinct 16-byte
          // columns bjb & 7 = l: no bank conflicts.
          float4 bv[4];
          int bjb = 0, bc = 0;
          if constexpr (BR == 2) {
            static_assert(BN == 64 && BK == 32 && kConvThreads == 128,
                          "one 4 x 4 block per converter thread");
            const int ct = (int)threadIdx.x - 64;
            const int l = ct & 7, g = ct >> 3;
            bjb = l + 8 * (g & 1);
            bc = ((g >> 1) + (l >> 1)) & 7;
            const float *raw = reinterpret_cast<const float *>(b_hi(s));
#pragma unroll
            for (int i = 0; i < 4; ++i)
              bv[i] = *reinterpret_cast<const float4 *>(raw + (4 * bc + i) * BN + 4 * bjb);
            mbar_arrive(b_read);
          }
          // Row `row` of each 128-row half of the landed tile: 16-byte
          // chunk c sits at chunk c ^ f(row) of its 64- or 128-byte line (the
          // TMA swizzle; f depends on the row's low bits only).
#pragma unroll 1
          for (int half = 0; half < (AK ? Cfg::MH : 0); ++half) {
          uint8_t *line = a_hi(s) + (half * 128 + row) * Cfg::ROW_BYTES;
          if constexpr (!X3) {
            // 1xTF32: round in place, nothing goes to tensor memory.  Chunks
            // are visited in swizzled order so a warp's 32 rows hit 32
            // different banks.
#pragma unroll
            for (int c = 0; c < BK / 4; ++c) {
              const int phys = (BK == 32) ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3));
              float4 *ptr = reinterpret_cast<float4 *>(line + phys * 16);
              float4 x = *ptr;
              x.x = tf32_rna(x.x);
              x.y = tf32_rna(x.y);
              x.z = tf32_rna(x.z);
              x.w = tf32_rna(x.w);
              *ptr = x;
            }
            fence_async_smem();
          } else {
            uint32_t lo[BK];
            uint32_t hi[BK];  // used (and kept in registers) only with A_hi in TMEM
#pragma unroll
            for (int c = 0; c < BK / 4; ++c) {
              const int phys = (BK == 32) ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3));
              float4 *ptr = reinterpret_cast<float4 *>(line + phys * 16);
              const float4 x = *ptr;
              float4 h;
              h.x = tf32_trunc(x.x);
              h.y = tf32_trunc(x.y);
              h.z = tf32_trunc(x.z);
              h.w = tf32_trunc(x.w);
              lo[4 * c + 0] = __float_as_uint(x.x - h.x);
              lo[4 * c + 1] = __float_as_uint(x.y - h.y);
              lo[4 * c + 2] = __float_as_uint(x.z - h.z);
              lo[4 * c + 3] = __float_as_uint(x.w - h.w);
              if constexpr (Cfg::HI_TMEM) {
                hi[4 * c + 0] = __float_as_uint(h.x);
                hi[4 * c + 1] = __float_as_uint(h.y);
                hi[4 * c + 2] = __float_as_uint(h.z);
                hi[4 * c + 3] = __float_as_uint(h.w);
              }
              // A_hi in shared memory: the tile as it landed already reads as
              // A_hi to the MMA, so nothing is written back
            }
            tmem_st<BK>(lane_base + (uint32_t)(Cfg::LO_COL0 + half * Cfg::LO_RING + s * BK), lo);
            if constexpr (Cfg::HI_TMEM)
              tmem_st<BK>(lane_base + (uint32_t)(Cfg::HI_COL0 + s * BK), hi);
            tmem_st_wait();
          }
          }  // halves
          if constexpr (BR == 1) {
            // B_lo = B - tf32_trunc(B), stored at B's own offsets in the B_lo
            // buffer (the split is elementwise and the swizzle only permutes
            // 16-byte chunks inside each line); 1xTF32 rounds B in place.
            // Consecutive threads take consecutive 16-byte chunks.
            static_assert(Cfg::B_BYTES % (16 * kConvThreads) == 0, "whole chunks per thread");
            const float4 *src = reinterpret_cast<const float4 *>(b_hi(s));
            float4 *dst = reinterpret_cast<float4 *>(X3 ? b_lo(s) : b_hi(s));
            const int ct = (int)threadIdx.x - 64;
            constexpr int PER_T = Cfg::B_BYTES / (16 * kConvThreads);
            float4 x[PER_T];
#pragma unroll
            for (int i = 0; i < PER_T; ++i) x[i] = src[ct + i * kConvThreads];
#pragma unroll
            for (int i = 0; i < PER_T; ++i) {
              float4 y;
              if constexpr (X3) {
                y.x = x[i].x - tf32_trunc(x[i].x);
                y.y = x[i].y - tf32_trunc(x[i].y);
                y.z = x[i].z - tf32_trunc(x[i].z);
                y.w = x[i].w - tf32_trunc(x[i].w);
              } else {
                y.x = tf32_rna(x[i].x);
                y.y = tf32_rna(x[i].y);
                y.z = tf32_rna(x[i].z);
                y.w = tf32_rna(x[i].w);
              }
              dst[ct + i * kConvThreads] = y;
            }
            fence_async_smem();  // the MMA (async proxy) reads what was written
          }
          if constexpr (BR == 2) {
            // Write back what was read before the A split: once every
            // converter thread has read its block (b_read), B_hi (the raw
            // values) and B_lo go to row n, 16-byte chunk c at its swizzled
            // place (c ^ (n & 7)), as the TMA would have put them.  For a
            // fixed r, a quarter warp's n & 7 = 4 (l & 1) + r and its c run
            // so that c ^ (n & 7) takes 8 distinct values: no bank conflicts.
            if (!__all_sync(0xffffffffu,
                            mbar_wait(b_read, (uint32_t)it & 1u, deadline, abort_flag))) {
              *abort_flag = 1;
              ok = false;
              break;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int n = 4 * bjb + r;
              const float4 hi = r == 0   ? make_float4(bv[0].x, bv[1].x, bv[2].x, bv[3].x)
                                : r == 1 ? make_float4(bv[0].y, bv[1].y, bv[2].y, bv[3].y)
                                : r == 2 ? make_float4(bv[0].z, bv[1].z, bv[2].z, bv[3].z)
                                         : make_float4(bv[0].w, bv[1].w, bv[2].w, bv[3].w);
              float4 lo;
              lo.x = hi.x - tf32_trunc(hi.x);
              lo.y = hi.y - tf32_trunc(hi.y);
              lo.z = hi.z - tf32_trunc(hi.z);
              lo.w = hi.w - tf32_trunc(hi.w);
              const int off = n * Cfg::ROW_BYTES + ((bc ^ (n & 7)) * 16);
              *reinterpret_cast<float4 *>(b_hi(s) + off) = hi;
              *reinterpret_cast<float4 *>(b_lo(s) + off) = lo;
            }
            fence_async_smem();  // the MMA (async proxy) reads what was written
          }
          if constexpr (AK != 0 && X3) tc_fence_before();
          mbar_arrive(&conv[s]);
        }
        if (!ok) break;
      }
      // ---- epilogue of this segment
      const bool got = mbar_wait(acc_full, (uint32_t)si & 1u, deadline, abort_flag);
      // tcgen05.ld is warp-collective: the whole warp drains or none of it
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool whole = sg.kb0 == 0 && sg.kb1 == p.num_kb;
      int64_t mt, nt;
      tile_coords(p, sg.tile, mt, nt);
      const int64_t m0 = mt * BM;
      const int64_t n0 = nt * BN;
      // streaming with beta != 0: C's old values of these rows came with A's
      // (the producer waited for them); this warp acquires the same flag
      // before reading them
      if (p.in_flag != nullptr && p.beta != 0.0f)
        flag_wait(p.in_flag + m0 / p.stream_rows, p.epoch, deadline, abort_flag);
      // each 128-row half of the tile sits in its own accumulator columns
#pragma unroll 1
      for (int h = 0; h < Cfg::MH; ++h) {
        const int tr0 = h * 128 + quarter * 32;  // this warp's first row within the tile
        const uint32_t lane_acc = lane_base + (uint32_t)(h * Cfg::ACC_HALF);
        // whole tiles go to C; partial tiles (stream-K) to this CTA's slot,
        // 0 for its first stream-K segment, 1 for its last
        float *dst_row0;
        int64_t ld, rows_in;
        if (whole) {
          dst_row0 = p.C + (m0 + tr0) * p.ldc + n0;
          ld = p.ldc;
          rows_in = p.M - (m0 + tr0);
        } else {
          dst_row0 = p.partial + ((int64_t)(blockIdx.x * 2 + sg.slot) * BM + tr0) * BN;
          ld = BN;
          rows_in = 32;
        }
        const int rows = rows_in < 0 ? 0 : (rows_in > 32 ? 32 : (int)rows_in);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(lane_acc + (uint32_t)c, r);
          if (CONCAT) {
            uint32_t r2[32];
            tmem_ld32(lane_acc + (uint32_t)(BN + c), r2);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q)
              r[q] = __float_as_uint(__uint_as_float(r[q]) + __uint_as_float(r2[q]));
          } else {
            tmem_ld_wait();
          }
          // C_TMEM: beta * old + alpha * acc here, row by row (the same
          // operations epi_store16 does), and the block is only stored
          bool folded = false;
          if constexpr (Cfg::C_TMEM) {
            if (whole && p.beta != 0.0f) {
              uint32_t o[32];
              tmem_ld32(lane_base + (uint32_t)(Cfg::OLD_COL0 + h * BN + c), o);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 32; ++q)
                r[q] = __float_as_uint(fmaf(p.beta, __uint_as_float(o[q]),
                                            p.alpha * __uint_as_float(r[q])));
              folded = true;
            }
          }
          const float *v = reinterpret_cast<const float *>(r);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int col = c + 16 * hh;
            if (whole) {
              const int64_t left = p.N - (n0 + col);
              const int cols = left < 0 ? 0 : (left > 16 ? 16 : (int)left);
              epi_store16(epi, v + 16 * hh, dst_row0 + col, ld, rows, cols, vec,
                          folded ? 1.0f : p.alpha, folded ? 0.0f : p.beta);
            } else {
              epi_store16(epi, v + 16 * hh, dst_row0 + col, ld, 32, 16, true, 1.0f, 0.0f);
            }
          }
        }
      }
      if (p.out_flag != nullptr && whole) {
        // streaming: this warp's rows of the tile are stored.  Its stores
        // are fenced, then counted; the last of the row block's 4 x (tiles
        // in the block) warps to get here publishes the block.
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          const int64_t blk = m0 / p.stream_rows;
          const int64_t left = p.M - blk * p.stream_rows;
          const int64_t rows = left < p.stream_rows ? left : p.stream_rows;
          const unsigned target = 4u * (unsigned)(((rows + BM - 1) / BM) * p.tiles_n);
          if (atomicAdd(&p.tile_cnt[blk], 1u) + 1u == target) {
            atomicExch(&p.tile_cnt[blk], 0u);
            __threadfence();
            atomicExch(&p.out_flag[blk], p.epoch);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);  // the accumulator may be overwritten
      ++si;
    }
    if (!ok) *abort_flag = 1;
  }

  if (!ok) atomicExch(&g_tc_status, GEMM_ERR_DEVICE_TIMEOUT);
  // streaming: a thread that gave up releases every row block, so copies
  // waiting on them go ahead (the call then reports the status word)
  if (!ok && p.out_flag != nullptr)
    for (int i = 0; i < p.stream_blocks; ++i) atomicExch(&p.out_flag[i], p.epoch);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  if (p.stamps != nullptr && threadIdx.x == 0) atomicMax(&p.stamps[1], globaltimer());
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode != nullptr;
}

// 2-D FP32 tensor map: inner dimension `inner` (contiguous), `outer` rows
// `stride_elems` apart; box = box_inner x box_rows with the swizzle that
// matches box_inner * 4 bytes (or none).
bool encode_2d(CUtensorMap *m, const float *base, int64_t inner, int64_t outer,
               int64_t stride_elems, int box_inner, int box_rows, bool swizzle = true) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(stride_elems * 4)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = !swizzle               ? CU_TENSOR_MAP_SWIZZLE_NONE
                                : box_inner * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                       : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t env_u64(const char *name, uint64_t dflt) {
  const char *v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::strtoull(v, nullptr, 10);
}

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

struct WsLayout {
  uint64_t a_hi, a_lo, b_hi, b_lo, partial, total;
  int64_t kp;
};

// Workspace regions: B_hi, B_lo (K-major; unless B is split in the kernel),
// A_hi, A_lo (unless A is split in the kernel), then for stream-K the partial
// tiles (2 per CTA).  The B planes come first so their place depends only on
// N, K and the mode: calls that share B (row blocks of one product) can
// reuse them.
WsLayout ws_layout(int64_t M, int64_t N, int64_t K, bool a_inkernel, bool b_inkernel,
                   int64_t streamk_ctas, int bm, int bn, bool x3) {
  WsLayout w{};
  // Planes' rows padded (with zeros) to a multiple of 32 floats: every TMA
  // box (16 or 32 K values of a row) then starts on a 128-byte line of its
  // own instead of straddling two (GB300, 1023 x 1025 x 777: kernel 26.0 ->
  // 22.5 us; 1500^3 31.0 -> 29.2 us).
  w.kp = round_up(K, 32);
  const uint64_t b_bytes = b_inkernel ? 0 : align256((uint64_t)N * w.kp * 4);
  const uint64_t b_lo_bytes = x3 ? b_bytes : 0;
  const uint64_t a_bytes = a_inkernel ? 0 : align256((uint64_t)M * w.kp * 4);
  const uint64_t a_lo_bytes = x3 ? a_bytes : 0;
  w.b_hi = 0;
  w.b_lo = b_bytes;
  w.a_hi = b_bytes + b_lo_bytes;
  w.a_lo = w.a_hi + a_bytes;
  w.partial = w.a_lo + a_lo_bytes;
  w.total = w.partial + (uint64_t)streamk_ctas * 2 * bm * bn * 4;
  return w;
}

template <int BM, int BN, int BK, int STAGES, int AK, bool CONCAT, int NPROD, int BR>
int launch_cfg(const gemm_plan_t &plan, const GemmArgs &a, char *ws, cudaStream_t s) {
  using Cfg = TcCfg<BM, BN, BK, STAGES, AK, CONCAT, NPROD, BR>;
  constexpr bool X3 = Cfg::X3;
  const int64_t tiles_m = ceil_div(a.M, BM), tiles_n = ceil_div(a.N, BN);
  const int64_t tiles = tiles_m * tiles_n;
  const int num_kb = (int)ceil_div(a.K, BK);
  // streaming: A arrives by TMA from device memory (split on chip), one CTA
  // per tile, row blocks of whole tile rows
  const bool streaming = a.in_flag != nullptr;
  if (streaming && (!AK || plan.stream_k || a.ta || !a.out_flag || !a.tile_cnt ||
                    a.stream_rows <= 0 || a.stream_rows % BM != 0 ||
                    a.stream_blocks != ceil_div(a.M, a.stream_rows)))
    return GEMM_ERR_UNSUPPORTED;
  const int64_t G = plan.stream_k ? plan.grid_ctas : tiles;
  if (G < 1 || G > 0x7fffffff || tiles > 0x7fffffff) return GEMM_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(a.M, a.N, a.K, AK, BR, plan.stream_k ? G : 0, BM, BN, X3);
  float *ahi = reinterpret_cast<float *>(ws + L.a_hi);
  float *alo = reinterpret_cast<float *>(ws + L.a_lo);
  float *bhi = reinterpret_cast<float *>(ws + L.b_hi);
  float *blo = reinterpret_cast<float *>(ws + L.b_lo);

  CUtensorMap tA0, tA1, tB0, tB1;
  bool ok;
  if (AK) {
    ok = encode_2d(&tA0, a.A, a.K, a.M, a.lda, BK, BM);
    tA1 = tA0;
  } else {
    ok = encode_2d(&tA0, ahi, L.kp, a.M, L.kp, BK, BM);
    tA1 = tA0;
    if (X3) ok = ok && encode_2d(&tA1, alo, L.kp, a.M, L.kp, BK, BM);
  }
  if (BR) {
    // raw B: stored N x K, BK x BN boxes like A's; stored K x N, BN x BK
    // boxes without swizzle (transposed on chip)
    if (a.tb != (BR == 1)) return GEMM_ERR_UNSUPPORTED;
    ok = ok && (BR == 1 ? encode_2d(&tB0, a.B, a.K, a.N, a.ldb, BK, BN)
                        : encode_2d(&tB0, a.B, a.N, a.K, a.ldb, BN, BK, /*swizzle=*/false));
    tB1 = tB0;
  } else {
    ok = ok && encode_2d(&tB0, bhi, L.kp, a.N, L.kp, BK, BN);
    tB1 = tB0;
    if (X3) ok = ok && encode_2d(&tB1, blo, L.kp, a.N, L.kp, BK, BN);
  }
  if (!ok) return GEMM_ERR_UNSUPPORTED;

  TcParams p;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.num_kb = num_kb;
  p.tiles_m = (int)tiles_m;
  p.tiles_n = (int)tiles_n;
  // Tile order: bands of group_n column-tiles (see tile_coords).
  // One CTA per tile (no stream-K): the CTAs resident at one time work on
  // about a wave of tiles; they stream, K block by K block, the A rows of the
  // band rows they cover and the B columns of the band, which L2 shares
  // between them.  Per wave that is (wave / group_n) row tiles of A bytes a
  // and group_n column tiles of B bytes b, least at group_n = sqrt(wave * a /
  // b).  GB300, 3xTF32 8192^3 (128 x 256 tiles, bands of 6): DRAM traffic
  // 3.68 GB per launch against 4.76 GB in plain column order, same time.
  // Stream-K grids: plain column order when B's bytes in the GEMM exceed A's
  // (B's planes are 8 bytes a value in 3xTF32, A split on chip 4), else plain
  // row order; the tiles left for the stream-K part come last and their
  // CTAs, at unrelated K positions, then share the larger operand in L2
  // (4096^3 with 152 persistent CTAs: 381 us per kernel in column order,
  // 408 us in bands of 6).
  // Tuning knobs: GEMM_TC_GROUP = group_n; GEMM_TC_ORDER = 0 (plain rows) /
  // 1 (plain columns).
  {
    const double a_bytes = (double)BM * (AK || !X3 ? 4.0 : 8.0);
    const double b_bytes = (double)BN * (X3 ? 8.0 : 4.0);
    int64_t gn;
    if (plan.stream_k) {
      gn = (a_bytes / BM) * (double)a.M < (b_bytes / BN) * (double)a.N ? 1 : tiles_n;
    } else {
      int64_t wave = (int64_t)current_props().sm_count * plan.ctas_per_sm;
      if (wave > tiles) wave = tiles;
      if (wave < 1) wave = 1;
      gn = (int64_t)std::lround(std::sqrt((double)wave * a_bytes / b_bytes));
    }
    if (streaming) gn = tiles_n;  // row order: tiles follow the rows as they land
    if (const char *o = std::getenv("GEMM_TC_ORDER")) gn = std::atoi(o) == 1 ? 1 : tiles_n;
    gn = (int64_t)env_u64("GEMM_TC_GROUP", (uint64_t)gn);
    if (gn < 1) gn = 1;
    if (gn > tiles_n) gn = tiles_n;
    p.group_n = (int)gn;
  }
  // Whole-tile waves first, the rest of the tiles stream-K (G == tiles
  // without stream-K: one wave).  A short stream-K part would give each CTA
  // only a few K blocks and the fix-up many parts per tile, so the last whole
  // wave is folded into it until each CTA gets at least 4 K blocks and a
  // tile at most ~250 parts (the fix-up sums up to 256).
  int64_t waves = tiles / G, rest = tiles - waves * G;
  while (rest > 0 && waves > 0 && (rest * num_kb < 4 * G || G > 250 * rest)) {
    --waves;
    rest += G;
  }
  p.waves = (int)waves;
  p.dp_tiles = waves * G;
  p.sk_units = rest * num_kb;
  // the fix-up sums at most kFixMaxParts parts of one tile
  if (plan.stream_k && p.sk_units > 0 && max_parts_per_tile(p.sk_units, num_kb, G) > kFixMaxParts)
    return GEMM_ERR_UNSUPPORTED;
  p.partial = reinterpret_cast<float *>(ws + L.partial);
  p.timeout_ns = env_u64("GEMM_DEBUG_WAIT_LIMIT_NS", 2000000000ull);
  p.in_flag = a.in_flag;
  p.out_flag = a.out_flag;
  p.tile_cnt = a.tile_cnt;
  p.epoch = a.epoch;
  p.stream_rows = a.stream_rows;
  p.stream_blocks = a.stream_blocks;
  p.stall_producer = (int)env_u64("GEMM_DEBUG_STALL_PRODUCER", 0);
  p.stamps = profile_stamps();
  auto kern = tc_tf32x3_kernel<BM, BN, BK, STAGES, AK, CONCAT, NPROD, BR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }

  // Split passes: each operand becomes K-major hi (and lo) planes.  An
  // operand stored with K contiguous (A as M x K, B as N x K) is split row
  // by row; one stored with K as its row index is split and transposed.
  // Programmatic dependent launch lets each kernel be scheduled while the one
  // before it drains (each waits for its predecessor before touching
  // memory).  With the caller's profiling events set, plain stream order is
  // kept so the events bracket the GEMM kernel alone; callers that chain the
  // GEMM behind cross-stream event waits ask for plain order as well.
  // Every check that can refuse the call has run by now: nothing was launched.
  const bool pdl = !profile_events_set() && !a.plain_order;
  // Both passes, when both run, are one launch.
  SplitJob jobs[2];
  int njobs = 0;
  if (!AK)
    jobs[njobs++] = a.ta ? split_transposed_job(a.A, a.lda, a.K, a.M, L.kp, ahi, X3 ? alo : nullptr)
                         : split_rows_job(a.A, a.lda, a.M, a.K, L.kp, ahi, X3 ? alo : nullptr);
  if (!BR && !a.b_presplit)
    jobs[njobs++] = a.tb ? split_rows_job(a.B, a.ldb, a.N, a.K, L.kp, bhi, X3 ? blo : nullptr)
                         : split_transposed_job(a.B, a.ldb, a.K, a.N, L.kp, bhi, X3 ? blo : nullptr);
  const cudaError_t se =
      njobs ? launch_splits(jobs[0], njobs > 1 ? &jobs[1] : nullptr, pdl, s) : cudaSuccess;
  if (se != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  // B's planes are in the workspace (stream-ordered before any later call);
  // a call that splits B on chip lays its workspace out from offset 0 (no B
  // region), so whatever it writes there may overwrite earlier planes
  if (a.b_planes_written != nullptr) {
    if (!BR && !a.b_presplit) *a.b_planes_written = 1;
    if (BR && L.total > 0) *a.b_planes_written = 0;
  }

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)G);
  lc.blockDim = dim3(kThreadsTC);
  lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  profile_mark_before(s);
  cudaError_t e = cudaLaunchKernelEx(&lc, kern, tA0, tA1, tB0, tB1, p);
  profile_mark_after(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (plan.stream_k) {
    e = launch_fixup(p, BM, BN, G, pdl, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
  }
  return GEMM_OK;
}

// B stored K x N split on chip: built for the 64-column, 32-deep tiles only
// (wider tiles lose more to the on-chip transpose than the pass costs).
template <int BM, int BN, int BK, int STAGES, int AK, bool CONCAT, int NPROD, bool BRS>
int launch_kn(const gemm_plan_t &plan, const GemmArgs &a, char *ws, cudaStream_t s) {
  if constexpr (BRS && BN == 64 && BK == 32 && NPROD == 3)
    return launch_cfg<BM, BN, BK, STAGES, AK, CONCAT, NPROD, 2>(plan, a, ws, s);
  return GEMM_ERR_UNSUPPORTED;
}

}  // namespace

// The tcgen05 kernels are built for sm_103a only.
bool tc_supported(const DeviceProps &dp) { return dp.cc_major == 10 && dp.cc_minor == 3; }

// Tile configurations the planner may pick: (bm, bn, bk, stages, A split in
// kernel (0 no, 1 with A_hi in shared memory, 2 with A_hi in tensor memory),
// concatenated B MMA, TF32 products per FP32 product, B split in kernel).
#define GG_TC_CONFIGS(X)                      \
  X(128, 64, 16, 6, 0, true, 3, false)      \
  X(128, 64, 32, 4, 0, true, 3, false)      \
  X(128, 256, 16, 5, 1, false, 3, false)    \
  X(128, 256, 16, 5, 2, false, 3, false)    \
  X(128, 128, 32, 4, 2, true, 3, false)     \
  X(128, 128, 32, 4, 1, true, 3, false)     \
  X(128, 64, 32, 6, 1, true, 3, false)      \
  X(128, 64, 32, 3, 1, true, 3, false)      \
  X(128, 64, 32, 2, 1, false, 3, false)     \
  X(128, 64, 16, 4, 1, false, 3, false)     \
  X(128, 256, 16, 4, 0, false, 3, false)    \
  X(128, 128, 16, 3, 0, true, 3, false)     \
  X(128, 128, 16, 6, 0, true, 3, false)     \
  X(256, 256, 16, 3, 0, false, 3, false)    \
  X(128, 256, 16, 8, 1, false, 1, false)    \
  X(128, 64, 32, 4, 1, false, 1, false)     \
  X(128, 256, 16, 8, 0, false, 1, false)    \
  X(256, 256, 16, 6, 0, false, 1, false)    \
  X(256, 256, 32, 3, 0, false, 1, false)    \
  X(128, 256, 16, 5, 2, false, 3, true)     \
  X(128, 128, 32, 4, 2, true, 3, true)      \
  X(128, 64, 32, 6, 1, true, 3, true)       \
  X(128, 64, 32, 4, 0, true, 3, true)

// a_inkernel: 0 A pre-split, 1 split on chip (A_hi in shared memory), 2 split
// on chip with A_hi in tensor memory.  b_inkernel: B split on chip.
#define GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)                        \
  (bm == BM_ && bn == BN_ && bk == BK_ && stages == ST_ && a_inkernel == (AK_) && \
   (concat != 0) == CC_ && nprod == NP_ && (b_inkernel != 0) == BR_)

bool tc_config_valid(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod,
                     int b_inkernel) {
#define GG_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_) \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)) return true;
  GG_TC_CONFIGS(GG_MATCH)
#undef GG_MATCH
  return false;
}

// Every configuration needs more than 113 registers a thread (134-176), so
// at most two CTAs of 192 threads share an SM's 65536 registers (those above
// 170 run one CTA per SM by shared memory anyway).
constexpr int kMaxCtasPerSm = 2;

// CTAs of one configuration that fit on an SM (shared memory, TMEM and
// registers).
int tc_ctas_per_sm(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod,
                   int b_inkernel, int smem_per_sm) {
#define GG_OCC(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)            \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)) {       \
    using C = TcCfg<BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_ ? 1 : 0>; \
    int by_smem = smem_per_sm / (C::SMEM_BYTES + 1024);         \
    int by_tmem = 512 / C::TMEM_COLS;                           \
    int n = by_smem < by_tmem ? by_smem : by_tmem;              \
    return n < kMaxCtasPerSm ? n : kMaxCtasPerSm;               \
  }
  GG_TC_CONFIGS(GG_OCC)
#undef GG_OCC
  return 0;
}

bool tc_plan_streaming(gemm_plan_t &plan, int64_t M, int64_t N, int64_t K) {
  if ((plan.kernel != GEMM_KERNEL_TC_TF32X3 && plan.kernel != GEMM_KERNEL_TC_TF32) ||
      !plan.a_split_in_kernel)
    return false;
  if (plan.stream_k) {
    plan.stream_k = 0;
    plan.launches -= 1;  // no fix-up
  }
  plan.grid_ctas = ceil_div(M, plan.bm) * ceil_div(N, plan.bn);
  plan.workspace_bytes = tc_workspace_bytes(plan, M, N, K);
  return true;
}

uint64_t tc_workspace_bytes(const gemm_plan_t &plan, int64_t M, int64_t N, int64_t K) {
  return ws_layout(M, N, K, plan.a_split_in_kernel != 0, plan.b_split_in_kernel != 0,
                   plan.stream_k ? plan.grid_ctas : 0, plan.bm, plan.bn,
                   plan.mode != GEMM_MODE_TF32)
      .total;
}

int launch_tc(const gemm_plan_t &plan, const GemmArgs &a, void *ws, size_t ws_bytes,
              cudaStream_t s) {
  if (!get_encoder()) return GEMM_ERR_UNSUPPORTED;
  const uint64_t need = tc_workspace_bytes(plan, a.M, a.N, a.K);
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return GEMM_ERR_WORKSPACE_TOO_SMALL;
  // the in-kernel A split reads A by TMA as M x K rows, the in-kernel B
  // split B as stored (N x K or K x N rows)
  if (plan.a_split_in_kernel &&
      (a.ta || (a.lda & 3) || (reinterpret_cast<uintptr_t>(a.A) & 15)))
    return GEMM_ERR_UNSUPPORTED;
  if (plan.b_split_in_kernel && ((a.ldb & 3) || (reinterpret_cast<uintptr_t>(a.B) & 15)))
    return GEMM_ERR_UNSUPPORTED;
  char *w = static_cast<char *>(ws);
  const int nprod = plan.mode == GEMM_MODE_TF32 ? 1 : 3;
  const int bm = plan.bm, bn = plan.bn, bk = plan.bk, stages = plan.stages;
  const int a_inkernel = plan.a_split_in_kernel ? (plan.a_hi_tmem ? 2 : 1) : 0;
  const int concat = plan.b_concat;
  const int b_inkernel = plan.b_split_in_kernel;
#define GG_LAUNCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)                                 \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_)) {                              \
    if (!BR_) return launch_cfg<BM_, BN_, BK_, ST_, AK_, CC_, NP_, 0>(plan, a, w, s);     \
    if (a.tb) return launch_cfg<BM_, BN_, BK_, ST_, AK_, CC_, NP_, (BR_ ? 1 : 0)>(plan, a, w, s); \
    return launch_kn<BM_, BN_, BK_, ST_, AK_, CC_, NP_, BR_>(plan, a, w, s);             \
  }
  GG_TC_CONFIGS(GG_LAUNCH)
#undef GG_LAUNCH
  return GEMM_ERR_UNSUPPORTED;
}

int tc_read_and_clear_status(cudaStream_t s) {
  const int fix = fixup_read_and_clear_status(s);
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    return v;
  }
  return fix;
}

}  // namespace gg
