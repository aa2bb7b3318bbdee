// 3xTF32 GEMM on the tcgen05 tensor cores (sm_103a).
//
// The course page points at Tensor Cores as the last rung of the GEMM
// ladder and notes that letting cuBLAS use TF32 would beat the FP32 peak
// ("Project - tiled matrix multiply", sections "Stage 3 - the reference
// ceiling: cuBLAS" and "What comes next").  TF32 alone keeps only 11
// significant bits, so each FP32 operand x is split in two,
//     x_hi = tf32_rna(x)   (exactly a TF32 value),
//     x_lo = x - x_hi      (exact in FP32; the MMA reads its leading 11
//                           significant bits, which changes the product by
//                           at most 2^-21 of |x| |y|),
// and the product is formed from three TF32 MMAs accumulated in FP32:
//     A*B ~= A_hi*B_lo + A_lo*B_hi + A_hi*B_hi
// (the dropped A_lo*B_lo term is below 2^-20 of |A||B|).
//
// 1xTF32 mode issues only A_hi*B_hi.
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
//   warps 2-5   (a) when A is split inside the kernel: convert each landed
//               FP32 A tile into its hi part (in place) and lo part, then
//               release it to the MMA warp; (b) epilogue: tcgen05.ld the
//               accumulator rows, apply C = alpha*acc + beta*C, store.
// A CTA walks a list of (tile, K-range) segments: whole tiles in waves, then
// an even share of the remaining tiles' K blocks (stream-K; see Walk), with
// the pipeline running across segment boundaries.
// Operands live in shared memory K-major with the TMA swizzle (64 B rows for
// BK = 16, 128 B rows for BK = 32), which is the layout the MMA's smem
// descriptors describe.  B is row-major (N contiguous) in global memory, so
// the split pass writes B_hi/B_lo transposed (N x K, K contiguous).
//
// Every mbarrier wait is bounded by a %globaltimer deadline; on expiry the
// kernel records GEMM_ERR_DEVICE_TIMEOUT in a device status word, stops
// issuing work, waits (bounded) for the copies and MMAs it already issued,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace gg {

namespace {

__device__ int g_tc_status;  // 0 = ok, else a GEMM_ERR_* code

constexpr int kThreadsTC = 192;
constexpr int kConvThreads = 128;  // warps 2..5

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity.  Gives up when the
// deadline passes or another role has raised the CTA's abort flag.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t deadline,
                                          volatile int *abort_flag) {
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() > deadline) return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, both K-major, kind::tf32.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every previously issued tcgen05 op of this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: wait for the previous kernel in the stream
// (no-op when launched without the attribute), and let the next one launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Shared-memory matrix descriptor of a K-major, swizzled operand tile whose
// 8-row groups are `sbo` bytes apart.  layout: 2 = 128 B swizzle, 4 = 64 B.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1u << 16;                            // leading byte offset (unused here)
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;        // stride byte offset
  d |= (uint64_t)1u << 46;                            // descriptor version for tcgen05
  d |= (uint64_t)layout << 61;
  return d;
}

// Instruction descriptor: D = F32, A = B = TF32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D(tmem) (+)= A(tmem) * B(smem)^T, kind::tf32 (A read from tensor memory).
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ the GEMM kernel

struct TcParams {
  int64_t M, N, K;
  float alpha, beta;
  float *C;
  int64_t ldc;
  int num_kb;        // K blocks per output tile
  int tiles_m, tiles_n;  // output tiles along M and N
  int col_order;     // tile t = n_tile * tiles_m + m_tile (1) or m_tile * tiles_n + n_tile (0)
  int waves;         // whole tiles per CTA before the stream-K part
  int64_t dp_tiles;  // waves * G: tiles done whole, in waves
  int64_t sk_units;  // (tiles - dp_tiles) * num_kb: units shared out stream-K
  float *partial;    // stream-K partial tiles: 2 slots of 128 x BN per CTA
  uint64_t timeout_ns;
  int stall_producer;  // test hook: the producer issues nothing
};

// Work split.  CTA c of G first takes `waves` whole tiles, c, c + G, ...:
// the CTAs of one wave start their tiles together and walk K in step, so the
// operand slices of a wave are shared through L2.  The (tile, K block) units
// of the tiles left over are then split evenly (stream-K): CTA c owns units
// [c*S/G, (c+1)*S/G) of them, walked tile by tile.  Without stream-K,
// G = tiles: one wave of one tile per CTA.
// Row-tile and column-tile of output tile t.
__host__ __device__ __forceinline__ void tile_coords(const TcParams &p, int64_t t, int64_t &mt,
                                                     int64_t &nt) {
  if (p.col_order) {
    mt = t % p.tiles_m;
    nt = t / p.tiles_m;
  } else {
    mt = t / p.tiles_n;
    nt = t % p.tiles_n;
  }
}

struct Segment {
  int tile, kb0, kb1;  // K blocks [kb0, kb1) of output tile `tile`
  int slot;            // stream-K partial slot: 0 first stream-K segment, 1 later ones
};

__host__ __device__ __forceinline__ int64_t unit_begin(int64_t total, int64_t c, int64_t G) {
  return total * c / G;
}

struct Walk {
  int64_t c, G, u, u1;
  int w;
  bool first_sk;

  __device__ __forceinline__ Walk(const TcParams &p, int64_t cta, int64_t grid)
      : c(cta), G(grid), u(unit_begin(p.sk_units, cta, grid)),
        u1(unit_begin(p.sk_units, cta + 1, grid)), w(0), first_sk(true) {}

  __device__ __forceinline__ bool next(const TcParams &p, Segment &sg) {
    if (w < p.waves) {
      sg.tile = (int)((int64_t)w * G + c);
      sg.kb0 = 0;
      sg.kb1 = p.num_kb;
      sg.slot = 0;
      ++w;
      return true;
    }
    if (u >= u1) return false;
    sg.tile = (int)(p.dp_tiles + u / p.num_kb);
    sg.kb0 = (int)(u % p.num_kb);
    const int64_t left = u1 - u;
    sg.kb1 = (int)(sg.kb0 + left < p.num_kb ? sg.kb0 + left : p.num_kb);
    u += sg.kb1 - sg.kb0;
    sg.slot = first_sk ? 0 : 1;
    first_sk = false;
    return true;
  }
};

// BN: output columns per CTA.  BK: K depth of one stage (16 -> 64-byte
// swizzle, 32 -> 128-byte swizzle).  AK: A arrives raw (FP32) and the
// converter warps split it, A_hi in place in shared memory and A_lo into a
// tensor-memory ring that the A_lo*B_hi MMA reads directly; otherwise A_hi
// and A_lo come pre-split from the workspace.  CONCAT: B_hi and B_lo sit
// next to each other in the stage, so A_hi*[B_hi | B_lo] is one MMA of width
// 2*BN into two accumulators that the epilogue adds.
template <int BM, int BN, int BK, int STAGES, bool AK, bool CONCAT, int NPROD>
struct TcCfg {
  static_assert(NPROD == 3 || NPROD == 1, "3xTF32 or 1xTF32");
  static_assert(NPROD == 3 || !CONCAT, "1xTF32 has no B_lo to concatenate");
  static_assert(BM == 128 || (BM == 256 && !AK && !CONCAT),
                "a 256-row tile takes pre-split operands and separate B planes");
  static constexpr bool X3 = NPROD == 3;
  static constexpr int MH = BM / 128;  // 128-row halves, one accumulator each
  static constexpr int A_BYTES = BM * BK * 4;
  static constexpr int A_HALF_BYTES = 128 * BK * 4;
  static constexpr int B_BYTES = BN * BK * 4;
  static constexpr int A_SMEM = (AK || !X3) ? A_BYTES : 2 * A_BYTES;  // A (raw/hi) [+ A_lo]
  static constexpr int B_SMEM = X3 ? 2 * B_BYTES : B_BYTES;           // B_hi [+ B_lo]
  static constexpr int STAGE_BYTES = A_SMEM + B_SMEM;
  static constexpr int TX_BYTES = STAGE_BYTES;
  static constexpr int ROW_BYTES = BK * 4;              // 64 or 128
  static constexpr uint32_t LAYOUT = ROW_BYTES == 128 ? 2u : 4u;
  static constexpr uint32_t SBO = 8 * ROW_BYTES;        // 8-row group stride
  static constexpr int ACC_COLS = MH * (CONCAT ? 2 * BN : BN);
  static constexpr int LO_COL0 = ACC_COLS;
  static constexpr int LO_COLS = (AK && X3) ? STAGES * BK : 0;
  static constexpr int TMEM_NEED = ACC_COLS + LO_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                   : TMEM_NEED <= 64  ? 64
                                   : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256
                                                      : 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(ROW_BYTES == 64 || ROW_BYTES == 128, "BK must be 16 or 32");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(!CONCAT || 2 * BN <= 256, "concatenated B must fit one MMA");
  static_assert(TMEM_NEED <= 512, "tensor memory");
};

template <int BM, int BN, int BK, int STAGES, bool AK, bool CONCAT, int NPROD>
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_tf32x3_kernel(const __grid_constant__ CUtensorMap tmA_hi,  // A fp32 when AK
                 const __grid_constant__ CUtensorMap tmA_lo,
                 const __grid_constant__ CUtensorMap tmB_hi,
                 const __grid_constant__ CUtensorMap tmB_lo, TcParams p) {
  using Cfg = TcCfg<BM, BN, BK, STAGES, AK, CONCAT, NPROD>;
  constexpr bool X3 = Cfg::X3;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t *conv = full + STAGES;    // A tile split (AK)
  uint64_t *empty = conv + STAGES;   // stage free again
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 1;
  uint64_t *drain = acc_empty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
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
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA_hi);
    prefetch_tmap(&tmB_hi);
    if (X3) prefetch_tmap(&tmB_lo);
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
          tma_load_2d(b_hi(s), &tmB_hi, &full[s], kx, n0);
          if (X3) tma_load_2d(b_lo(s), &tmB_lo, &full[s], kx, n0);
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
          if (!mbar_wait(AK ? &conv[s] : &full[s], ph, deadline, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ah = smem_u32(a_hi(s)), al = smem_u32(a_lo(s));
          const uint32_t bh = smem_u32(b_hi(s)), bl = smem_u32(b_lo(s));
          const uint32_t lo_t = tmem_base + (uint32_t)(Cfg::LO_COL0 + s * BK);
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
              const uint32_t d = tmem_base + (uint32_t)(h * BN);
              const uint64_t dah = smem_desc(ah_h, Cfg::SBO, Cfg::LAYOUT);
              if (!X3) {
                mma_tf32(d, dah, dbh, idesc, acc);  // 1xTF32: A_hi * B_hi only
              } else if (CONCAT) {
                // columns [0, BN): A_hi*B_hi (+ A_lo*B_hi); [BN, 2BN): A_hi*B_lo
                mma_tf32(d, dah, dbh, idesc2, acc);
                if (AK)
                  mma_tf32_ts(d, lo_t + kk * 8, dbh, idesc, 1u);
                else
                  mma_tf32(d, smem_desc(al_h, Cfg::SBO, Cfg::LAYOUT), dbh, idesc, 1u);
              } else {
                const uint64_t dbl = smem_desc(bl + off, Cfg::SBO, Cfg::LAYOUT);
                mma_tf32(d, dah, dbl, idesc, acc);  // small terms first
                if (AK)
                  mma_tf32_ts(d, lo_t + kk * 8, dbh, idesc, 1u);
                else
                  mma_tf32(d, smem_desc(al_h, Cfg::SBO, Cfg::LAYOUT), dbh, idesc, 1u);
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
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
    int it = 0, si = 0;
    Walk walk(p, blockIdx.x, G);
    Segment sg;
    while (ok && walk.next(p, sg)) {
      if (AK) {
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          // tcgen05.st below is warp-collective: the warp proceeds or stops as one
          if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, deadline, abort_flag))) {
            ok = false;
            break;
          }
          // Row `row` of the landed tile: 16-byte chunk c sits at chunk
          // c ^ f(row) of its 64- or 128-byte line (the TMA swizzle).
          uint8_t *line = a_hi(s) + row * Cfg::ROW_BYTES;
          if (!X3) {
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
            mbar_arrive(&conv[s]);
            continue;
          }
          uint32_t lo[BK];
#pragma unroll
          for (int c = 0; c < BK / 4; ++c) {
            const int phys = (BK == 32) ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3));
            float4 *ptr = reinterpret_cast<float4 *>(line + phys * 16);
            const float4 x = *ptr;
            float4 h;
            h.x = tf32_rna(x.x);
            h.y = tf32_rna(x.y);
            h.z = tf32_rna(x.z);
            h.w = tf32_rna(x.w);
            lo[4 * c + 0] = __float_as_uint(x.x - h.x);
            lo[4 * c + 1] = __float_as_uint(x.y - h.y);
            lo[4 * c + 2] = __float_as_uint(x.z - h.z);
            lo[4 * c + 3] = __float_as_uint(x.w - h.w);
            *ptr = h;
          }
          tmem_st<BK>(lane_base + (uint32_t)(Cfg::LO_COL0 + s * BK), lo);
          tmem_st_wait();
          fence_async_smem();  // A_hi written by this thread -> visible to the MMA
          tc_fence_before();
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
      // each 128-row half of the tile sits in its own accumulator columns
#pragma unroll 1
      for (int h = 0; h < Cfg::MH; ++h) {
        const int tr = h * 128 + row;  // row within the tile
        const int64_t grow = m0 + tr;
        const uint32_t lane_acc = lane_base + (uint32_t)(h * BN);
        // partial tiles: slot 0 for this CTA's first stream-K segment, 1 for its last
        float *prow = p.partial + ((int64_t)(blockIdx.x * 2 + sg.slot) * BM + tr) * BN;
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
          if (!whole) {
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4 *>(prow + c + q) =
                  make_float4(__uint_as_float(r[q]), __uint_as_float(r[q + 1]),
                              __uint_as_float(r[q + 2]), __uint_as_float(r[q + 3]));
          } else if (grow < p.M) {
            float *dst = p.C + grow * p.ldc + n0 + c;
            const int64_t left = p.N - (n0 + c);
            if (vec && left >= 32) {
#pragma unroll
              for (int q = 0; q < 32; q += 4) {
                float4 o = make_float4(p.alpha * __uint_as_float(r[q]),
                                       p.alpha * __uint_as_float(r[q + 1]),
                                       p.alpha * __uint_as_float(r[q + 2]),
                                       p.alpha * __uint_as_float(r[q + 3]));
                if (p.beta != 0.0f) {
                  const float4 old = *reinterpret_cast<const float4 *>(dst + q);
                  o.x = fmaf(p.beta, old.x, o.x);
                  o.y = fmaf(p.beta, old.y, o.y);
                  o.z = fmaf(p.beta, old.z, o.z);
                  o.w = fmaf(p.beta, old.w, o.w);
                }
                *reinterpret_cast<float4 *>(dst + q) = o;
              }
            } else {
#pragma unroll
              for (int q = 0; q < 32; ++q) {
                if (q < left) {
                  float o = p.alpha * __uint_as_float(r[q]);
                  if (p.beta != 0.0f) o = fmaf(p.beta, dst[q], o);
                  dst[q] = o;
                }
              }
            }
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// Stream-K fix-up: an output tile whose K blocks were split between CTAs
// gets C = alpha * (sum of its partial tiles, in CTA order) + beta * C.
// Block j looks at the boundary between CTAs j and j+1 in the stream-K unit
// space; the block whose boundary is the first one strictly inside a tile
// handles that tile, all other blocks return at once (whole tiles were
// written by the GEMM).
constexpr int kFixMaxParts = 256;

__global__ void __launch_bounds__(256)
streamk_fixup_kernel(TcParams p, int BM, int BN, int64_t G) {
  __shared__ int64_t part_off[kFixMaxParts];
  __shared__ int nparts;
  grid_dependency_wait();  // the GEMM's partial tiles
  const int64_t c = (int64_t)blockIdx.x + 1;  // boundary between CTAs c-1 and c
  // boundaries live in the stream-K unit space (tiles after the whole-tile waves)
  const int64_t b = unit_begin(p.sk_units, c, G);
  const int64_t tl = b / p.num_kb;
  const int64_t t = p.dp_tiles + tl;
  const int64_t first = tl * p.num_kb, last = first + p.num_kb - 1;
  if (b == first || b > last) return;                       // not strictly inside a tile
  if (unit_begin(p.sk_units, c - 1, G) > first) return;     // an earlier boundary owns it
  if (threadIdx.x == 0) {
    int n = 0;
    for (int64_t cta = c - 1; cta < G && unit_begin(p.sk_units, cta, G) <= last; ++cta) {
      const int64_t ub = unit_begin(p.sk_units, cta, G), ue = unit_begin(p.sk_units, cta + 1, G);
      if (ub == ue) continue;  // no work
      // the tile is this CTA's first segment (slot 0) or its last (slot 1)
      const int slot = (ub >= first) ? 0 : 1;
      if (n < kFixMaxParts) part_off[n++] = (cta * 2 + slot) * (int64_t)BM * BN;
    }
    nparts = n;
  }
  __syncthreads();
  const int n = nparts;
  // blockIdx.y picks 32 of the tile's BM rows; each thread keeps four
  // independent 16-byte sums so several loads are in flight
  int64_t mt, nt;
  tile_coords(p, t, mt, nt);
  const int64_t m0 = mt * BM + blockIdx.y * 32;
  const int64_t n0 = nt * BN;
  const int64_t row0 = (int64_t)blockIdx.y * 32 * BN;  // offset of these rows in a part
  const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
  const int span = 32 * BN;
  for (int e0 = threadIdx.x * 4; e0 < span; e0 += blockDim.x * 16) {
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float *base = p.partial + part_off[i] + row0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * blockDim.x * 4;
        if (e < span) {
          const float4 v = *reinterpret_cast<const float4 *>(base + e);
          acc[u].x += v.x;
          acc[u].y += v.y;
          acc[u].z += v.z;
          acc[u].w += v.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * blockDim.x * 4;
      if (e >= span) continue;
      const int r = e / BN, col = e % BN;
      const int64_t gr = m0 + r, gc = n0 + col;
      if (gr >= p.M || gc >= p.N) continue;
      float *dst = p.C + gr * p.ldc + gc;
      const float a4[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
      if (vec && gc + 4 <= p.N) {
        float4 o = make_float4(p.alpha * a4[0], p.alpha * a4[1], p.alpha * a4[2], p.alpha * a4[3]);
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4 *>(dst);
          o.x = fmaf(p.beta, old.x, o.x);
          o.y = fmaf(p.beta, old.y, o.y);
          o.z = fmaf(p.beta, old.z, o.z);
          o.w = fmaf(p.beta, old.w, o.w);
        }
        *reinterpret_cast<float4 *>(dst) = o;
      } else {
        for (int q = 0; q < 4 && gc + q < p.N; ++q) {
          float o = p.alpha * a4[q];
          if (p.beta != 0.0f) o = fmaf(p.beta, dst[q], o);
          dst[q] = o;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ split pass

// dst_hi/dst_lo (rows x kp, row-major) <- split of src (rows x k, ld), zero for k <= c < kp
// (lo == nullptr: the hi part only, for 1xTF32).
__global__ void split_rows_kernel(const float *__restrict__ src, int64_t ld, int64_t rows,
                                  int64_t k, int64_t kp, float *__restrict__ hi,
                                  float *__restrict__ lo) {
  grid_launch_dependents();
  const int64_t groups = rows * (kp / 4);
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / (kp / 4);
    const int64_t c = (g % (kp / 4)) * 4;
    const float *s = src + r * ld + c;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (c + i < k) ? __ldg(s + i) : 0.0f;
    float4 h, l;
    h.x = tf32_rna(v[0]); l.x = v[0] - h.x;
    h.y = tf32_rna(v[1]); l.y = v[1] - h.y;
    h.z = tf32_rna(v[2]); l.z = v[2] - h.z;
    h.w = tf32_rna(v[3]); l.w = v[3] - h.w;
    *reinterpret_cast<float4 *>(hi + r * kp + c) = h;
    if (lo) *reinterpret_cast<float4 *>(lo + r * kp + c) = l;
  }
}

// B (k x n, ld, row-major) -> Bt_hi/Bt_lo (n x kp, row-major), columns
// k <= c < kp zero.  One CTA of 256 threads moves a 32 (k) x 128 (n) tile:
// each thread loads four 16-byte pieces along n (all in flight at once),
// the tile goes through shared memory, and each thread then stores four
// 16-byte pieces of hi and of lo along k.  `vec` (ld % 4 == 0 and a 16-byte
// aligned B) enables the 16-byte loads; the stores are 16-byte aligned
// because kp is a multiple of 4.
constexpr int kTrK = 32, kTrN = 128;

__global__ void __launch_bounds__(256)
split_transpose_kernel(const float *__restrict__ src, int64_t ld, int64_t k, int64_t n,
                       int64_t kp, int vec, float *__restrict__ hi, float *__restrict__ lo) {
  __shared__ float tile[kTrK][kTrN + 1];
  grid_dependency_wait();   // A_hi/A_lo pass before this one (if any) is done
  grid_launch_dependents();  // the GEMM may launch; it waits for this grid to finish
  const int64_t k0 = (int64_t)blockIdx.y * kTrK;
  const int64_t n0 = (int64_t)blockIdx.x * kTrN;
  const int t = threadIdx.x;
  // loads: piece p = t + 256 * i covers row p / 32, columns 4 * (p % 32) .. +3
  float4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = t + 256 * i;
    const int64_t kk = k0 + p / 32, nn = n0 + 4 * (p % 32);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kk < k) {
      const float *s = src + kk * ld + nn;
      if (vec && nn + 4 <= n) {
        x = __ldg(reinterpret_cast<const float4 *>(s));
      } else {
        if (nn + 0 < n) x.x = __ldg(s + 0);
        if (nn + 1 < n) x.y = __ldg(s + 1);
        if (nn + 2 < n) x.z = __ldg(s + 2);
        if (nn + 3 < n) x.w = __ldg(s + 3);
      }
    }
    v[i] = x;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = t + 256 * i;
    float *row = &tile[p / 32][4 * (p % 32)];
    row[0] = v[i].x;
    row[1] = v[i].y;
    row[2] = v[i].z;
    row[3] = v[i].w;
  }
  __syncthreads();
  // stores: piece q = t + 256 * i covers output row n0 + q / 8, k quad q % 8
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = t + 256 * i;
    const int nl = q / 8, kq = 4 * (q % 8);
    const int64_t nn = n0 + nl, kk = k0 + kq;
    if (nn < n && kk < kp) {
      float4 h, l;
      const float a0 = tile[kq + 0][nl], a1 = tile[kq + 1][nl];
      const float a2 = tile[kq + 2][nl], a3 = tile[kq + 3][nl];
      h.x = tf32_rna(a0); l.x = a0 - h.x;
      h.y = tf32_rna(a1); l.y = a1 - h.y;
      h.z = tf32_rna(a2); l.z = a2 - h.z;
      h.w = tf32_rna(a3); l.w = a3 - h.w;
      *reinterpret_cast<float4 *>(hi + nn * kp + kk) = h;
      if (lo) *reinterpret_cast<float4 *>(lo + nn * kp + kk) = l;
    }
  }
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
// matches box_inner * 4 bytes.
bool encode_2d(CUtensorMap *m, const float *base, int64_t inner, int64_t outer,
               int64_t stride_elems, int box_inner, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(stride_elems * 4)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      box_inner * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
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

// Workspace regions: B_hi, B_lo (K-major), A_hi, A_lo (unless A is split
// in the kernel), then for stream-K the partial tiles (2 per CTA).  The B
// planes come first so their place depends only on N, K and the mode: calls
// that share B (row blocks of one product) can reuse them.
WsLayout ws_layout(int64_t M, int64_t N, int64_t K, bool a_inkernel, int64_t streamk_ctas,
                   int bm, int bn, bool x3) {
  WsLayout w{};
  w.kp = round_up(K, 4);
  const uint64_t b_bytes = align256((uint64_t)N * w.kp * 4);
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

template <int BM, int BN, int BK, int STAGES, bool AK, bool CONCAT, int NPROD>
int launch_cfg(const gemm_plan_t &plan, const GemmArgs &a, char *ws, cudaStream_t s) {
  using Cfg = TcCfg<BM, BN, BK, STAGES, AK, CONCAT, NPROD>;
  constexpr bool X3 = Cfg::X3;
  const int64_t tiles_m = ceil_div(a.M, BM), tiles_n = ceil_div(a.N, BN);
  const int64_t tiles = tiles_m * tiles_n;
  const int num_kb = (int)ceil_div(a.K, BK);
  const int64_t G = plan.stream_k ? plan.grid_ctas : tiles;
  if (G < 1 || G > 0x7fffffff || tiles > 0x7fffffff) return GEMM_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(a.M, a.N, a.K, AK, plan.stream_k ? G : 0, BM, BN, X3);
  float *ahi = reinterpret_cast<float *>(ws + L.a_hi);
  float *alo = reinterpret_cast<float *>(ws + L.a_lo);
  float *bhi = reinterpret_cast<float *>(ws + L.b_hi);
  float *blo = reinterpret_cast<float *>(ws + L.b_lo);

  // Split passes: each operand becomes K-major hi (and lo) planes.  An
  // operand stored with K contiguous (A as M x K, B as N x K) is split row
  // by row; one stored with K as its row index is split and transposed.
  auto split_k_major = [&](const float *src, int64_t ld, int64_t rows, float *hi, float *lo) {
    int64_t blocks = ceil_div(rows * (L.kp / 4), 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    split_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, ld, rows, a.K, L.kp, hi, lo);
  };
  auto split_transposed = [&](const float *src, int64_t ld, int64_t cols, float *hi, float *lo) {
    const int vec = ((ld & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) ? 1 : 0;
    dim3 grid((unsigned)ceil_div(cols, kTrN), (unsigned)ceil_div(L.kp, kTrK));
    split_transpose_kernel<<<grid, 256, 0, s>>>(src, ld, a.K, cols, L.kp, vec, hi, lo);
  };
  if (!AK) {
    if (a.ta) split_transposed(a.A, a.lda, a.M, ahi, X3 ? alo : nullptr);
    else split_k_major(a.A, a.lda, a.M, ahi, X3 ? alo : nullptr);
  }
  if (!a.b_presplit) {
    if (a.tb) split_k_major(a.B, a.ldb, a.N, bhi, X3 ? blo : nullptr);
    else split_transposed(a.B, a.ldb, a.N, bhi, X3 ? blo : nullptr);
  }
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;

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
  ok = ok && encode_2d(&tB0, bhi, L.kp, a.N, L.kp, BK, BN);
  tB1 = tB0;
  if (X3) ok = ok && encode_2d(&tB1, blo, L.kp, a.N, L.kp, BK, BN);
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
  // Tile order.  The tiles left for the stream-K part come last; their CTAs
  // sit at unrelated K positions, so whichever operand they share must stay
  // in L2.  Numbering tiles down the columns puts them in a few column
  // blocks (sharing B's planes); along the rows, in a few row blocks
  // (sharing A).  Take the order that shares the operand with more bytes in
  // the GEMM: B (hi + lo, 8 bytes a value in 3xTF32) against A (4 bytes raw
  // when split on chip, 8 pre-split; 1xTF32: 4 and 4).  GB300, 3xTF32 with
  // 128 x 256 tiles, rows / columns: 4096^3 460 / 445 us, 3072 x 4096 x 4096
  // 399 / 367 us, 6144^3 1.54 / 1.48 ms, 2048 x 8192 x 4096 513 / 491 us,
  // 8192 x 2048 x 4096 457 / 469 us; even for 256 x 256 tiles.
  // Tuning knob: GEMM_TC_ORDER = 0 (rows) / 1 (columns).
  {
    const double a_bytes = (double)a.M * (AK || !X3 ? 4.0 : 8.0);
    const double b_bytes = (double)a.N * (X3 ? 8.0 : 4.0);
    p.col_order = (int)env_u64("GEMM_TC_ORDER", a_bytes < b_bytes ? 1 : 0);
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
  p.partial = reinterpret_cast<float *>(ws + L.partial);
  p.timeout_ns = env_u64("GEMM_DEBUG_WAIT_LIMIT_NS", 2000000000ull);
  p.stall_producer = (int)env_u64("GEMM_DEBUG_STALL_PRODUCER", 0);

  auto kern = tc_tf32x3_kernel<BM, BN, BK, STAGES, AK, CONCAT, NPROD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  // Programmatic dependent launch lets each kernel be scheduled while the one
  // before it drains (each waits for its predecessor before reading its
  // output).  With the caller's profiling events set, plain stream order is
  // kept so the events bracket the GEMM kernel alone; callers that chain the
  // GEMM behind cross-stream event waits ask for plain order as well.
  const bool pdl = !profile_events_set() && !a.plain_order;
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
    cudaLaunchConfig_t fc = {};
    fc.gridDim = dim3((unsigned)(G - 1), BM / 32);
    fc.blockDim = dim3(256);
    fc.stream = s;
    fc.attrs = attr;
    fc.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&fc, streamk_fixup_kernel, p, (int)BM, (int)BN, G);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
  }
  return GEMM_OK;
}

}  // namespace

// The tcgen05 kernels are built for sm_103a only.
bool tc_supported(const DeviceProps &dp) { return dp.cc_major == 10 && dp.cc_minor == 3; }

// Tile configurations the planner may pick: (bm, bn, bk, stages, A split in
// kernel, concatenated B MMA, TF32 products per FP32 product).
#define GG_TC_CONFIGS(X)                  \
  X(128, 256, 16, 5, true, false, 3)      \
  X(128, 128, 32, 4, true, true, 3)       \
  X(128, 64, 32, 6, true, true, 3)        \
  X(128, 64, 32, 3, true, true, 3)        \
  X(128, 64, 32, 2, true, false, 3)       \
  X(128, 64, 16, 4, true, false, 3)       \
  X(128, 256, 16, 4, false, false, 3)     \
  X(128, 128, 16, 3, false, true, 3)      \
  X(256, 256, 16, 3, false, false, 3)     \
  X(128, 256, 16, 8, true, false, 1)      \
  X(128, 64, 32, 4, true, false, 1)       \
  X(128, 256, 16, 8, false, false, 1)     \
  X(256, 256, 16, 6, false, false, 1)     \
  X(256, 256, 32, 3, false, false, 1)

#define GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_)                                  \
  (bm == BM_ && bn == BN_ && bk == BK_ && stages == ST_ && (a_inkernel != 0) == AK_ && \
   (concat != 0) == CC_ && nprod == NP_)

bool tc_config_valid(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod) {
#define GG_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_) \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_)) return true;
  GG_TC_CONFIGS(GG_MATCH)
#undef GG_MATCH
  return false;
}

// CTAs of one configuration that fit on an SM (shared memory and TMEM).
int tc_ctas_per_sm(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod,
                   int smem_per_sm) {
#define GG_OCC(BM_, BN_, BK_, ST_, AK_, CC_, NP_)              \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_)) {         \
    using C = TcCfg<BM_, BN_, BK_, ST_, AK_, CC_, NP_>;         \
    int by_smem = smem_per_sm / (C::SMEM_BYTES + 1024);         \
    int by_tmem = 512 / C::TMEM_COLS;                           \
    return by_smem < by_tmem ? by_smem : by_tmem;               \
  }
  GG_TC_CONFIGS(GG_OCC)
#undef GG_OCC
  return 0;
}

uint64_t tc_workspace_bytes(const gemm_plan_t &plan, int64_t M, int64_t N, int64_t K) {
  return ws_layout(M, N, K, plan.a_split_in_kernel != 0, plan.stream_k ? plan.grid_ctas : 0,
                   plan.bm, plan.bn, plan.mode != GEMM_MODE_TF32)
      .total;
}

int launch_tc(const gemm_plan_t &plan, const GemmArgs &a, void *ws, size_t ws_bytes,
              cudaStream_t s) {
  if (!get_encoder()) return GEMM_ERR_UNSUPPORTED;
  if (ws_bytes < tc_workspace_bytes(plan, a.M, a.N, a.K) || ws == nullptr)
    return GEMM_ERR_WORKSPACE_TOO_SMALL;
  // the in-kernel A split reads A by TMA as M x K rows
  if (plan.a_split_in_kernel &&
      (a.ta || (a.lda & 3) || (reinterpret_cast<uintptr_t>(a.A) & 15)))
    return GEMM_ERR_UNSUPPORTED;
  char *w = static_cast<char *>(ws);
  const int nprod = plan.mode == GEMM_MODE_TF32 ? 1 : 3;
  const int bm = plan.bm, bn = plan.bn, bk = plan.bk, stages = plan.stages;
  const int a_inkernel = plan.a_split_in_kernel, concat = plan.b_concat;
#define GG_LAUNCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_)  \
  if (GG_TC_MATCH(BM_, BN_, BK_, ST_, AK_, CC_, NP_)) \
    return launch_cfg<BM_, BN_, BK_, ST_, AK_, CC_, NP_>(plan, a, w, s);
  GG_TC_CONFIGS(GG_LAUNCH)
#undef GG_LAUNCH
  return GEMM_ERR_UNSUPPORTED;
}

int tc_read_and_clear_status(cudaStream_t s) {
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
  return GEMM_OK;
}

}  // namespace gg
