// Shared by the tensor-core GEMM kernel (tc_tf32x3.cu) and its split and
// fix-up passes (tc_split.cu): inline-PTX wrappers for tcgen05, TMA and
// mbarriers, the kernel's parameter block, the tile numbering and the work
// walk (whole-tile waves, then stream-K).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace gg {
namespace tc {

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

// Waits (bounded, like mbar_wait) until *flag - epoch >= 0 as a 32-bit cyclic
// compare, with acquire semantics at GPU scope: data written to device
// memory before the flag was set is visible afterwards.
__device__ __forceinline__ bool flag_wait(const unsigned *flag, unsigned epoch, uint64_t deadline,
                                          volatile int *abort_flag) {
  uint32_t spins = 0;
  while (true) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if ((int)(v - epoch) >= 0) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() > deadline) return false;
    }
    __nanosleep(200);
  }
}

// Orders this thread's earlier global-memory accesses (generic proxy)
// before its later TMA accesses of global memory (async proxy).
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Requests the 128-byte line holding *ptr into L2 (a hint: nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
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

// The TF32 value the tensor core reads from an FP32 word: the word with its
// low 13 mantissa bits cleared (its leading 11 significant bits).  Exactly a
// TF32 value, and x - tf32_trunc(x) is exact in FP32.
__device__ __forceinline__ float tf32_trunc(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
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

struct TcParams {
  int64_t M, N, K;
  float alpha, beta;
  float *C;
  int64_t ldc;
  int num_kb;        // K blocks per output tile
  int tiles_m, tiles_n;  // output tiles along M and N
  int group_n;       // tile order: bands of group_n column-tiles, each walked down its rows
  int waves;         // whole tiles per CTA before the stream-K part
  int64_t dp_tiles;  // waves * G: tiles done whole, in waves
  int64_t sk_units;  // (tiles - dp_tiles) * num_kb: units shared out stream-K
  float *partial;    // stream-K partial tiles: 2 slots of BM x BN per CTA
  uint64_t timeout_ns;
  // streaming (GemmArgs::in_flag): row block i of A (and C) has landed once
  // in_flag[i] - epoch >= 0; out_flag[i] = epoch once its tiles are stored
  const unsigned *in_flag;
  unsigned *out_flag, *tile_cnt;
  unsigned epoch;
  int64_t stream_rows;
  int stream_blocks;
  int stall_producer;  // test hook: the producer issues nothing
  unsigned long long *stamps;  // measurement aid (gemm_set_profile_stamps), or nullptr
};

// Row-tile and column-tile of output tile t.  Tiles are numbered in bands of
// group_n column-tiles (the last band may be narrower): band b holds tiles
// [b * group_n * tiles_m, (b + 1) * group_n * tiles_m), walked row by row
// across the band.  group_n = 1 is plain column order, group_n = tiles_n
// plain row order; in between, the tiles resident at one time cover a block
// of about (G / group_n) row-tiles by group_n column-tiles.
__host__ __device__ __forceinline__ void tile_coords(const TcParams &p, int64_t t, int64_t &mt,
                                                     int64_t &nt) {
  const int64_t band_tiles = (int64_t)p.group_n * p.tiles_m;
  const int64_t band = t / band_tiles;
  const int64_t first_n = band * p.group_n;
  const int64_t left = p.tiles_n - first_n;
  const int64_t width = left < p.group_n ? left : p.group_n;
  const int64_t local = t - band * band_tiles;
  mt = local / width;
  nt = first_n + local % width;
}

// Work split.  CTA c of G first takes `waves` whole tiles, c, c + G, ...:
// the CTAs of one wave start their tiles together and walk K in step, so the
// operand slices of a wave are shared through L2.  The (tile, K block) units
// of the tiles left over are then split evenly (stream-K): CTA c owns units
// [c*S/G, (c+1)*S/G) of them, walked tile by tile.  Without stream-K,
// G = tiles: one wave of one tile per CTA.
struct Segment {
  int tile, kb0, kb1;  // K blocks [kb0, kb1) of output tile `tile`
  int slot;            // stream-K partial slot: 0 first stream-K segment, 1 later ones
};

__host__ __device__ __forceinline__ int64_t unit_begin(int64_t total, int64_t c, int64_t G) {
  return total * c / G;
}

// The CTA whose stream-K range holds unit u: the largest c with
// unit_begin(total, c, G) <= u.
__host__ __device__ __forceinline__ int64_t unit_owner(int64_t total, int64_t u, int64_t G) {
  return ((u + 1) * G - 1) / total;
}

// Most CTAs that share one stream-K tile (an upper bound on the parts the
// fix-up sums for any tile): tile tl spans units [tl*num_kb, (tl+1)*num_kb).
__host__ __device__ __forceinline__ int64_t max_parts_per_tile(int64_t total, int64_t num_kb,
                                                               int64_t G) {
  int64_t most = 0;
  for (int64_t first = 0; first < total; first += num_kb) {
    const int64_t n = unit_owner(total, first + num_kb - 1, G) - unit_owner(total, first, G) + 1;
    if (n > most) most = n;
  }
  return most;
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

// Passes around the GEMM kernel (tc_split.cu).  Each returns the launch error.
// pdl: launched with programmatic dependent launch, so it may be scheduled
// while the kernel before it drains; it waits for that kernel before touching
// memory.
// One operand's TF32 split into hi (and lo) planes, K-major.  transposed =
// 0: dst (a = rows x kp) <- src (rows x b = k, row stride ld); transposed =
// 1: dst (b = cols x kp) <- the transpose of src (a = k x cols, row stride
// ld).  Columns k..kp-1 are zero; lo == nullptr: the hi part only (1xTF32).
struct SplitJob {
  const float *src;
  int64_t ld, a, b, kp;
  float *hi, *lo;
  int transposed, vec;
  int64_t blocks;  // thread blocks of this job
  int64_t grid_x;  // transposed: blocks along cols
};
SplitJob split_rows_job(const float *src, int64_t ld, int64_t rows, int64_t k, int64_t kp,
                        float *hi, float *lo);
SplitJob split_transposed_job(const float *src, int64_t ld, int64_t k, int64_t cols, int64_t kp,
                              float *hi, float *lo);
// One launch running job a, then (b != nullptr) job b, in separate blocks.
cudaError_t launch_splits(const SplitJob &a, const SplitJob *b, bool pdl, cudaStream_t s);
// Sums the parts of the tiles shared between stream-K CTAs into C.  At most
// kFixMaxParts parts per tile (the launcher checks max_parts_per_tile first;
// a tile with more sets the fix-up's status word to GEMM_ERR_UNSUPPORTED and
// is left alone).
constexpr int kFixMaxParts = 256;
cudaError_t launch_fixup(const TcParams &p, int bm, int bn, int64_t G, bool pdl, cudaStream_t s);

// Reads and clears the fix-up's device status word (0 = ok, else a GEMM_ERR_*
// code), after synchronising `s`.
int fixup_read_and_clear_status(cudaStream_t s);

}  // namespace tc
}  // namespace gg
