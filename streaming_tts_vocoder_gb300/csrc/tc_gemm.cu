// Tensor-core implicit GEMM for the decoder's dense contractions (causal and
// dilated Conv1d, the transposed convs in their phase-GEMM form, the
// transformer linears) on sm_103a: TMA loads of 32-channel k-blocks into
// swizzled shared memory, tcgen05.mma issued by one thread with the fp32
// accumulator in TMEM, and an epilogue that reads TMEM back with tcgen05.ld
// and applies bias / residual / MRF average / GELU / ring scatter.
//
// Precision: each operand is split into fp16 hi + lo parts (x = hi + lo to
// about 22 bits) and every k-step issues hi*hi + hi*lo + lo*hi, so the result
// carries close to fp32 operand accuracy while running on the f16 tensor
// pipe.  A single fp16 or bf16 pass misses the decoder's 1e-3 waveform bound
// by more than 10x on random weights.  The tensor core adds each MMA's
// products to the fp32 accumulator with truncation, not rounding; over the
// hundreds of k-steps of a long conv that bias alone costs about 20x in the
// output error.  So a tile's k-loop is cut into chunks of 16 k-steps: each
// chunk starts from a zero accumulator, and the epilogue folds every chunk
// into per-row fp32 sums in registers with rounded adds, in chunk order.  The
// truncation then acts on 16-step partial sums only, and the decoder's output
// error stays within a small factor of an fp32 FMA loop's.
//
// Operand layout: in the three-pass mode a k-block's hi and lo halves share
// one 128-byte row ([rows][Cin/32][32 hi | 32 lo], the same for the weights),
// so one 128-byte-swizzled TMA box brings both; the kernel is bound by its
// copies as much as by its MMAs, and a copy costs about one cycle per row.
// The single-pass mode reads the hi plane alone in 64-byte rows.
//
// Implicit GEMM: output row t of stream segment b takes, for tap j, the
// input row base(b) + t - shift_j, so a k-block is one TMA box at a shifted
// row coordinate; the [history | chunk] rows in front of each segment supply
// the causal left context, and an M-tile never crosses a stream segment,
// except for dense single-tap contractions (the transformer linears), whose
// M-tiles run over all segments' rows back to back.
//
// Tiles: an M-tile is 128 rows.  For N > 128 a CTA tile is one M-tile by an
// N-tile of up to 256 columns (one MMA of N = 256 per k-step and pass); for
// N <= 128 it is two M-tiles sharing the N-tile, so each B (weight) tile in
// shared memory still feeds 256 x N outputs.
//
// Roles (384 threads in three warpgroups, one CTA per SM, persistent):
//   warpgroup 0  warp 0: TMA producer (one thread); warp 1: TMEM allocator
//                and MMA issuer (one thread); gives registers away
//   warpgroups 1, 2  epilogue: with two M-tiles, warpgroup 1 + g takes
//                M-tile g; with one, it takes columns 128 g .. 128 g + 127
// A warp of an epilogue warpgroup reads TMEM lanes 32 (w % 4) .. +31.  Two to
// four TMEM buffers (as many as fit in 512 columns) rotate between chunks, so
// the epilogue drains one while the MMA fills the next.  Every wait is
// bounded: when one expires the CTA raises a flag, stops, drains its copies
// and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "tc_gemm.h"

namespace codec {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 32;              // fp16 per k-block (hi or lo): 64 bytes; the three-pass layout
                                     // puts a k-block's hi and lo in one 128-byte row
constexpr int kThreads = 384;        // 3 warpgroups
constexpr int kEpiWarps = 8;
constexpr int kMaxBN = 256;          // 2 buffers x 256 columns = 512
constexpr int kEpiCols = 128;        // columns one epilogue thread sums
constexpr int kMaxBufs = 4;          // TMEM chunk buffers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSpinLimit = kDefaultWaitPolls;   // drains of work already in flight
constexpr int kSmemBudget = 227 * 1024;   // the opt-in maximum per CTA
// one 32 x 32 fp32 block per epilogue warp, then 32 ints per warp (the q/K/V
// scatter's ring rows of the warp's 32 rows)
constexpr int kStageOutBytes = kEpiWarps * 32 * 32 * 4 + kEpiWarps * 32 * 4;
constexpr uint32_t kAPlaneBytes = kBM * kBK * 2;   // 8 KB: one M-tile, one plane
constexpr int kChunkKb = 8;          // 8 k-blocks = 256 of K = 16 MMA k-steps per TMEM chunk

struct TcParams {
    int n_row_tiles;
    int mtiles;         // M-tiles per CTA tile: 2 when BN <= 128, else 1
    int issuers;        // MMA-issuing threads: one per M-tile, or two halves of one tile's N
    uint32_t iss_a;     // the second issuer's offsets: its A box (bytes into the stage),
    uint32_t iss_b;     //   its B rows (bytes into the stage's B box)
    uint32_t iss_d;     //   and its accumulator columns
    int b_early;        // 1: B may be loaded before the grid dependency resolves
    int n_mgroups;      // ceil(n_row_tiles / mtiles)
    int n_tiles_n;
    int BN;
    int nkb;            // k-blocks: ntaps * Cin / kBK
    int cin_blocks;     // Cin / kBK
    int ntaps;
    int stages;
    uint32_t stage_bytes;
    uint32_t tx_bytes;  // bytes the TMA loads of a stage deliver
    uint32_t idesc;
    uint32_t buf_cols;    // TMEM columns per buffer: mtiles x round32(BN) <= 256
    uint32_t mt_cols;     // TMEM column offset between the M-tiles of a buffer
    int nbuf;             // TMEM buffers (512 / buf_cols, at most kMaxBufs)
    int epi_cols;         // columns of one M-tile an epilogue warpgroup finishes (<= kEpiCols)
    int chunk_kb;         // k-blocks accumulated in TMEM before the epilogue folds them in
    int n_chunks;         // chunks of a tile's k-loop
    int n_splits;         // CTA tiles per output tile along K (1: fold in registers)
    int cps;              // chunks per split
    float* ws;            // n_splits > 1: chunk partials [n_chunks][n_row_tiles][128][N]
    float unscale;
    const float* unscale_dev;   // when set, the accumulator scale is read from here
    int* err;
    uint32_t wait_polls;        // polls before a wait gives up
    int unarrived_wait;         // verification: the epilogue's first wait targets a barrier nobody arrives on
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
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

// Wait for the phase of the given parity; false if it did not complete
// within `polls` polls or another role of the CTA gave up first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t polls)
{
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (i >= polls) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile with 64-byte swizzle: rows of 64 bytes, 8-row groups
// 512 bytes apart (stride byte offset); the leading byte offset is unused for
// swizzled K-major layouts.  Bits 46-47 carry the descriptor version.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}

// The same with 128-byte swizzle: rows of 128 bytes (a k-block's 32 hi then
// 32 lo values), 8-row groups 1024 bytes apart.  A k-step's operand starts
// 32 bytes further per 16 elements inside the row (hi at 0 / 32, lo at 64 /
// 96); the MMA takes the swizzle phase from the address bits.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive columns of this warp's 32 lanes, no wait (pair with tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v)
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Instruction descriptor of kind::f16: D f32, A and B f16, both K-major.
constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct TileRows {
    int b, t0, nrows;
    long long in_base;    // input row of output row t0 (tap shift 0)
};

__device__ __forceinline__ TileRows tile_rows(const GemmArgs& a, const PlanView& plan, int mt)
{
    TileRows r;
    if (a.dense) {
        const int total = __ldg(plan.cf + plan.B) * a.in_l.r;
        r.b = -1;
        r.t0 = mt * kBM;
        r.nrows = min(kBM, total - r.t0);
        r.in_base = r.t0;
        return r;
    }
    r.b = find_seg(a.tcum, plan.B, mt);
    const int seg_rows = (__ldg(plan.cf + r.b + 1) - __ldg(plan.cf + r.b)) * a.in_l.r;
    r.t0 = (mt - __ldg(a.tcum + r.b)) * kBM;
    r.nrows = min(kBM, seg_rows - r.t0);
    r.in_base = seg_base(a.in_l, plan.cf, r.b) + r.t0;
    return r;
}

// The epilogue leaves TMEM with one row per thread (32 rows x 32 columns per
// warp and load).  Written to global memory that way, every warp access
// touches 32 rows, 16 bytes each; so each 32 x 32 block first goes through
// shared memory, and the global loads and stores then cover four rows of 128
// contiguous bytes per warp access.  The 16-byte chunks of a staged row are
// XOR-swizzled by the row so that the row-wise writes and the column-quad
// reads are both free of bank conflicts.
__device__ __forceinline__ void stage_put(float4* stg, int lane, const float* v)
{
#pragma unroll
    for (int j = 0; j < 8; j++)
        stg[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

__device__ __forceinline__ float4 stage_get(const float4* stg, int r, int cq)
{
    return stg[r * 8 + (cq ^ (r & 7))];
}

// Ring row (slot x ring_R + position mod ring_R) of the keys and values of
// output row t (the projection's row; b < 0: dense tiling, t over all segments).
__device__ __forceinline__ int qkv_ring_row(const GemmArgs& a, const PlanView& plan, int b, int t)
{
    if (b < 0) {
        b = find_seg_r(plan.cf, plan.B, t, a.pos_r);
        t -= __ldg(plan.cf + b) * a.pos_r;
    }
    const long long pos = __ldg(plan.pos0 + b) * a.pos_r + t;
    return (int)((long long)__ldg(plan.slot + b) * a.ring_R + (pos & (a.ring_R - 1)));
}

// Destination of four consecutive output columns n .. n+3 of output row t
// (row out_row of the output layout), or null when they cannot be moved as
// one aligned float4 (fewer than four valid, or a misaligned row).
__device__ __forceinline__ float* epi_dst4(const GemmArgs& a, const PlanView& plan, int b, int t,
                                           long long out_row, int n, int cnt)
{
    if (cnt < 4) return nullptr;
    if (a.epi == EPI_QKV) {
        if (a.d & 3) return nullptr;
        if (n < a.d) return a.out + out_row * a.d + n;
        if (b < 0) {                // dense tiling: t is the row over all segments
            b = find_seg_r(plan.cf, plan.B, t, a.pos_r);
            t -= __ldg(plan.cf + b) * a.pos_r;
        }
        const long long pos = __ldg(plan.pos0 + b) * a.pos_r + t;
        const long long rr = (long long)__ldg(plan.slot + b) * a.ring_R + (pos & (a.ring_R - 1));
        return n < 2 * a.d ? a.kring + rr * a.d + (n - a.d) : a.vring + rr * a.d + (n - 2 * a.d);
    }
    const long long idx = out_row * a.out_C + n;
    return (idx & 3) ? nullptr : a.out + idx;
}

// The per-element epilogue of the modes that read nothing back (store,
// GELU, q/K/V scatter): sum x unscale + bias, then GELU.
__device__ __forceinline__ float epi_plain(const GemmArgs& a, float v, float bias, float unscale)
{
    float y = __fmul_rn(v, unscale);
    if (a.bias) y = __fadd_rn(y, bias);
    if (a.epi == EPI_GELU) y = gelu_f(y);
    return y;
}

// The same for the modes that add the residual r (and the earlier MRF sum o).
__device__ __forceinline__ float epi_resid(const GemmArgs& a, float v, float bias, float r, float o, float unscale)
{
    float y = __fmul_rn(v, unscale);
    if (a.bias) y = __fadd_rn(y, bias);
    y = r + y;
    if (a.epi == EPI_MRF_ADD) y = o + y;
    if (a.epi == EPI_MRF_LAST) y = (o + y) * a.scale;
    return y;
}

// Columns that cannot move as one aligned float4: element by element.
__device__ __noinline__ void epi_store_slow(const GemmArgs& a, const PlanView& plan, int b, int t, long long out_row,
                                            int n, int cnt, float4 v, float unscale)
{
    const float ve[4] = {v.x, v.y, v.z, v.w};
    for (int e = 0; e < cnt && e < 4; e++) gemm_store(a, plan, b, t, out_row, n + e, __fmul_rn(ve[e], unscale));
}

// Pull the lines this row's epilogue will read (residual, earlier MRF sum)
// towards L2 while the tile's MMAs run.
__device__ __forceinline__ void epi_prefetch(const GemmArgs& a, long long out_row, int n0, int ncols)
{
    const bool has_res = a.epi == EPI_RESID || a.epi == EPI_MRF_FIRST || a.epi == EPI_MRF_ADD || a.epi == EPI_MRF_LAST;
    const bool has_old = a.epi == EPI_MRF_ADD || a.epi == EPI_MRF_LAST;
    const long long idx = out_row * a.out_C + n0;
    for (int c = 0; c < ncols; c += 32) {
        if (has_res) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.res + idx + c));
        if (has_old) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.out + idx + c));
    }
}

// kPasses: 3 for the hi/lo split (hi*hi + hi*lo + lo*hi), 1 for a single
// fp16 pass over the hi planes only.  A compile-time parameter: the copy and
// MMA loops stay branch-free.
//   3 passes: ma / mb map the interleaved operands ([rows][Cin/32][32 hi | 32
//   lo], [N][K/32][32 hi | 32 lo]); a stage holds per M-tile one 128 x 128-byte
//   A box and one BN x 128-byte B box, 128-byte swizzled: a k-block's hi and
//   lo parts arrive in the same TMA row, half the copies of separate planes.
//   1 pass: the hi planes alone in 64-byte rows, 64-byte swizzled.
template <int kPasses>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap ma,
                                                              const __grid_constant__ CUtensorMap mb,
                                                              const GemmArgs a, const PlanView plan, const TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float4* stage_out = reinterpret_cast<float4*>(smem + (size_t)p.stages * p.stage_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * p.stage_bytes + kStageOutBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + p.stages;
    uint64_t* tfull = bars + 2 * p.stages;
    uint64_t* tempty = tfull + kMaxBufs;
    uint64_t* drain = tempty + kMaxBufs;
    uint64_t* unarrived = drain + 1;    // verification only: initialised, never arrived on
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(unarrived + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // stage layout: A box of M-tile g at g x kABox, then the B box
    constexpr uint32_t kRow = kPasses == 3 ? 128u : 64u;      // bytes per operand row in a stage
    constexpr uint32_t kABox = kBM * kRow;                    // one M-tile's A box
    constexpr int kBoxK = kPasses == 3 ? 2 * kBK : kBK;       // box width in elements
    if (threadIdx.x == 0) {
        // every MMA-issuing thread commits once per stage, chunk and drain
        for (int s = 0; s < p.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], p.issuers);
        }
        for (int i = 0; i < p.nbuf; i++) {
            mbar_init(&tfull[i], p.issuers);
            mbar_init(&tempty[i], kEpiWarps);
        }
        mbar_init(drain, p.issuers);
        mbar_init(unarrived, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int total_tiles = p.n_mgroups * p.n_tiles_n * p.n_splits;
    // Weights written before any kernel of the stream ran (p.b_early) do not
    // depend on the earlier kernels: the copy thread issues the B boxes of its
    // first tile's first stages now, while an earlier kernel may still run.
    int b_pre = 0;
    if (warp == 0 && lane == 0) prefetch_tensormap(&ma);   // a kernel parameter: no dependency
    if (p.b_early && warp == 0 && lane == 0 && (int)blockIdx.x < total_tiles) {
        prefetch_tensormap(&mb);
        const int tile = blockIdx.x;
        const int sp = tile % p.n_splits, mn = tile / p.n_splits;
        const int n0 = (mn % p.n_tiles_n) * p.BN;
        const int kb_lo = sp * p.cps * p.chunk_kb, kb_hi = min(p.nkb, kb_lo + p.cps * p.chunk_kb);
        b_pre = min(p.stages, kb_hi - kb_lo);
        uint8_t* st = smem;
        for (int q = 0; q < b_pre; q++, st += p.stage_bytes) {
            mbar_expect_tx(&full[q], p.tx_bytes);
            tma_load_2d(st + p.mtiles * kABox, &mb, &full[q], (kb_lo + q) * kBoxK, n0);
        }
    }
    // the set-up above touches shared memory, TMEM and the weights only;
    // global memory written by earlier kernels is read from here on
    pdl_wait();
    pdl_launch();
    const uint32_t tmem_base = *tmem_slot;
    const float unscale = p.unscale_dev ? *p.unscale_dev : p.unscale;
    const int wg = warp >> 2;

    if (wg == 0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------- producer --
            // One thread: every dependent instruction costs its full latency,
            // so the k-loop keeps its indices by increments (no division).
            prefetch_tensormap(&ma);
            prefetch_tensormap(&mb);
            int it = 0, s = 0;
            uint32_t ph = 0;
            uint8_t* st = smem;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const int sp = tile % p.n_splits, mn = tile / p.n_splits;
                const int mg = mn / p.n_tiles_n;
                const long long in0 = tile_rows(a, plan, p.mtiles * mg).in_base;
                const long long in1 =
                    (p.mtiles == 2 && 2 * mg + 1 < p.n_row_tiles) ? tile_rows(a, plan, 2 * mg + 1).in_base : in0;
                const int n0 = (mn % p.n_tiles_n) * p.BN;
                const int kb_lo = sp * p.cps * p.chunk_kb, kb_hi = min(p.nkb, kb_lo + p.cps * p.chunk_kb);
                // k-block kb = tap j x cin_blocks + channel block cb
                int j = kb_lo / p.cin_blocks, cb = kb_lo - j * p.cin_blocks;
                int row0 = (int)(in0 - a.shift[j]), row1 = (int)(in1 - a.shift[j]);
                for (int kb = kb_lo; kb < kb_hi; kb++) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.wait_polls)) { ok = false; break; }
                    const int c0 = cb * kBoxK;
                    // the first b_pre stages were armed, and their B boxes issued, above
                    if (it >= b_pre) mbar_expect_tx(&full[s], p.tx_bytes);
                    tma_load_2d(st, &ma, &full[s], c0, row0);
                    if (p.mtiles == 2) tma_load_2d(st + kABox, &ma, &full[s], c0, row1);
                    if (it >= b_pre) tma_load_2d(st + p.mtiles * kABox, &mb, &full[s], kb * kBoxK, n0);
                    it++;
                    st += p.stage_bytes;
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                        st = smem;
                    }
                    if (++cb == p.cin_blocks) {
                        cb = 0;
                        if (++j < p.ntaps) {
                            row0 = (int)(in0 - a.shift[j]);
                            row1 = (int)(in1 - a.shift[j]);
                        }
                    }
                }
            }
            // drain: every stage's last armed load has landed before exit
            for (int q = 0; q < p.stages && q < it; q++) {
                const int last = q + ((it - 1 - q) / p.stages) * p.stages;
                mbar_drain(&full[q], (uint32_t)(last / p.stages) & 1u);
            }
        } else if ((warp == 1 || (warp == 2 && p.issuers == 2)) && lane == 0) {
            // --------------------------------------------------- MMA issue --
            // The k-loop of a tile is cut into chunks of chunk_kb k-blocks; each
            // chunk accumulates from zero into one of the TMEM buffers, which
            // the epilogue folds into rounded fp32 sums while the next chunk
            // runs.  Indices by increments, as in the producer.  Two M-tiles
            // get an issuing thread each (warp 1: M-tile 0, warp 2: M-tile 1):
            // for narrow tiles one thread's issue loop, not the tensor pipe,
            // set the pace.  An accumulator gets its MMAs in one fixed order
            // from one thread.  A lone M-tile in a latency-bound call may
            // instead be cut into two column halves, one per issuing thread
            // (the per-element result of an MMA does not depend on its width).
            const int mi = warp - 1;
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            const uint32_t smem0 = smem_u32(smem);
            uint32_t sa = smem0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const int sp = tile % p.n_splits;
                const int kb_lo = sp * p.cps * p.chunk_kb, kb_hi = min(p.nkb, kb_lo + p.cps * p.chunk_kb);
                for (int kb0 = kb_lo; kb0 < kb_hi && ok; kb0 += p.chunk_kb) {
                    if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.wait_polls)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d0 = tmem_base + (uint32_t)acc * p.buf_cols + (uint32_t)mi * p.iss_d;
                    const int kb1 = min(p.nkb, kb0 + p.chunk_kb);
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!mbar_wait(&full[s], ph, abort_flag, p.wait_polls)) { ok = false; break; }
                        tc_fence_after();
                        // descriptors of the stage's boxes: one base plus constant
                        // steps; in three-pass mode the lo part of a row sits 64
                        // bytes after its hi part
                        const uint64_t base = kPasses == 3 ? sdesc_sw128(sa) : sdesc_sw64(sa);
                        const uint64_t ah = base + (((uint32_t)mi * p.iss_a) >> 4);
                        const uint64_t al = ah + (64 >> 4);
                        const uint64_t bh = base + (((uint32_t)p.mtiles * kABox + (uint32_t)mi * p.iss_b) >> 4);
                        const uint64_t bl = bh + (64 >> 4);
#pragma unroll
                        for (int k = 0; k < kBK / 16; k++) {
                            const uint64_t o = (uint64_t)((k * 32) >> 4);
                            const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
                            mma_f16(d0, ah + o, bh + o, p.idesc, accum);
                            if (kPasses == 3) {
                                mma_f16(d0, ah + o, bl + o, p.idesc, 1u);
                                mma_f16(d0, al + o, bh + o, p.idesc, 1u);
                            }
                        }
                        mma_commit(&empty[s]);
                        sa += p.stage_bytes;
                        if (++s == p.stages) {
                            s = 0;
                            ph ^= 1u;
                            sa = smem0;
                        }
                    }
                    if (!ok) break;
                    mma_commit(&tfull[acc]);
                    if (++acc == p.nbuf) {
                        acc = 0;
                        aph ^= 1u;
                    }
                }
            }
            // all issued MMAs complete before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;" ::: "memory");
        // ------------------------------------------------------ epilogue --
        // With two M-tiles, warpgroup 1 + g finishes M-tile g; with one, it
        // finishes columns E g .. E g + E - 1 (E = p.epi_cols: 128, or half a
        // narrower tile in 32-column slices).  Thread (warp w, lane l)
        // owns row 32 (w % 4) + l and keeps its <= 128 column sums in
        // registers across the chunks.
        const int g = wg - 1;
        const int my_mt = p.mtiles == 2 ? g : 0;
        const int col0 = p.mtiles == 2 ? 0 : g * p.epi_cols;
        const int ncol = max(0, min(p.epi_cols, p.BN - col0));
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const int cq = lane & 7;        // column quad of the transposed pass
        float4* stg = stage_out + (warp - 4) * 256;
        int* srow = reinterpret_cast<int*>(stage_out + kEpiWarps * 256) + (warp - 4) * 32;
        const bool has_res = a.epi == EPI_RESID || a.epi == EPI_MRF_FIRST || a.epi == EPI_MRF_ADD || a.epi == EPI_MRF_LAST;
        const bool has_old = a.epi == EPI_MRF_ADD || a.epi == EPI_MRF_LAST;
        int chunk_it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            const int sp = tile % p.n_splits, mn = tile / p.n_splits;
            const int kb_lo = sp * p.cps * p.chunk_kb, kb_hi = min(p.nkb, kb_lo + p.cps * p.chunk_kb);
            const int mt = p.mtiles * (mn / p.n_tiles_n) + my_mt;
            const int n0 = (mn % p.n_tiles_n) * p.BN + col0;
            const int nvalid = min(ncol, a.N - n0);
            TileRows tr{0, 0, 0, 0};
            if (mt < p.n_row_tiles) tr = tile_rows(a, plan, mt);
            const long long out_base = (mt < p.n_row_tiles && !a.dense) ? seg_base(a.out_l, plan.cf, tr.b) : 0;
            if (p.n_splits == 1 && nvalid > 0 && m < tr.nrows)
                epi_prefetch(a, out_base + (long long)(tr.t0 + m) * a.out_step, n0, nvalid);
            float sum[kEpiCols];
#pragma unroll
            for (int i = 0; i < kEpiCols; i++) sum[i] = 0.f;
            for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += p.chunk_kb, chunk_it++) {
                const int acc = chunk_it % p.nbuf;
                const uint32_t aph = (uint32_t)(chunk_it / p.nbuf) & 1u;
                // one lane polls, the warp follows its verdict (tcgen05.ld needs a converged warp)
                int w_ok = 1;
                uint64_t* wbar = (p.unarrived_wait && chunk_it == 0) ? unarrived : &tfull[acc];
                if (lane == 0) w_ok = mbar_wait(wbar, aph, abort_flag, p.wait_polls) ? 1 : 0;
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) { ok = false; break; }
                tc_fence_after();
                const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * p.buf_cols +
                                           (uint32_t)my_mt * p.mt_cols + (uint32_t)col0;
                // split tiles hand each chunk's partial to the reduce kernel:
                // partials [chunk][row tile][128][N]
                float* wtile = p.n_splits > 1
                                   ? p.ws + ((size_t)(kb0 / p.chunk_kb) * p.n_row_tiles + mt) * kBM * a.N + n0
                                   : nullptr;
#pragma unroll
                for (int c = 0; c < kEpiCols; c += 32) {
                    if (c < ncol) {
                        uint32_t r[32];
                        tmem_ld32_async(lane_base + (uint32_t)c, r);
                        tmem_wait_ld();
                        if (p.n_splits == 1) {
#pragma unroll
                            for (int i = 0; i < 32; i++) sum[c + i] = __fadd_rn(sum[c + i], __uint_as_float(r[i]));
                        } else if (c < nvalid && mt < p.n_row_tiles && tr.nrows <= 16) {
                            // a tile of a few rows (a frame or two): each lane
                            // stores its own row's 16 or 32 columns, with no
                            // transpose through shared memory
                            if (m < tr.nrows) {
                                float4* dst = reinterpret_cast<float4*>(wtile + (size_t)m * a.N + c);
                                const int cnt = min(32, nvalid - c);
#pragma unroll
                                for (int i = 0; i < 8; i++)
                                    if (4 * i < cnt)
                                        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                             __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                            }
                        } else if (c < nvalid && mt < p.n_row_tiles) {
                            stage_put(stg, lane, reinterpret_cast<const float*>(r));
                            __syncwarp();
                            if (c + 4 * cq < nvalid) {
#pragma unroll
                                for (int i = 0; i < 8; i++) {
                                    const int mr = q * 32 + 4 * i + (lane >> 3);
                                    if (mr < tr.nrows)
                                        *reinterpret_cast<float4*>(wtile + (size_t)mr * a.N + c + 4 * cq) =
                                            stage_get(stg, 4 * i + (lane >> 3), cq);
                                }
                            }
                            __syncwarp();
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
            }
            if (!ok) break;
            if (p.n_splits > 1 || mt >= p.n_row_tiles || nvalid <= 0) continue;
            // Transposed pass, one 32-column slice at a time: lane takes column
            // quad cq of rows 4 i + lane / 8.  The loop is not unrolled (its
            // body is long); the slice's sums are always sum[0..31], the rest
            // move down by 32 after each slice.
            const bool vec_ok = a.epi == EPI_QKV ? (a.d & 3) == 0 : (a.out_C & 3) == 0;
            // q/K/V scatter: each lane finds the ring row of one of the warp's 32
            // rows once per tile (a segment search); the slices then read it
            const bool qkv4 = a.epi == EPI_QKV && vec_ok;
            if (qkv4) {
                const int mr = q * 32 + lane;
                srow[lane] = mr < tr.nrows ? qkv_ring_row(a, plan, tr.b, tr.t0 + mr) : 0;
                __syncwarp();
            }
#pragma unroll 1
            for (int c = 0; c < nvalid; c += 32) {
                stage_put(stg, lane, sum);
                __syncwarp();
                const int n = n0 + c + 4 * cq;
                const int cnt = min(4, nvalid - c - 4 * cq);
                float bias4[4] = {0.f, 0.f, 0.f, 0.f};
                if (a.bias && cnt > 0) {
                    int bi = n % a.bias_mod;
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        if (e < cnt) bias4[e] = __ldg(a.bias + bi);
                        bi = (bi + 1 == a.bias_mod) ? 0 : bi + 1;
                    }
                }
                if (cnt == 4 && vec_ok && has_res) {
                    // every load of the slice is in flight before the first store
                    float4 rv[8], ov[8];
                    long long off[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int mr = q * 32 + 4 * i + (lane >> 3);
                        off[i] = -1;
                        rv[i] = ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (mr < tr.nrows) {
                            off[i] = (out_base + (long long)(tr.t0 + mr) * a.out_step) * a.out_C + n;
                            rv[i] = *reinterpret_cast<const float4*>((a.res ? a.res : a.out) + off[i]);
                            if (has_old) ov[i] = *reinterpret_cast<const float4*>(a.out + off[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        if (off[i] >= 0) {
                            const float4 v = stage_get(stg, 4 * i + (lane >> 3), cq);
                            float4 y;
                            y.x = epi_resid(a, v.x, bias4[0], rv[i].x, ov[i].x, unscale);
                            y.y = epi_resid(a, v.y, bias4[1], rv[i].y, ov[i].y, unscale);
                            y.z = epi_resid(a, v.z, bias4[2], rv[i].z, ov[i].z, unscale);
                            y.w = epi_resid(a, v.w, bias4[3], rv[i].w, ov[i].w, unscale);
                            *reinterpret_cast<float4*>(a.out + off[i]) = y;
                        }
                    }
                } else if (cnt == 4 && vec_ok) {
#pragma unroll 2
                    for (int i = 0; i < 8; i++) {
                        const int r = 4 * i + (lane >> 3);
                        const int mr = q * 32 + r;
                        if (mr < tr.nrows) {
                            const int t = tr.t0 + mr;
                            const float4 v = stage_get(stg, r, cq);
                            float4 y;
                            y.x = epi_plain(a, v.x, bias4[0], unscale);
                            y.y = epi_plain(a, v.y, bias4[1], unscale);
                            y.z = epi_plain(a, v.z, bias4[2], unscale);
                            y.w = epi_plain(a, v.w, bias4[3], unscale);
                            const long long orow = out_base + (long long)t * a.out_step;
                            float* dst;
                            if (qkv4 && n >= a.d) {
                                const long long rr = srow[r];
                                dst = n < 2 * a.d ? a.kring + rr * a.d + (n - a.d) : a.vring + rr * a.d + (n - 2 * a.d);
                            } else {
                                dst = epi_dst4(a, plan, tr.b, t, orow, n, cnt);
                            }
                            if (dst) *reinterpret_cast<float4*>(dst) = y;
                            else epi_store_slow(a, plan, tr.b, t, orow, n, cnt, v, unscale);
                        }
                    }
                } else if (cnt > 0) {
#pragma unroll 1
                    for (int i = 0; i < 8; i++) {
                        const int r = 4 * i + (lane >> 3);
                        const int mr = q * 32 + r;
                        if (mr < tr.nrows) {
                            const int t = tr.t0 + mr;
                            epi_store_slow(a, plan, tr.b, t, out_base + (long long)t * a.out_step, n, cnt,
                                           stage_get(stg, r, cq), unscale);
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int j = 0; j < kEpiCols - 32; j++) sum[j] = sum[j + 32];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(p.err, 1);
}

// Split tiles: fold the chunk partials of each output in chunk order with
// rounded adds, exactly as the unsplit epilogue folds them in registers, then
// apply the same per-element epilogue.  One thread per (row, 4 columns); the
// partial loads of up to 16 chunks are in flight at once.
constexpr int kReduceRows = 32;
__global__ void __launch_bounds__(kReduceRows * 8) tc_reduce_kernel(const GemmArgs a, const PlanView plan,
                                                                   const float* __restrict__ ws, int n_chunks,
                                                                   int n_row_tiles, float unscale,
                                                                   const float* __restrict__ unscale_dev)
{
    pdl_wait();
    pdl_launch();
    const int mt = blockIdx.x;
    const int m = blockIdx.z * kReduceRows + (threadIdx.x >> 3);
    const int n = (blockIdx.y * 8 + (threadIdx.x & 7)) * 4;
    const TileRows tr = tile_rows(a, plan, mt);
    if (m >= tr.nrows || n >= a.N) return;
    const float us = unscale_dev ? *unscale_dev : unscale;
    const size_t stride = (size_t)n_row_tiles * kBM * a.N;
    const float* src = ws + ((size_t)mt * kBM + m) * a.N + n;
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
    const bool v4 = n + 4 <= a.N && (a.N & 3) == 0;
    int c = 0;
    if (v4) {
        for (; c + 16 <= n_chunks; c += 16) {
            float4 p[16];
#pragma unroll
            for (int u = 0; u < 16; u++) p[u] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(c + u) * stride));
#pragma unroll
            for (int u = 0; u < 16; u++) {
                sum[0] = __fadd_rn(sum[0], p[u].x);
                sum[1] = __fadd_rn(sum[1], p[u].y);
                sum[2] = __fadd_rn(sum[2], p[u].z);
                sum[3] = __fadd_rn(sum[3], p[u].w);
            }
        }
        for (; c + 8 <= n_chunks; c += 8) {
            float4 p[8];
#pragma unroll
            for (int u = 0; u < 8; u++) p[u] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(c + u) * stride));
#pragma unroll
            for (int u = 0; u < 8; u++) {
                sum[0] = __fadd_rn(sum[0], p[u].x);
                sum[1] = __fadd_rn(sum[1], p[u].y);
                sum[2] = __fadd_rn(sum[2], p[u].z);
                sum[3] = __fadd_rn(sum[3], p[u].w);
            }
        }
        for (; c + 4 <= n_chunks; c += 4) {
            float4 p[4];
#pragma unroll
            for (int u = 0; u < 4; u++) p[u] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(c + u) * stride));
#pragma unroll
            for (int u = 0; u < 4; u++) {
                sum[0] = __fadd_rn(sum[0], p[u].x);
                sum[1] = __fadd_rn(sum[1], p[u].y);
                sum[2] = __fadd_rn(sum[2], p[u].z);
                sum[3] = __fadd_rn(sum[3], p[u].w);
            }
        }
    }
    for (; c < n_chunks; c++)
        for (int e = 0; e < 4; e++)
            if (n + e < a.N) sum[e] = __fadd_rn(sum[e], __ldg(src + (size_t)c * stride + e));
    const int t = tr.t0 + m;
    const long long out_row = (a.dense ? 0 : seg_base(a.out_l, plan.cf, tr.b)) + (long long)t * a.out_step;
    for (int e = 0; e < 4; e++)
        if (n + e < a.N) gemm_store(a, plan, tr.b, t, out_row, n + e, __fmul_rn(sum[e], us));
}

// hi = fp16(a), lo = fp16(a - hi), a = Snake(x), GELU(x) or x; eight consecutive
// channels (32 bytes in, 16 out per plane) per thread and one unit per
// thread, so every load of the grid can be in flight at once.  The Snake
// parameters are read as float4 when aligned (4 loads per thread, not 16).
// interleaved: [rows][Cin / 32][32 hi | 32 lo] (three-pass mode: a 32-channel
// k-block of a row is one 128-byte TMA row); else the hi plane [rows][Cin].
__global__ void __launch_bounds__(256) tc_prep_kernel(const float4* __restrict__ x, const float* __restrict__ alpha,
                                                      const float* __restrict__ inv_alpha, bool vec_alpha,
                                                      unsigned units, unsigned cin8, uint4* __restrict__ hi,
                                                      bool interleaved, bool gelu)
{
    pdl_wait();
    pdl_launch();
    const unsigned u = blockIdx.x * 256u + threadIdx.x;
    if (u >= units) return;
    const float4 p0 = __ldg(x + 2 * (size_t)u), p1 = __ldg(x + 2 * (size_t)u + 1);
    float v[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const unsigned c8 = u % cin8;
    if (alpha) {
        const unsigned c = c8 * 8u;
        float al[8], ia[8];
        if (vec_alpha) {
            const float4 a0 = __ldg(reinterpret_cast<const float4*>(alpha + c));
            const float4 a1 = __ldg(reinterpret_cast<const float4*>(alpha + c) + 1);
            const float4 i0 = __ldg(reinterpret_cast<const float4*>(inv_alpha + c));
            const float4 i1 = __ldg(reinterpret_cast<const float4*>(inv_alpha + c) + 1);
            al[0] = a0.x; al[1] = a0.y; al[2] = a0.z; al[3] = a0.w;
            al[4] = a1.x; al[5] = a1.y; al[6] = a1.z; al[7] = a1.w;
            ia[0] = i0.x; ia[1] = i0.y; ia[2] = i0.z; ia[3] = i0.w;
            ia[4] = i1.x; ia[5] = i1.y; ia[6] = i1.z; ia[7] = i1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) {
                al[e] = __ldg(alpha + c + e);
                ia[e] = __ldg(inv_alpha + c + e);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; e++) v[e] = snake_f(v[e], al[e], ia[e]);
    } else if (gelu) {
#pragma unroll
        for (int e = 0; e < 8; e++) v[e] = gelu_f(v[e]);
    }
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const __half h0 = __float2half_rn(v[2 * e]), h1 = __float2half_rn(v[2 * e + 1]);
        const __half l0 = __float2half_rn(v[2 * e] - __half2float(h0));
        const __half l1 = __float2half_rn(v[2 * e + 1] - __half2float(h1));
        h[e] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
        l[e] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
    if (interleaved) {
        // [rows][Cin / 32][32 hi | 32 lo]: unit u = (row, c8) lands at
        // 2 u - (c8 % 4) (hi) and 4 units further (lo)
        const size_t at = 2 * (size_t)u - (c8 & 3u);
        hi[at] = make_uint4(h[0], h[1], h[2], h[3]);
        hi[at + 4] = make_uint4(l[0], l[1], l[2], l[3]);
    } else {
        hi[u] = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D fp16 tensor map over [outer][inner] with a box of box_inner x box_outer
// and 64-byte swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    // 64-element (128-byte) boxes take the 128-byte swizzle, 32-element ones the 64-byte one
    const CUtensorMapSwizzle sw = box_inner * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

uint32_t round1024(uint32_t x) { return (x + 1023u) & ~1023u; }

// N-tile: 32, 64, 96, 128 or 256, the one that pads N least (ties: the
// wider).  Tiles of at most 128 columns pair two M-tiles with an MMA-issuing
// thread each, and a 256-column MMA runs at the pipe's rate; the widths in
// between (160 to 224) ran one M-tile from one issuing thread, which set the
// pace below the pipe's rate.
int pick_bn(int N)
{
    int best = 32;
    for (int bn = 32; bn <= kMaxBN; bn += 32) {
        if (bn > 128 && bn < kMaxBN) continue;
        const int pad = (N + bn - 1) / bn * bn, best_pad = (N + best - 1) / best * best;
        if (pad < best_pad || (pad == best_pad && bn > best)) best = bn;
    }
    return best;
}

}  // namespace

cudaError_t tc_configure()
{
    for (const void* k : {(const void*)tc_gemm_kernel<1>, (const void*)tc_gemm_kernel<3>}) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool tc_eligible(int Cin, int N) { return Cin >= kBK && Cin % kBK == 0 && N >= 16 && N % 16 == 0; }

bool tc_pack_weights(const float* wkn, int ntaps, int Cin, int N, int passes, TcWeights* out,
                     std::vector<void*>& allocs)
{
    out->passes = passes;
    const size_t K = (size_t)ntaps * Cin;
    float mx = 0.f;
    for (size_t i = 0; i < K * (size_t)N; i++) mx = std::fmax(mx, std::fabs(wkn[i]));
    const int e = mx > 0.f ? -(int)std::floor(std::log2(mx)) : 0;
    const float scale = std::ldexp(1.0f, e);
    // passes == 3: one [N][2K] buffer, each 32-wide k-block stored as its 32 hi
    // then its 32 lo values (one 128-byte TMA row per k-block and n); passes
    // == 1: the hi plane [N][K] alone
    const size_t KP = passes == 3 ? 2 * K : K;
    std::vector<__half> pl(KP * N);
    for (int n = 0; n < N; n++)
        for (size_t k = 0; k < K; k++) {
            const float w = wkn[k * N + n] * scale;
            const __half h = __float2half_rn(w);
            if (passes == 3) {
                const size_t at = (size_t)n * KP + (k / kBK) * (2 * kBK) + (k % kBK);
                pl[at] = h;
                pl[at + kBK] = __float2half_rn(w - __half2float(h));
            } else {
                pl[(size_t)n * KP + k] = h;
            }
        }
    void* dh = nullptr;
    if (cudaMalloc(&dh, pl.size() * sizeof(__half)) != cudaSuccess) return false;
    allocs.push_back(dh);
    if (cudaMemcpy(dh, pl.data(), pl.size() * sizeof(__half), cudaMemcpyHostToDevice) != cudaSuccess) return false;
    out->hi = dh;
    out->unscale = std::ldexp(1.0f, -e);
    out->BN = pick_bn(N);
    out->n_tiles = (N + out->BN - 1) / out->BN;
    out->b_static = true;   // the synchronous copy above completes before any later kernel
    if (!make_map(&out->map_hi, dh, KP, (uint64_t)N, passes == 3 ? 2 * kBK : kBK, (uint32_t)out->BN)) return false;
    out->n_alt = 0;
    for (const int bn : {128, 64}) {
        if (bn >= out->BN) continue;
        if (!make_map(&out->map_alt[out->n_alt], dh, KP, (uint64_t)N, passes == 3 ? 2 * kBK : kBK, (uint32_t)bn))
            return false;
        out->bn_alt[out->n_alt++] = bn;
    }
    return true;
}

bool tc_scratch_alloc(TcScratch* s, size_t elems, size_t b_elems, size_t ws_floats, std::vector<void*>& allocs)
{
    if (ws_floats) {
        if (cudaMalloc(&s->ws, ws_floats * sizeof(float)) != cudaSuccess) return false;
        allocs.push_back(s->ws);
        s->ws_floats = ws_floats;
    }
    // each operand's two planes in one block (lo right after hi): the
    // three-pass layout interleaves them over the whole block
    s->op.b_elems = b_elems;
    if (cudaMalloc(&s->op.b_hi, 2 * std::max<size_t>(b_elems, 1) * sizeof(__half)) != cudaSuccess) return false;
    allocs.push_back(s->op.b_hi);
    s->op.b_lo = static_cast<__half*>(s->op.b_hi) + std::max<size_t>(b_elems, 1);
    if (cudaMalloc(&s->op.words, kOpWords * sizeof(int)) != cudaSuccess) return false;
    allocs.push_back(s->op.words);
    if (cudaMalloc(&s->a_hi, 2 * elems * sizeof(__half)) != cudaSuccess) return false;
    allocs.push_back(s->a_hi);
    s->a_lo = static_cast<__half*>(s->a_hi) + elems;
    if (cudaMalloc(&s->err, sizeof(int)) != cudaSuccess) return false;
    allocs.push_back(s->err);
    if (cudaMemset(s->err, 0, sizeof(int)) != cudaSuccess) return false;
    s->elems = elems;
    s->op.a_hi = s->a_hi;
    s->op.a_lo = s->a_lo;
    s->op.a_elems = elems;
    s->op.err = s->err;
    return true;
}

cudaError_t launch_tc_prep(const float* x, const float* alpha, const float* inv_alpha, long long rows, int Cin,
                           TcScratch* scratch, bool with_lo, cudaStream_t s, bool gelu)
{
    const long long n = rows * Cin;
    if (n <= 0) return cudaSuccess;
    if ((size_t)n > scratch->elems || Cin % 8 != 0 || n / 8 >= (1LL << 32)) return cudaErrorInvalidValue;
    const unsigned units = (unsigned)(n / 8);
    const bool vec_alpha = alpha && ((reinterpret_cast<uintptr_t>(alpha) | reinterpret_cast<uintptr_t>(inv_alpha)) & 15) == 0;
    launch_pdl(tc_prep_kernel, dim3((units + 255) / 256), dim3(256), 0, s, reinterpret_cast<const float4*>(x),
               alpha, inv_alpha, vec_alpha, units, (unsigned)(Cin / 8), static_cast<uint4*>(scratch->a_hi),
               with_lo, gelu);
    return cudaGetLastError();
}

namespace {

cudaError_t tc_gemm_core(const GemmArgs& a, const TcWeights& w, const float* unscale_dev, PlanView plan,
                         int n_row_tiles, const void* a_planes, long long a_rows, int* err, TcWaitLimit wl,
                         int num_sms, cudaStream_t s, float* ws, size_t ws_floats, int* launches)
{
    if (n_row_tiles <= 0) return cudaSuccess;
    // A: the interleaved [rows][2 Cin] operand (three passes) or the hi plane
    alignas(64) CUtensorMap ma;
    const int box_k = w.passes == 3 ? 2 * kBK : kBK;
    const uint64_t a_inner = (uint64_t)a.Cin * (w.passes == 3 ? 2 : 1);
    if (!make_map(&ma, a_planes, a_inner, (uint64_t)a_rows, box_k, kBM)) return cudaErrorInvalidValue;
    TcParams p;
    p.n_row_tiles = n_row_tiles;
    p.cin_blocks = a.Cin / kBK;
    p.ntaps = a.ntaps;
    p.nkb = a.ntaps * p.cin_blocks;
    // a short k-loop (<= 12 k-blocks, 24 k-steps) accumulates in one chunk;
    // longer ones are cut every kChunkKb k-blocks
    p.chunk_kb = p.nkb <= 12 ? p.nkb : kChunkKb;
    p.n_chunks = (p.nkb + p.chunk_kb - 1) / p.chunk_kb;
    const int sms = num_sms > 0 ? num_sms : 152;
    // One candidate N-tile width: M-tile pairing, split count and the time of
    // the busiest CTA in MMA cycles.
    struct Shape {
        int bn, n_tiles, mtiles, cps, n_splits;
        const CUtensorMap* map;
        double est;
    };
    auto shape_for = [&](int bn, const CUtensorMap* map) {
        Shape c{bn, (a.N + bn - 1) / bn, 1, p.n_chunks, 1, map, 0.0};
        // two M-tiles share each B tile when N is narrow, unless pairing would
        // leave SMs idle (few rows: latency matters more than B traffic).  Each
        // M-tile's MMAs are the same either way, so the pairing never changes a
        // result's bits.
        c.mtiles = (bn <= 128 && ((n_row_tiles + 1) / 2) * c.n_tiles >= sms) ? 2 : 1;
        // Too few tiles to fill the GPU: split the k-loop over CTAs by whole
        // chunks.  The reduce kernel folds the chunk partials in the same order
        // as the unsplit epilogue, so splitting never changes a result's bits.
        // Pick the split count that minimises waves / splits, the time of the
        // busiest CTA in units of a whole tile's k-loop: with few tiles (a
        // one-frame call) it spreads every tile over many CTAs; with a little
        // over one wave (1600 rows of a transformer linear: 156 tiles on 152
        // SMs) it evens out the second wave.  A split pays for its partials'
        // round trip and the reduction, so it must win by more than 10 %.
        const int tiles = ((n_row_tiles + c.mtiles - 1) / c.mtiles) * c.n_tiles;
        const size_t need = (size_t)p.n_chunks * n_row_tiles * kBM * a.N;
        if (ws && p.n_chunks >= 2 && need <= ws_floats && tiles < 4 * sms) {
            double best = (double)((tiles + sms - 1) / sms);
            for (int ns = 2; ns <= p.n_chunks; ns++) {
                const int cps = (p.n_chunks + ns - 1) / ns;
                const int nsplit = (p.n_chunks + cps - 1) / cps;
                const double t = (double)((tiles * nsplit + sms - 1) / sms) * cps / p.n_chunks;
                if (t < best * 0.9) {
                    best = t;
                    c.cps = cps;
                }
            }
            c.n_splits = (p.n_chunks + c.cps - 1) / c.cps;
        }
        // a 128 x bn x 16 MMA: about bn / 2 cycles, never under ~48
        const double mma = std::max(48.0, 0.49 * bn) * c.mtiles;
        c.est = (double)((tiles * c.n_splits + sms - 1) / sms) * c.cps * mma;
        return c;
    };
    Shape sh = shape_for(w.BN, &w.map_hi);
    // A call of one or two row tiles (a frame or two) is bound by latency: a
    // narrower tile over the same weight planes may finish sooner (the
    // per-element result of an MMA does not depend on the tile width, so
    // neither do the bits); it must win by 10 %.  With more rows the
    // partials' traffic of the extra splits was measured to cancel the gain.
    if (n_row_tiles <= 2 && sh.n_tiles < sms)
        for (int i = 0; i < w.n_alt; i++) {
            const Shape c = shape_for(w.bn_alt[i], &w.map_alt[i]);
            if (c.est < sh.est * 0.9) sh = c;
        }
    p.mtiles = sh.mtiles;
    p.n_mgroups = (n_row_tiles + p.mtiles - 1) / p.mtiles;
    p.n_tiles_n = sh.n_tiles;
    p.BN = sh.bn;
    p.b_early = w.b_static ? 1 : 0;
    // operand rows in a stage: 128 bytes (a k-block's hi and lo) or 64 (hi only)
    const uint32_t row = w.passes == 3 ? 128u : 64u;
    p.stage_bytes = (uint32_t)p.mtiles * kBM * row + round1024((uint32_t)p.BN * row);
    p.tx_bytes = (uint32_t)p.mtiles * kBM * row + (uint32_t)p.BN * row;
    const int extra = 1024 + 512 + kStageOutBytes;   // alignment slack, barriers and flags, the epilogue's staging
    p.stages = std::min(8, (kSmemBudget - extra) / (int)p.stage_bytes);
    if (p.stages < 2) return cudaErrorInvalidValue;
    p.mt_cols = (uint32_t)((p.BN + 31) / 32 * 32);
    p.buf_cols = (uint32_t)p.mtiles * p.mt_cols;
    // Epilogue: with two M-tiles each warpgroup finishes one; with one, the
    // two warpgroups share its columns in 32-column slices (a lone tile of
    // at most 128 columns used to leave the second warpgroup idle).
    p.epi_cols = (p.mtiles == 2 || p.BN > kEpiCols) ? kEpiCols : std::max(32, ((p.BN + 1) / 2 + 31) / 32 * 32);
    // Second issuing thread: the second M-tile, or (one M-tile, at most one
    // CTA tile per SM: latency-bound) the second half of the tile's columns.
    // Half of a 32-multiple is a 16-multiple (a valid MMA width) and starts
    // its B rows on a whole swizzle atom.
    p.issuers = 1;
    p.iss_a = p.iss_b = p.iss_d = 0;
    p.idesc = idesc_f16(kBM, p.BN);
    if (p.mtiles == 2) {
        p.issuers = 2;
        p.iss_a = (uint32_t)kBM * row;
        p.iss_d = p.mt_cols;
    } else if (p.BN % 32 == 0 && (long long)p.n_mgroups * p.n_tiles_n * sh.n_splits <= sms) {
        p.issuers = 2;
        p.iss_b = (uint32_t)(p.BN / 2) * row;
        p.iss_d = (uint32_t)(p.BN / 2);
        p.idesc = idesc_f16(kBM, p.BN / 2);
    }
    p.nbuf = std::min<int>(kMaxBufs, (int)(kTmemCols / p.buf_cols));
    p.cps = sh.cps;
    p.n_splits = sh.n_splits;
    p.ws = p.n_splits > 1 ? ws : nullptr;
    p.unscale = w.unscale;
    p.unscale_dev = unscale_dev;
    p.err = err;
    p.wait_polls = wl.polls;
    p.unarrived_wait = wl.unarrived_wait;
    const size_t smem = (size_t)p.stages * p.stage_bytes + extra;
    const int tiles = p.n_mgroups * p.n_tiles_n * p.n_splits;
    const int grid = std::min(tiles, sms);
    if (w.passes == 3)
        launch_pdl(tc_gemm_kernel<3>, dim3(grid), dim3(kThreads), smem, s, ma, *sh.map, a, plan, p);
    else
        launch_pdl(tc_gemm_kernel<1>, dim3(grid), dim3(kThreads), smem, s, ma, *sh.map, a, plan, p);
    cudaError_t e = cudaGetLastError();
    if (launches) (*launches)++;
    if (e != cudaSuccess || p.n_splits == 1) return e;
    launch_pdl(tc_reduce_kernel, dim3(n_row_tiles, (a.N + 31) / 32, kBM / kReduceRows), dim3(kReduceRows * 8), 0,
               s, a, plan, p.ws, p.n_chunks, n_row_tiles, p.unscale, unscale_dev);
    if (launches) (*launches)++;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm(const GemmArgs& a, const TcWeights& w, PlanView plan, int n_row_tiles,
                           const TcScratch* scratch, long long a_rows, int num_sms, cudaStream_t s, int* launches)
{
    return tc_gemm_core(a, w, nullptr, plan, n_row_tiles, scratch->a_hi, a_rows, scratch->err, scratch->wait,
                        num_sms, s, scratch->ws, scratch->ws_floats, launches);
}

// ------------------------------------------------------- standalone conv --
// One causal dilated Conv1d through the same prep + tcgen05 kernels, with the
// weights packed on the device and every scratch array (operand planes, the
// one-segment plan, the weight scale) in the memory TcOpScratch points to.

namespace {

// word layout of TcOpScratch::words: plan (8 ints), weight |max| bits, the
// accumulator scale, then 1/alpha for up to kOpMaxCin channels
constexpr int kOpPlan = 0, kOpWmax = 8, kOpUnscale = 9, kOpInvAlpha = 16;

__global__ void op_setup_kernel(int* words, int T, const float* __restrict__ alpha, int Cin)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) {
        long long* pos0 = reinterpret_cast<long long*>(words + kOpPlan);
        pos0[0] = 0;                         // words 0, 1
        words[kOpPlan + 2] = 0;              // cf = {0, T}
        words[kOpPlan + 3] = T;
        words[kOpPlan + 4] = 0;              // slot
        words[kOpPlan + 5] = 0;              // bidx
        words[kOpPlan + 6] = 0;              // 128-row tiles = {0, ceil(T / 128)}
        words[kOpPlan + 7] = (T + kBM - 1) / kBM;
        words[kOpWmax] = 0;
    }
    if (alpha && i < Cin) reinterpret_cast<float*>(words + kOpInvAlpha)[i] = 1.0f / alpha[i];
}

__global__ void op_wmax_kernel(const float* __restrict__ w, long long n, unsigned* __restrict__ out)
{
    unsigned m = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        m = max(m, __float_as_uint(fabsf(w[i])));      // non-negative floats order like their bits
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

// w [Cout][Cin][k] -> w * 2^e (e from |w|max), K = k Cin tap-major, in the
// three-pass layout [Cout][K / 32][32 hi | 32 lo]
__global__ void op_wpack_kernel(const float* __restrict__ w, int Cout, int Cin, int k, int* words,
                                __half* __restrict__ out)
{
    const float mx = __uint_as_float(static_cast<unsigned>(words[kOpWmax]));
    const int e = mx > 0.f ? -(int)floorf(log2f(mx)) : 0;
    const float scale = ldexpf(1.0f, e);
    const long long K = (long long)k * Cin, n = (long long)Cout * K;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long co = i / K, kk = i - co * K;
        const long long j = kk / Cin, ci = kk - j * Cin;
        const float v = w[(co * Cin + ci) * k + j] * scale;
        const __half h = __float2half_rn(v);
        const long long at = co * 2 * K + (kk / kBK) * (2 * kBK) + (kk % kBK);
        out[at] = h;
        out[at + kBK] = __float2half_rn(v - __half2float(h));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<float*>(words)[kOpUnscale] = ldexpf(1.0f, -e);
}

}  // namespace

int check_tc_conv1d(const TcOpScratch& sc, int T, int Cin, bool has_alpha, int Cout, int k, int dil)
{
    if (T < 1 || k < 1 || k > kMaxTaps || dil < 1 || !tc_eligible(Cin, Cout)) return OP_BAD_ARG;
    if (has_alpha && Cin > kOpMaxCin) return OP_BAD_ARG;
    const long long H = (long long)(k - 1) * dil;
    const long long rows = H + T;
    const long long K = (long long)k * Cin;
    if ((size_t)(rows * Cin) > sc.a_elems || (size_t)(K * Cout) > sc.b_elems) return OP_TOO_BIG;
    if (rows > (1LL << 30)) return OP_TOO_BIG;
    return OP_OK;
}

int run_tc_conv1d(const TcOpScratch& sc, const float* x, int T, int Cin, const float* w,
                                const float* bias, const float* alpha, int Cout, int k, int dil, float* y,
                                int num_sms, cudaStream_t s)
{
    const int chk = check_tc_conv1d(sc, T, Cin, alpha != nullptr, Cout, k, dil);
    if (chk != OP_OK) return chk;
    const long long H = (long long)(k - 1) * dil;
    const long long rows = H + T;
    const long long K = (long long)k * Cin;
    int* words = sc.words;
    const float* inv_alpha = reinterpret_cast<const float*>(words + kOpInvAlpha);
    op_setup_kernel<<<(std::max(Cin, 1) + 255) / 256, 256, 0, s>>>(words, T, alpha, Cin);
    if (cudaGetLastError() != cudaSuccess) return OP_CUDA;
    const long long wn = K * Cout;
    const int wblocks = (int)std::min<long long>((wn + 255) / 256, 152LL * 8);
    op_wmax_kernel<<<wblocks, 256, 0, s>>>(w, wn, reinterpret_cast<unsigned*>(words + kOpWmax));
    op_wpack_kernel<<<wblocks, 256, 0, s>>>(w, Cout, Cin, k, words, static_cast<__half*>(sc.b_hi));
    if (cudaGetLastError() != cudaSuccess) return OP_CUDA;
    TcScratch as;
    as.a_hi = sc.a_hi;
    as.a_lo = sc.a_lo;
    as.elems = sc.a_elems;
    as.err = sc.err;
    if (launch_tc_prep(x, alpha, alpha ? inv_alpha : nullptr, rows, Cin, &as, true, s) != cudaSuccess) return OP_CUDA;
    TcWeights tw;
    tw.passes = 3;
    tw.hi = sc.b_hi;
    tw.BN = pick_bn(Cout);
    tw.n_tiles = (Cout + tw.BN - 1) / tw.BN;
    if (!make_map(&tw.map_hi, sc.b_hi, (uint64_t)(2 * K), (uint64_t)Cout, 2 * kBK, (uint32_t)tw.BN)) return OP_CUDA;
    GemmArgs a{};
    a.in = x;
    a.in_l = Layout{1, (int)H};
    a.Cin = Cin;
    a.ntaps = k;
    for (int j = 0; j < k; j++) a.shift[j] = (k - 1 - j) * dil;
    a.N = Cout;
    a.K = (int)K;
    a.bias = bias;
    a.bias_mod = Cout;
    a.out = y;
    a.out_l = Layout{1, 0};
    a.out_C = Cout;
    a.out_step = 1;
    a.epi = EPI_STORE;
    a.scale = 1.f;
    a.pos_r = 1;
    a.tcum = words + kOpPlan + 6;
    a.bm = kBM;
    PlanView plan{1, words + kOpPlan + 2, words + kOpPlan + 4, reinterpret_cast<const long long*>(words + kOpPlan),
                  words + kOpPlan + 5, nullptr};
    const int n_row_tiles = (T + kBM - 1) / kBM;
    if (tc_gemm_core(a, tw, reinterpret_cast<const float*>(words) + kOpUnscale, plan, n_row_tiles, sc.a_hi,
                     rows, sc.err, sc.wait, num_sms, s, nullptr, 0, nullptr) != cudaSuccess)
        return OP_CUDA;
    return OP_OK;
}

}  // namespace codec
