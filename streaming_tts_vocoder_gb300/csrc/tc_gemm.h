// Tensor-core (tcgen05 / TMEM / TMA) implicit-GEMM path with fp16 hi/lo
// split operands.  Declarations shared by the host runtime and tc_gemm.cu.
#pragma once

#include <cuda.h>

#include <vector>

#include "common.cuh"

namespace codec {

// Weight planes of one contraction for the tensor cores: B = W^T, K-major
// [N][K], scaled by 2^e (max |W 2^e| in [1, 2)) and split into fp16 hi and lo.
struct TcWeights {
    CUtensorMap map_hi;      // over `hi` (CUtensorMap is itself 64-byte aligned)
    void* hi = nullptr;      // passes 3: __half [N][K / 32][32 hi | 32 lo]; passes 1: __half [N][K] (hi)
    float unscale = 1.f;     // 2^-e, applied to the accumulator
    int BN = 0;              // N tile (multiple of 32, <= 256)
    int n_tiles = 0;
    int passes = 3;          // 3: hi*hi + hi*lo + lo*hi; 1: hi*hi only (single fp16 pass)
    // the planes were complete before any kernel that may precede a GEMM in
    // its stream ran (uploaded by a synchronous copy): the GEMM may load them
    // before its grid dependency resolves
    bool b_static = false;
    // Narrower N tiles over the same planes (128 and/or 64 columns, when BN is
    // wider), for calls with too few tiles to fill the GPU: a 128 x N x 16 MMA
    // costs about N / 2 cycles above a floor near 48, so a narrow tile ends a
    // chunk sooner and more CTAs share the work.
    CUtensorMap map_alt[2];
    int bn_alt[2] = {0, 0};
    int n_alt = 0;
};

// Scratch of one standalone tensor-core conv: operand planes, and kOpWords
// words for its one-segment plan, weight scale and 1/alpha.
constexpr int kOpMaxCin = 4096;
constexpr int kOpWords = 16 + kOpMaxCin;
// Bounded waits of the GEMM kernel: every mbarrier wait gives up after
// `polls` polls (the CTA then raises the error flag, drains its copies and
// MMAs, frees TMEM and returns).  unarrived_wait != 0 is for verifying that
// path: the epilogue's first wait of each CTA then targets a barrier no role
// ever arrives on, so it runs out after `polls` polls on any input.
constexpr uint32_t kDefaultWaitPolls = 1u << 25;
struct TcWaitLimit {
    uint32_t polls = kDefaultWaitPolls;
    int unarrived_wait = 0;
};

struct TcOpScratch {
    TcWaitLimit wait;
    void* a_hi = nullptr;     // 2 a_elems fp16 from here on: a_lo == a_hi + a_elems
    void* a_lo = nullptr;
    size_t a_elems = 0;
    void* b_hi = nullptr;     // 2 b_elems fp16 from here on: b_lo == b_hi + b_elems
    void* b_lo = nullptr;
    size_t b_elems = 0;
    int* words = nullptr;
    int* err = nullptr;
};

// Per-state scratch for the A-operand planes (Snake applied, split into fp16
// hi and lo), big enough for the widest input of any contraction, plus the
// sticky flag a kernel sets when one of its bounded waits expires.
struct TcScratch {
    TcWaitLimit wait;
    void* a_hi = nullptr;     // 2 elems fp16 from here on (a_lo == a_hi + elems): the three-pass
    void* a_lo = nullptr;     // layout interleaves hi and lo over all of it, the one-pass mode uses hi
    size_t elems = 0;
    int* err = nullptr;
    float* ws = nullptr;  // chunk partials of split GEMMs
    size_t ws_floats = 0;
    TcOpScratch op;       // the same planes plus weight planes for codec_state_conv1d
};

// Sets the GEMM kernel's shared-memory carve-out; called once per codec.
cudaError_t tc_configure();
bool tc_eligible(int Cin, int N);
bool tc_pack_weights(const float* wkn, int ntaps, int Cin, int N, int passes, TcWeights* out,
                     std::vector<void*>& allocs);
bool tc_scratch_alloc(TcScratch* s, size_t elems, size_t b_elems, size_t ws_floats, std::vector<void*>& allocs);

// A-operand planes of rows x Cin: hi = fp16(a), lo = fp16(a - hi) (lo only
// when with_lo) with a = Snake(x) when alpha is given, else GELU(x) when gelu,
// else x.
cudaError_t launch_tc_prep(const float* x, const float* alpha, const float* inv_alpha, long long rows, int Cin,
                           TcScratch* scratch, bool with_lo, cudaStream_t s, bool gelu = false);
// The GEMM over the planes prepared by launch_tc_prep (a_rows rows); when it
// has too few tiles for the GPU it also launches the split reduction.
// *launches is incremented per kernel launched.
cudaError_t launch_tc_gemm(const GemmArgs& a, const TcWeights& w, PlanView plan, int n_row_tiles,
                           const TcScratch* scratch, long long a_rows, int num_sms, cudaStream_t s,
                           int* launches);

// y = conv(Snake_alpha(x)) + bias for one sequence: x [(k-1) dil + T][Cin]
// (history rows first), w [Cout][Cin][k], y [T][Cout], all device fp32;
// alpha and bias may be null.  Returns one of OP_*.
enum { OP_OK = 0, OP_BAD_ARG = 1, OP_TOO_BIG = 2, OP_CUDA = 3 };
// The argument and capacity checks of run_tc_conv1d alone (enqueues nothing):
// OP_BAD_ARG for an unsupported shape, then OP_TOO_BIG for one beyond sc.
int check_tc_conv1d(const TcOpScratch& sc, int T, int Cin, bool has_alpha, int Cout, int k, int dil);
int run_tc_conv1d(const TcOpScratch& sc, const float* x, int T, int Cin, const float* w, const float* bias,
                  const float* alpha, int Cout, int k, int dil, float* y, int num_sms, cudaStream_t s);

}  // namespace codec
