// Tensor-core (tcgen05 / TMEM / TMA) implicit-GEMM path with fp16 hi/lo
// split operands.  Declarations shared by the host runtime and tc_gemm.cu.
#pragma once

#include <vector>

#include "common.cuh"

namespace codec {

// Weight planes of one contraction for the tensor cores: B = W^T in K-major
// [N][K] fp16 hi and lo planes, scaled by 2^wexp before the split.
struct TcWeights {
    void* hi = nullptr;      // __half [N][K]
    void* lo = nullptr;
    float unscale = 1.f;     // 2^-wexp, applied to the accumulator
};

// Per-state scratch for the A-operand planes (Snake applied, split into
// fp16 hi and lo), big enough for the widest input of any contraction.
struct TcScratch {
    void* a_hi = nullptr;
    void* a_lo = nullptr;
    size_t elems = 0;
};

bool tc_eligible(int Cin, int N);
bool tc_pack_weights(const float* wkn, int ntaps, int Cin, int N, TcWeights* out,
                     std::vector<void*>& allocs);
bool tc_scratch_alloc(TcScratch* s, size_t elems, std::vector<void*>& allocs);
cudaError_t launch_gemm_tc(const GemmArgs& a, const TcWeights& w, PlanView plan, int n_row_tiles,
                           TcScratch* scratch, cudaStream_t s, int* launches);

}  // namespace codec
