// Sliding-window attention on the tensor cores for long windows (head width
// 64, window >= 128: the latent-input decoder's 251 positions at 200 Hz,
// blixt/phonon "Speed" item 7; softmax with max subtraction, item 11).
//
// A block takes up to 32 consecutive queries of one stream and one head, as
// the CUDA-core kernel does, and stages the keys and values they can see in
// shared memory (asynchronous 16-byte copies).  The keys start at a position
// rounded down to a multiple of 16, so that the value sums below run over
// groups of 16 keys fixed by absolute position: a query's result then does
// not depend on the block (and so the chunk) it came in.
//
//   scores  S = Q K^T / sqrt(64): warp-level fp16 MMAs (m16n8k16, fp32
//           accumulate) on the hi/lo split of both operands, hi*hi + hi*lo +
//           lo*hi per 16-dim step (the three-pass split of the GEMMs);
//   softmax a warp per query over its own window (max subtraction, fixed
//           butterflies), probabilities written in place and zero elsewhere;
//   output  O = P V / z with the same three-pass MMAs over 16-key groups.
//
// The split puts both operands within about 2^-22 of their fp32 values; a
// zero probability contributes exact zeros.
#include <cuda_fp16.h>

#include "kernels.h"

namespace codec {

namespace {

constexpr int kQ = 32;              // queries per block
constexpr int kDh = 64;             // head width
constexpr int kThreads = 512;       // 16 warps
constexpr int kLdK = kDh + 8;       // padded rows of K and Q (float2 row reads: conflict-free)
constexpr int kLdV = kDh + 4;       // padded rows of V (column reads across rows: conflict-free)

__device__ __forceinline__ void cp16(void* smem, const void* gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}

// hi = fp16(x), lo = fp16(x - hi) for two values, packed as the MMA reads them
// (the first value in the low half).
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo)
{
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// c += a b for one 16 x 8 x 16 step (a: 16 x 16 row-major fragment, b: 16 x 8
// column-major fragment, fp32 accumulators).
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, const uint32_t* b)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma3(float* c, const uint32_t* ah, const uint32_t* al, const uint32_t* bh,
                                     const uint32_t* bl)
{
    mma16816(c, ah, bh);
    mma16816(c, ah, bl);
    mma16816(c, al, bh);
}

__host__ __device__ __forceinline__ int round_up(int x, int m) { return (x + m - 1) / m * m; }

__global__ void __launch_bounds__(kThreads) swa_mma_kernel(
    const float* __restrict__ q, float* __restrict__ o, const float* __restrict__ kring,
    const float* __restrict__ vring, int d, int W, int R, int pos_r, PlanView plan, const int* __restrict__ qcum,
    void* planes, int planes_il)
{
    pdl_wait();
    pdl_launch();
    extern __shared__ float4 am_sm4[];
    const int h = blockIdx.y, blk = blockIdx.x;
    const int b = find_seg(qcum, plan.B, blk);
    const int n = (__ldg(plan.cf + b + 1) - __ldg(plan.cf + b)) * pos_r;
    const int tq0 = (blk - __ldg(qcum + b)) * kQ;
    const int nq = min(kQ, n - tq0);
    const long long p0 = __ldg(plan.pos0 + b) * pos_r + tq0;     // position of the block's first query
    const long long k_lo = p0 - W + 1 > 0 ? p0 - W + 1 : 0;
    const long long kst = k_lo & ~15LL;                            // first staged key, a multiple of 16
    const int nk = (int)(p0 + nq - kst);
    const int nk16 = round_up(nk, 16);
    const int ldp = round_up(nk16, 32) + 8;                        // padded rows of P (float2 row reads)
    float* sk = reinterpret_cast<float*>(am_sm4);                  // [nk16][kLdK]
    float* sv = sk + (size_t)nk16 * kLdK;                          // [nk16][kLdV]
    float* sq = sv + (size_t)nk16 * kLdV;                          // [kQ][kLdK]; later the output [kQ][kLdK]
    float* sp = sq + (size_t)kQ * kLdK;                            // [kQ][ldp]
    float* sz = sp + (size_t)kQ * ldp;                             // [kQ]
    const long long slot_base = (long long)__ldg(plan.slot + b) * R;
    const long long row0 = (long long)__ldg(plan.cf + b) * pos_r + tq0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;

    // staging: keys and values of positions kst .. kst + nk - 1 (zero rows up
    // to nk16), queries 0 .. nq - 1 (zero rows up to 32)
    for (int i = tid; i < nk16 * (kDh / 4); i += kThreads) {
        const int r = i / (kDh / 4), c4 = i - r * (kDh / 4);
        if (r < nk) {
            const long long at = (slot_base + ((kst + r) & (R - 1))) * d + h * kDh + 4 * c4;
            cp16(sk + r * kLdK + 4 * c4, kring + at);
            cp16(sv + r * kLdV + 4 * c4, vring + at);
        } else {
            *reinterpret_cast<float4*>(sk + r * kLdK + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(sv + r * kLdV + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    for (int i = tid; i < kQ * (kDh / 4); i += kThreads) {
        const int r = i / (kDh / 4), c4 = i - r * (kDh / 4);
        if (r < nq) cp16(sq + r * kLdK + 4 * c4, q + (row0 + r) * d + h * kDh + 4 * c4);
        else *reinterpret_cast<float4*>(sq + r * kLdK + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // scores: warp w takes query tile w & 1 and key tiles w >> 1, + 8, ...
    {
        const int qt = warp & 1;
        uint32_t ah[4][4], al[4][4];
#pragma unroll
        for (int ks = 0; ks < kDh / 16; ks++) {
            const float* r0 = sq + (qt * 16 + gid) * kLdK + 16 * ks + 2 * tig;
            const float* r1 = r0 + 8 * kLdK;
            const float2 x0 = *reinterpret_cast<const float2*>(r0), x1 = *reinterpret_cast<const float2*>(r1);
            const float2 x2 = *reinterpret_cast<const float2*>(r0 + 8), x3 = *reinterpret_cast<const float2*>(r1 + 8);
            split2(x0.x, x0.y, ah[ks][0], al[ks][0]);
            split2(x1.x, x1.y, ah[ks][1], al[ks][1]);
            split2(x2.x, x2.y, ah[ks][2], al[ks][2]);
            split2(x3.x, x3.y, ah[ks][3], al[ks][3]);
        }
        for (int kt = warp >> 1; kt < nk16 / 8; kt += kThreads / 64) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < kDh / 16; ks++) {
                const float* kr = sk + (kt * 8 + gid) * kLdK + 16 * ks + 2 * tig;
                const float2 y0 = *reinterpret_cast<const float2*>(kr), y1 = *reinterpret_cast<const float2*>(kr + 8);
                uint32_t bh[2], bl[2];
                split2(y0.x, y0.y, bh[0], bl[0]);
                split2(y1.x, y1.y, bh[1], bl[1]);
                mma3(c, ah[ks], al[ks], bh, bl);
            }
            const float scale = 0.125f;                         // 1 / sqrt(64)
            float* pr = sp + (qt * 16 + gid) * ldp + kt * 8 + 2 * tig;
            *reinterpret_cast<float2*>(pr) = make_float2(c[0] * scale, c[1] * scale);
            *reinterpret_cast<float2*>(pr + 8 * ldp) = make_float2(c[2] * scale, c[3] * scale);
        }
    }
    __syncthreads();

    // softmax of each query over its window; every other staged key gets 0
    for (int qi = warp; qi < kQ; qi += kThreads / 32) {
        float* pr = sp + qi * ldp;
        if (qi >= nq) {
            for (int i = lane; i < nk16; i += 32) pr[i] = 0.f;
            continue;
        }
        const long long pos = p0 + qi;
        const long long lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
        const int a = (int)(lo - kst), e = (int)(pos - kst);      // the window's first and last staged index
        float m = -INFINITY;
        for (int i = a + lane; i <= e; i += 32) m = fmaxf(m, pr[i]);
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
        float z = 0.f;
        for (int i = lane; i < nk16; i += 32) {
            float pe = 0.f;
            if (i >= a && i <= e) {
                pe = expf(pr[i] - m);
                z += pe;
            }
            pr[i] = pe;
        }
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) z += __shfl_xor_sync(0xffffffffu, z, sh);
        if (lane == 0) sz[qi] = 1.0f / z;
    }
    __syncthreads();

    // output: warp w takes query tile w & 1 and the 8 head channels 8 (w >> 1) ..
    {
        const int qt = warp & 1, dt = warp >> 1;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ks = 0; ks < nk16 / 16; ks++) {
            const float* p0r = sp + (qt * 16 + gid) * ldp + 16 * ks + 2 * tig;
            const float* p1r = p0r + 8 * ldp;
            const float2 x0 = *reinterpret_cast<const float2*>(p0r), x1 = *reinterpret_cast<const float2*>(p1r);
            const float2 x2 = *reinterpret_cast<const float2*>(p0r + 8), x3 = *reinterpret_cast<const float2*>(p1r + 8);
            uint32_t ah[4], al[4];
            split2(x0.x, x0.y, ah[0], al[0]);
            split2(x1.x, x1.y, ah[1], al[1]);
            split2(x2.x, x2.y, ah[2], al[2]);
            split2(x3.x, x3.y, ah[3], al[3]);
            const float* vr = sv + (16 * ks + 2 * tig) * kLdV + dt * 8 + gid;
            uint32_t bh[2], bl[2];
            split2(vr[0], vr[kLdV], bh[0], bl[0]);
            split2(vr[8 * kLdV], vr[9 * kLdV], bh[1], bl[1]);
            mma3(c, ah, al, bh, bl);
        }
        const int qa = qt * 16 + gid;
        float* so = sq + qa * kLdK + dt * 8 + 2 * tig;            // the queries are no longer needed
        const float za = sz[qa], zb = sz[qa + 8];
        *reinterpret_cast<float2*>(so) = make_float2(c[0] * za, c[1] * za);
        *reinterpret_cast<float2*>(so + 8 * kLdK) = make_float2(c[2] * zb, c[3] * zb);
    }
    __syncthreads();
    for (int i = tid; i < nq * (kDh / 4); i += kThreads) {
        const int r = i / (kDh / 4), c4 = i - r * (kDh / 4);
        const float4 y = *reinterpret_cast<const float4*>(sq + r * kLdK + 4 * c4);
        const int ch = h * kDh + 4 * c4;
        if (planes) plane_store4(planes, planes_il, row0 + r, d, ch, y);
        else *reinterpret_cast<float4*>(o + (row0 + r) * d + ch) = y;
    }
}

}  // namespace

size_t swa_mma_smem_bytes(int window)
{
    const int nk16 = round_up(kQ - 1 + window + 15, 16);
    const int ldp = round_up(nk16, 32) + 8;
    return sizeof(float) * ((size_t)nk16 * kLdK + (size_t)nk16 * kLdV + (size_t)kQ * kLdK + (size_t)kQ * ldp + kQ);
}

bool swa_mma_eligible(int dh, int window)
{
    return dh == kDh && window >= 128 && window <= kSwaWindowMax && swa_mma_smem_bytes(window) <= kSwaSmemMax;
}

cudaError_t configure_swa_mma()
{
    return cudaFuncSetAttribute(swa_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSwaSmemMax);
}

cudaError_t launch_swa_mma(const float* q, float* o, const float* kring, const float* vring, int d, int heads,
                           int window, int ring_R, int pos_r, PlanView plan, const int* qcum, int n_qblocks,
                           cudaStream_t s, void* planes, int planes_il)
{
    if (n_qblocks <= 0) return cudaSuccess;
    if (d / heads != kDh || !swa_mma_eligible(kDh, window) || (planes && d % 32 != 0)) return cudaErrorInvalidValue;
    launch_pdl(swa_mma_kernel, dim3(n_qblocks, heads), dim3(kThreads), swa_mma_smem_bytes(window), s, q, o, kring,
               vring, d, window, ring_R, pos_r, plan, qcum, planes, planes_il);
    return cudaGetLastError();
}

}  // namespace codec
