// Shared definitions of the CUDA library: launch descriptors, per-call plan
// layout and the small device helpers every kernel uses.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace codec {

constexpr int kMaxTaps = 16;
// Queries of one stream that one sliding-window attention block takes (the
// per-call plan counts each stream's attention blocks in these units).
constexpr int kSwaQueries = 32;

// Epilogue modes of the implicit-GEMM kernels (what happens to acc = A*B).
enum Epi : int {
    EPI_STORE = 0,   // out = acc + bias
    EPI_RESID = 1,   // out = res + acc + bias
    EPI_GELU = 2,    // out = gelu(acc + bias)
    EPI_MRF_FIRST = 3,  // out = res + acc + bias                (first resblock of an MRF)
    EPI_MRF_ADD = 4,    // out = out + (res + acc + bias)
    EPI_MRF_LAST = 5,   // out = (out + (res + acc + bias)) * scale
    EPI_QKV = 6,     // n < d: q[row][n] = acc; d <= n < 2d: K ring; 2d <= n: V ring
};

// Rows of a tensor in the per-call packed layout.  Stream segment b of a
// "level" with rate r (rows per frame) holds n_b * r chunk rows.  A prefixed
// layout puts P history rows in front of every segment, so that segment b's
// chunk row 0 sits at cf[b] * r + (b + 1) * P; a dense layout (P = 0) packs the
// chunk rows back to back.
struct Layout {
    int r;     // rows per frame
    int P;     // history rows in front of each segment (0 = dense)
};

__host__ __device__ inline long long seg_base(const Layout& L, const int* cf, int b)
{
    return (long long)cf[b] * L.r + (long long)(b + 1) * L.P;
}

// Per-call plan, uploaded to the device before the launches.  All arrays are
// indexed by batch entry b < B.
struct PlanView {
    int B;
    const int* cf;          // [B + 1] cumulative frames
    const int* slot;        // [B] state slot of batch entry b
    const long long* pos0;  // [B] frames the stream had decoded before this call
    const int* bidx;        // [B] row of b in the caller's codes / audio arrays
    const int* skip;        // [B] leading frames of b whose audio is not written (recompute
                            // mode's left context), or null for none
};

// Implicit-GEMM launch descriptor: out rows t of segment b are
//   epi( sum_{tap j} sum_{ci} A(in[base_in(b) + t - shift_j][ci]) * W[j*Cin + ci][n] ).
struct GemmArgs {
    const float* in;
    Layout in_l;
    int Cin;
    int ntaps;
    int shift[kMaxTaps];
    const float* alpha;      // Snake parameters on the A operand, or null
    const float* inv_alpha;
    int N, K;                // K = ntaps * Cin
    const float* w;          // fp32 [K][N] (CUDA-core path)
    const float* bias;       // bias[n % bias_mod] or null
    int bias_mod;
    float* out;
    Layout out_l;
    int out_C;               // elements per output row
    int out_step;            // output rows per input row (transposed-conv stride, else 1)
    const float* res;        // residual, same layout as out
    int epi;
    float scale;             // EPI_MRF_LAST
    // EPI_QKV
    float* kring;
    float* vring;
    int ring_R;              // ring rows per slot (power of two)
    int d;
    int pos_r;               // transformer rows (positions) per frame
    // tiling
    const int* tcum;         // [B + 1] cumulative row tiles of the input level
    int bm;
    // 1: input and output dense (P = 0), one tap, out_step 1 - row tiles run
    // over all segments' rows back to back (tile mt = rows 128 mt ...), since
    // no row reads another row; the q/K/V scatter finds each row's segment.
    int dense;
};

__device__ __forceinline__ int find_seg(const int* cum, int B, int x)
{
    // largest b with cum[b] <= x (cum[0] = 0, cum nondecreasing)
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cum + mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The same over rows of a level with r rows per frame: largest b with
// cum[b] * r <= x.
__device__ __forceinline__ int find_seg_r(const int* cum, int B, long long x, int r)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((long long)__ldg(cum + mid) * r <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Programmatic dependent launch.  The decoder's kernels are launched with
// programmatic stream serialisation, so a kernel may start (and do set-up that
// touches no global memory) while its predecessor in the stream still runs.
// pdl_wait() returns once every prerequisite grid has completed and its memory
// operations are visible (at once when there is none): every kernel calls it
// before its first global memory access and before any of its threads can
// exit, so a kernel's completion still implies its predecessors'.  Then
// pdl_launch() lets the kernel's own successor begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Enqueue kernel<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args)
{
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A tensor-core GEMM operand written by its producer instead of the prep
// kernel: value v of column n of `row` split into fp16 hi = fp16(v) and lo =
// fp16(v - hi), bit for bit as the prep kernel splits it, in the interleaved
// [rows][C / 32][32 hi | 32 lo] layout (il) or as the hi plane [rows][C].
__device__ __forceinline__ void plane_store1(void* planes, int il, long long row, int C, int n, float v)
{
    __half* p = static_cast<__half*>(planes);
    const __half h = __float2half_rn(v);
    if (il) {
        const long long at = row * 2 * C + (n >> 5) * 64 + (n & 31);
        p[at] = h;
        p[at + 32] = __float2half_rn(v - __half2float(h));
    } else {
        p[row * C + n] = h;
    }
}

// The same for four columns n .. n + 3 (n % 4 == 0): one 8-byte store per plane.
__device__ __forceinline__ void plane_store4(void* planes, int il, long long row, int C, int n, float4 v)
{
    const float e[4] = {v.x, v.y, v.z, v.w};
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const __half h0 = __float2half_rn(e[2 * i]), h1 = __float2half_rn(e[2 * i + 1]);
        const __half l0 = __float2half_rn(e[2 * i] - __half2float(h0));
        const __half l1 = __float2half_rn(e[2 * i + 1] - __half2float(h1));
        hw[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
        lw[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
    __half* p = static_cast<__half*>(planes);
    if (il) {
        const long long at = row * 2 * C + (n >> 5) * 64 + (n & 31);
        *reinterpret_cast<uint2*>(p + at) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(p + at + 32) = make_uint2(lw[0], lw[1]);
    } else {
        *reinterpret_cast<uint2*>(p + row * C + n) = make_uint2(hw[0], hw[1]);
    }
}

// Snake, x + sin(a x)^2 / a, with explicit roundings so every kernel that
// evaluates it produces the same bits for the same input.
__device__ __forceinline__ float snake_f(float x, float a, float inv_a)
{
    float s = sinf(__fmul_rn(a, x));
    return __fadd_rn(x, __fmul_rn(__fmul_rn(s, s), inv_a));
}

__device__ __forceinline__ float gelu_f(float x)
{
    return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

// Epilogue of both GEMM paths for one output element: acc is the finished
// dot product of output row t of batch entry b (row out_row of the output
// layout), column n.
__device__ __forceinline__ void gemm_store(const GemmArgs& a, const PlanView& plan, int b, int t,
                                           long long out_row, int n, float acc)
{
    float v = acc;
    if (a.bias) v += __ldg(a.bias + (n % a.bias_mod));
    const long long idx = out_row * a.out_C + n;
    switch (a.epi) {
    case EPI_STORE: a.out[idx] = v; break;
    case EPI_RESID: a.out[idx] = a.res[idx] + v; break;
    case EPI_GELU: a.out[idx] = gelu_f(v); break;
    case EPI_MRF_FIRST: a.out[idx] = a.res[idx] + v; break;
    case EPI_MRF_ADD: a.out[idx] = a.out[idx] + (a.res[idx] + v); break;
    case EPI_MRF_LAST: a.out[idx] = (a.out[idx] + (a.res[idx] + v)) * a.scale; break;
    case EPI_QKV: {
        if (n < a.d) {
            a.out[out_row * a.d + n] = v;
        } else {
            if (b < 0) {            // dense tiling: t is the row over all segments
                b = find_seg_r(plan.cf, plan.B, t, a.pos_r);
                t -= __ldg(plan.cf + b) * a.pos_r;
            }
            const long long pos = __ldg(plan.pos0 + b) * a.pos_r + t;
            const long long rr = (long long)__ldg(plan.slot + b) * a.ring_R + (pos & (a.ring_R - 1));
            if (n < 2 * a.d) a.kring[rr * a.d + (n - a.d)] = v;
            else a.vring[rr * a.d + (n - 2 * a.d)] = v;
        }
        break;
    }
    default: break;
    }
}

}  // namespace codec
