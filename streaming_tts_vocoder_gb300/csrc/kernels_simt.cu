// CUDA-core kernels of the decoder: codebook gather-sum, fp32 implicit-GEMM
// convolution (the reference-precision contraction and the path for layers too
// narrow for the tensor cores), RMSNorm, sliding-window attention over the
// ring KV, the final Snake + conv + tanh stencil, and the per-call history
// bookkeeping (fill, commit, reset).
#include <math.h>

#include "kernels.h"

namespace codec {

// ---------------------------------------------------------------- gather --
// e[row] = sum_q CB_q[code[q][t]] in fp32, q ascending (vllm-omni "Edge TTS
// design", section 1.3: RVQ embedding sum).  One block per (frame t, batch
// entry b) of a grid of the call's longest chunk x its entries (blocks past
// an entry's frames return at once), one float4 of channels per thread:
// every load is a 128-bit load of a codebook row.  A code outside [0, V)
// zeroes the row and sets the slot's sticky bit.
__global__ void __launch_bounds__(128) rvq_gather_kernel(
    const float* __restrict__ cb, int Q, int V, int E, const int* __restrict__ codes, int T_max,
    PlanView plan, const int* __restrict__ bidx, float* __restrict__ e, Layout el,
    unsigned* __restrict__ err_words)
{
    pdl_wait();
    pdl_launch();
    __shared__ int sc[64];
    __shared__ int sbad;
    const int b = blockIdx.y, t = blockIdx.x;
    if (t >= __ldg(plan.cf + b + 1) - __ldg(plan.cf + b)) return;
    if (threadIdx.x == 0) sbad = 0;
    __syncthreads();
    const int* cr = codes + ((long long)__ldg(bidx + b) * Q) * T_max + t;
    for (int q = threadIdx.x; q < Q; q += blockDim.x) {
        int c = __ldg(cr + (long long)q * T_max);
        sc[q] = c;
        if (c < 0 || c >= V) atomicOr(&sbad, 1);
    }
    __syncthreads();
    float4* out = reinterpret_cast<float4*>(e + (seg_base(el, plan.cf, b) + t) * E);
    const int E4 = E >> 2;
    if (sbad) {
        for (int c4 = threadIdx.x; c4 < E4; c4 += blockDim.x) out[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (threadIdx.x == 0) atomicOr(err_words + __ldg(plan.slot + b), 1u);
        return;
    }
    for (int c4 = threadIdx.x; c4 < E4; c4 += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < Q; q++) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(cb + ((long long)q * V + sc[q]) * E) + c4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        out[c4] = acc;
    }
}

cudaError_t launch_rvq_gather(const float* cb, int Q, int V, int E, const int* codes, int T_max,
                              PlanView plan, float* e, Layout el, unsigned* err_words,
                              int max_frames, cudaStream_t s)
{
    if (max_frames <= 0 || plan.B <= 0) return cudaSuccess;
    launch_pdl(rvq_gather_kernel, dim3(max_frames, plan.B), dim3(128), 0, s, cb, Q, V, E, codes, T_max, plan,
               plan.bidx, e, el, err_words);
    return cudaGetLastError();
}

// ---------------------------------------------------------- latent fill --
// Latent-input decoder: e[row] = x[row] * sigma + mu (per channel, one
// rounding) for every frame of the call, from the caller's [B][T_max][L]
// latents into the level-0 buffer, whose rows are ldo >= L floats apart
// (blixt/phonon "Weights": the codec's latents are denormalised before the
// projection).  One thread per float4.
__global__ void __launch_bounds__(256) latent_fill_kernel(const float* __restrict__ x, int L, int T_max,
                                                          PlanView plan, const float* __restrict__ mu,
                                                          const float* __restrict__ sigma, float* __restrict__ e,
                                                          Layout el, int total_rows, int ldo)
{
    pdl_wait();
    pdl_launch();
    const int L4 = L >> 2;
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= (long long)total_rows * L4) return;
    const int row = (int)(i / L4), c4 = (int)(i - (long long)row * L4);
    const int b = find_seg(plan.cf, plan.B, row);
    const int t = row - __ldg(plan.cf + b);
    const float4 v = __ldg(reinterpret_cast<const float4*>(x + ((long long)__ldg(plan.bidx + b) * T_max + t) * L) + c4);
    const float4 m = __ldg(reinterpret_cast<const float4*>(mu) + c4);
    const float4 sg = __ldg(reinterpret_cast<const float4*>(sigma) + c4);
    reinterpret_cast<float4*>(e + (seg_base(el, plan.cf, b) + t) * ldo)[c4] =
        make_float4(__fmaf_rn(v.x, sg.x, m.x), __fmaf_rn(v.y, sg.y, m.y), __fmaf_rn(v.z, sg.z, m.z),
                    __fmaf_rn(v.w, sg.w, m.w));
}

cudaError_t launch_latent_fill(const float* x, int L, int T_max, PlanView plan, const float* mu,
                               const float* sigma, float* e, Layout el, int total_rows, cudaStream_t s, int ldo)
{
    if (total_rows <= 0) return cudaSuccess;
    if (ldo <= 0) ldo = L;
    if (L % 4 != 0 || ldo % 4 != 0 || ldo < L) return cudaErrorInvalidValue;
    const long long n = (long long)total_rows * (L / 4);
    launch_pdl(latent_fill_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, x, L, T_max, plan, mu, sigma,
               e, el, total_rows, ldo);
    return cudaGetLastError();
}

// ------------------------------------------------------ fp32 implicit GEMM --
// out[t][n] = epi( sum_j sum_ci A(in[base(b) + t - shift_j][ci]) W[j Cin + ci][n] )
// 64 x 64 output tile per block, 16-deep K slices in shared memory, 4 x 4
// outputs per thread.  Each output's sum runs over (tap, channel) in
// ascending order whatever the tile or batch it falls in, so the result of a
// row does not depend on how the streams were packed.
constexpr int SB_M = 64, SB_N = 64, SB_K = 16;

__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a, PlanView plan)
{
    pdl_wait();
    pdl_launch();
    __shared__ float As[SB_K][SB_M + 4];
    __shared__ float Bs[SB_K][SB_N + 4];
    const int tile = blockIdx.x;
    const int b = find_seg(a.tcum, plan.B, tile);
    const int seg_rows = (__ldg(plan.cf + b + 1) - __ldg(plan.cf + b)) * a.in_l.r;
    const int t0 = (tile - __ldg(a.tcum + b)) * SB_M;
    const int nrows = min(SB_M, seg_rows - t0);
    const long long in_base = seg_base(a.in_l, plan.cf, b) + t0;
    const int n0 = blockIdx.y * SB_N;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;

    const int am = tid >> 2, ak = (tid & 3) * 4;   // A: row am, channels ak..ak+3
    const int bk = tid >> 4, bn = (tid & 15) * 4;  // B: k row bk, columns bn..bn+3
    for (int j = 0; j < a.ntaps; j++) {
        const long long rowA = in_base - a.shift[j];
        for (int c0 = 0; c0 < a.Cin; c0 += SB_K) {
            float av[4] = {0.f, 0.f, 0.f, 0.f};
            if (am < nrows && c0 + ak < a.Cin) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(a.in + (rowA + am) * a.Cin + c0 + ak));
                av[0] = x.x; av[1] = x.y; av[2] = x.z; av[3] = x.w;
                if (a.alpha) {
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        av[i] = snake_f(av[i], __ldg(a.alpha + c0 + ak + i), __ldg(a.inv_alpha + c0 + ak + i));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; i++) As[ak + i][am] = av[i];
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c0 + bk < a.Cin && n0 + bn < a.N)
                w = __ldg(reinterpret_cast<const float4*>(a.w + (long long)(j * a.Cin + c0 + bk) * a.N + n0 + bn));
            Bs[bk][bn + 0] = w.x; Bs[bk][bn + 1] = w.y; Bs[bk][bn + 2] = w.z; Bs[bk][bn + 3] = w.w;
            __syncthreads();
#pragma unroll
            for (int k = 0; k < SB_K; k++) {
                float ar[4], br[4];
#pragma unroll
                for (int i = 0; i < 4; i++) { ar[i] = As[k][ty * 4 + i]; br[i] = Bs[k][tx * 4 + i]; }
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) acc[i][jj] = fmaf(ar[i], br[jj], acc[i][jj]);
            }
            __syncthreads();
        }
    }
    const long long out_base = seg_base(a.out_l, plan.cf, b);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int m = ty * 4 + i;
        if (m >= nrows) continue;
        const int t = t0 + m;
        const long long out_row = out_base + (long long)t * a.out_step;
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int n = n0 + tx * 4 + jj;
            if (n < a.N) gemm_store(a, plan, b, t, out_row, n, acc[i][jj]);
        }
    }
}

cudaError_t launch_gemm_simt(const GemmArgs& a, PlanView plan, int n_row_tiles, cudaStream_t s)
{
    if (n_row_tiles <= 0) return cudaSuccess;
    // A rows and W rows are read as float4s
    if (a.Cin % 4 != 0 || a.N % 4 != 0) return cudaErrorInvalidValue;
    dim3 grid(n_row_tiles, (a.N + SB_N - 1) / SB_N);
    launch_pdl(gemm_simt_kernel, dim3(grid), dim3(256), 0, s, a, plan);
    return cudaGetLastError();
}

// --------------------------------------------------------------- RMSNorm --
// y = x / sqrt(mean(x^2) + eps) * g, one warp per row; the row's sum of
// squares runs lane-strided then through a fixed butterfly.
// planes set: the normalised row goes straight into a tensor-core GEMM's
// operand planes (row of layout yl) instead of y.  PR: float4s of the row a
// lane keeps in registers (the whole row is loaded at once, d <= 128 PR),
// or 0 for a loop over any width.  Rows of dense layouts (no history rows in
// either) need no segment lookup: row r is layout row r.
template <int PR, bool kGainsEarly>
__global__ void rms_norm_kernel(const float* __restrict__ x, Layout xl, const float* __restrict__ g,
                                float eps, float* __restrict__ y, Layout yl, int d, PlanView plan,
                                int total_rows, void* planes, int planes_il)
{
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int d4 = d >> 2;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    // the gains are weights, written before any kernel of the stream ran:
    // with few rows (latency-bound) they are loaded before the wait for the
    // earlier kernels; with many, the registers that takes cost occupancy
    float4 gw[PR > 0 && kGainsEarly ? PR : 1];
    if constexpr (PR > 0 && kGainsEarly) {
#pragma unroll
        for (int i = 0; i < PR; i++) {
            const int c = lane + 32 * i;
            gw[i] = c < d4 ? __ldg(g4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();
    pdl_launch();
    if (row >= total_rows) return;
    long long xrow = row, yrow = row;
    if (xl.P != 0 || yl.P != 0) {
        // xl.r rows per frame (yl has the same rate)
        const int b = find_seg_r(plan.cf, plan.B, row, xl.r);
        const int t = row - __ldg(plan.cf + b) * xl.r;
        xrow = seg_base(xl, plan.cf, b) + t;
        yrow = seg_base(yl, plan.cf, b) + t;
    }
    const float4* xr = reinterpret_cast<const float4*>(x + xrow * d);
    float4* yr = reinterpret_cast<float4*>(y + yrow * d);
    float ss = 0.f;
    if constexpr (PR > 0) {
        float4 v[PR > 0 ? PR : 1];
#pragma unroll
        for (int i = 0; i < PR; i++) {
            const int c = lane + 32 * i;
            v[i] = c < d4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < PR; i++)
            if (lane + 32 * i < d4) {
                ss = fmaf(v[i].x, v[i].x, ss); ss = fmaf(v[i].y, v[i].y, ss);
                ss = fmaf(v[i].z, v[i].z, ss); ss = fmaf(v[i].w, v[i].w, ss);
            }
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss / (float)d + eps);
#pragma unroll
        for (int i = 0; i < PR; i++) {
            const int c = lane + 32 * i;
            if (c < d4) {
                float4 w;
                if constexpr (kGainsEarly) w = gw[i];
                else w = __ldg(g4 + c);
                const float4 o = make_float4(v[i].x * r * w.x, v[i].y * r * w.y, v[i].z * r * w.z, v[i].w * r * w.w);
                if (planes) plane_store4(planes, planes_il, yrow, d, 4 * c, o);
                else yr[c] = o;
            }
        }
    } else {
        for (int c = lane; c < d4; c += 32) {
            const float4 v = xr[c];
            ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss); ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss / (float)d + eps);
        for (int c = lane; c < d4; c += 32) {
            const float4 v = xr[c], w = __ldg(g4 + c);
            const float4 o = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
            if (planes) plane_store4(planes, planes_il, yrow, d, 4 * c, o);
            else yr[c] = o;
        }
    }
}

cudaError_t launch_rms_norm(const float* x, Layout xl, const float* g, float eps, float* y, Layout yl,
                            int d, PlanView plan, int total_rows, cudaStream_t s, void* planes, int planes_il)
{
    if (planes && (d % 32 != 0)) return cudaErrorInvalidValue;
    if (total_rows <= 0) return cudaSuccess;
    const int threads = 256, rows_per_block = threads / 32;
    const dim3 grid((total_rows + rows_per_block - 1) / rows_per_block);
    if (d <= 1024 && total_rows <= 2048)
        launch_pdl(rms_norm_kernel<8, true>, grid, dim3(threads), 0, s, x, xl, g, eps, y, yl, d, plan, total_rows,
                   planes, planes_il);
    else if (d <= 1024)
        launch_pdl(rms_norm_kernel<8, false>, grid, dim3(threads), 0, s, x, xl, g, eps, y, yl, d, plan, total_rows,
                   planes, planes_il);
    else
        launch_pdl(rms_norm_kernel<0, false>, grid, dim3(threads), 0, s, x, xl, g, eps, y, yl, d, plan, total_rows,
                   planes, planes_il);
    return cudaGetLastError();
}

// 16-byte global -> shared copy that bypasses the registers (both addresses
// 16-byte aligned), and its group commit / wait.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------- sliding-window attention --
// A block takes up to kSwaQueries consecutive queries of one stream and one
// head.  It stages the keys and values of every position they can see (at
// most kSwaQueries + W - 1 rows of the stream's ring: position p lives in
// ring row p mod R) in shared memory once, by asynchronous 16-byte copies,
// then runs three passes over the whole block: every (query, key) score (a
// thread per 4 x 4 tile of pairs, each dot product over the head's channels
// in ascending order), the softmax of each query (a warp per query: lane i
// takes keys lo + i, lo + 32 + i, ... of the query's own window lo .. p, max
// and denominator through a fixed butterfly), and every output channel (a
// thread per pair of queries and four channels, each value sum over its
// query's window keys in position order).  This is the CUDA-core kernel;
// long windows with 64-wide heads take the tensor-core one in the
// tensor-core precision modes (attention_mma.cu).
// A query at absolute position p attends positions max(0, p - W + 1) .. p, and
// every sum it takes runs in an order fixed by its own window, so its result
// never depends on how the stream was chunked (blixt/phonon "Speed" item 7:
// a ring of keys and values; item 11: softmax with max subtraction).
constexpr int kSwaMaxW = kSwaWindowMax;
constexpr int kSwaMaxDh = 128;
constexpr int kSwaThreads = 512;
constexpr int kSwaWarps = kSwaThreads / 32;
constexpr int kSwaMaxSmem = (int)kSwaSmemMax;

// planes set: the attention output goes straight into the out-projection's
// tensor-core operand planes (dense rows) instead of o.
__global__ void __launch_bounds__(kSwaThreads, 2) swa_kernel(
    const float* __restrict__ q, float* __restrict__ o, const float* __restrict__ kring,
    const float* __restrict__ vring, int d, int heads, int W, int R, int pos_r, PlanView plan,
    const int* __restrict__ qcum, void* planes, int planes_il)
{
    pdl_wait();
    pdl_launch();
    extern __shared__ float4 swa_sm4[];
    const int dh = d / heads;
    const int dh4 = dh >> 2;
    const int ld4 = dh4 + 1;                            // padded rows (float4 units): conflict-free row reads
    const int maxk = kSwaQueries + W - 1;
    const int lds = maxk + 1;
    float4* sk = swa_sm4;                               // [maxk][ld4]
    float4* sv = sk + (size_t)maxk * ld4;               // [maxk][ld4]
    float4* sq = sv + (size_t)maxk * ld4;               // [kSwaQueries][ld4]
    float* sp = reinterpret_cast<float*>(sq + (size_t)kSwaQueries * ld4);   // [kSwaQueries][lds] scores, then e^(s - m)
    float* sz = sp + (size_t)kSwaQueries * lds;         // [kSwaQueries] 1 / denominator
    const int h = blockIdx.y;
    const int blk = blockIdx.x;
    const int b = find_seg(qcum, plan.B, blk);
    // pos_r transformer rows (positions) per frame
    const int n = (__ldg(plan.cf + b + 1) - __ldg(plan.cf + b)) * pos_r;
    const int tq0 = (blk - __ldg(qcum + b)) * kSwaQueries;
    const int nq = min(kSwaQueries, n - tq0);
    const long long p0 = __ldg(plan.pos0 + b) * pos_r + tq0;   // position of the block's first query
    const long long kstart = p0 - W + 1 > 0 ? p0 - W + 1 : 0;
    const int nk = (int)(p0 + nq - kstart);             // keys the block's queries can see
    const long long slot_base = (long long)__ldg(plan.slot + b) * R;
    const long long row0 = (long long)__ldg(plan.cf + b) * pos_r + tq0;
    const int tid = threadIdx.x;
    // staging by asynchronous 16-byte copies, every one of a thread's in
    // flight at once: keys and queries (group 0), then values (group 1),
    // which land while the scores and the softmax run
    for (int i = tid; i < nk * dh4; i += kSwaThreads) {
        const int r = i / dh4, c4 = i - r * dh4;
        const long long at = (slot_base + ((kstart + r) & (R - 1))) * d + h * dh + 4 * c4;
        cp_async16(sk + r * ld4 + c4, kring + at);
    }
    for (int i = tid; i < nq * dh4; i += kSwaThreads) {
        const int r = i / dh4, c4 = i - r * dh4;
        cp_async16(sq + r * ld4 + c4, q + (row0 + r) * d + h * dh + 4 * c4);
    }
    cp_async_commit();
    for (int i = tid; i < nk * dh4; i += kSwaThreads) {
        const int r = i / dh4, c4 = i - r * dh4;
        const long long at = (slot_base + ((kstart + r) & (R - 1))) * d + h * dh + 4 * c4;
        cp_async16(sv + r * ld4 + c4, vring + at);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    // scores of every (query, key) pair the block holds, in register tiles of
    // 4 queries x 4 keys per thread (8 shared loads per 64 FMAs); each dot
    // product still runs over the channels in ascending order.  A thread's keys
    // are j, j + nk4, j + 2 nk4, j + 3 nk4, so consecutive threads read
    // consecutive key rows (conflict-free 128-bit loads); keys outside a
    // query's window are skipped
    const float scale = 1.0f / sqrtf((float)dh);
    const int nk4 = (nk + 3) >> 2;
    const int nq4 = (nq + 3) >> 2;
    for (int i = tid; i < nq4 * nk4; i += kSwaThreads) {
        const int qg = i / nk4, j = i - qg * nk4;
        const float4* kr[4];
        const float4* qr[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            kr[u] = sk + min(j + u * nk4, nk - 1) * ld4;
            qr[u] = sq + min(4 * qg + u, nq - 1) * ld4;
        }
        float dot[4][4];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int u = 0; u < 4; u++) dot[a][u] = 0.f;
        for (int c4 = 0; c4 < dh4; c4++) {
            float4 k4[4], q4[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                k4[u] = kr[u][c4];
                q4[u] = qr[u][c4];
            }
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    dot[a][u] = fmaf(q4[a].x, k4[u].x, dot[a][u]);
                    dot[a][u] = fmaf(q4[a].y, k4[u].y, dot[a][u]);
                    dot[a][u] = fmaf(q4[a].z, k4[u].z, dot[a][u]);
                    dot[a][u] = fmaf(q4[a].w, k4[u].w, dot[a][u]);
                }
        }
#pragma unroll
        for (int a = 0; a < 4; a++) {
            const int qi = 4 * qg + a;
            const long long pos = p0 + qi;
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int jj = j + u * nk4;
                const long long kp = kstart + jj;
                if (qi < nq && jj < nk && kp <= pos && kp >= pos - W + 1) sp[qi * lds + jj] = dot[a][u] * scale;
            }
        }
    }
    __syncthreads();
    const int wib = tid >> 5, lane = tid & 31;
    for (int qi = wib; qi < nq; qi += kSwaWarps) {
        const long long pos = p0 + qi;
        const long long lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
        const int nkq = (int)(pos - lo + 1);
        float* pr = sp + qi * lds + (int)(lo - kstart);  // the query's window, key lo first
        float m = -INFINITY;
        for (int i = lane; i < nkq; i += 32) m = fmaxf(m, pr[i]);
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
        float z = 0.f;
        for (int i = lane; i < nkq; i += 32) {
            const float pe = expf(pr[i] - m);
            pr[i] = pe;
            z += pe;
        }
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) z += __shfl_xor_sync(0xffffffffu, z, sh);
        if (lane == 0) sz[qi] = 1.0f / z;
    }
    cp_async_wait<0>();
    __syncthreads();
    // outputs: a thread takes two consecutive queries and one float4 column
    // (consecutive threads read consecutive 16-byte columns: conflict-free),
    // so each value row it loads serves both queries.  Their windows differ
    // by one key at each end: the first query's is union keys 0 .. n0 - 1,
    // the second's d1 .. n0 (d1 = 0 while both windows start at position 0);
    // each channel's sum runs over its own query's keys in position order.
    const int npair = (nq + 1) >> 1;
    for (int i = tid; i < npair * dh4; i += kSwaThreads) {
        const int qp = i / dh4, c4 = i - qp * dh4;
        const int qa = 2 * qp;
        const bool two = qa + 1 < nq;
        const long long pos = p0 + qa;
        const long long lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
        const int n0 = (int)(pos - lo + 1);
        const int d1 = pos + 1 - W + 1 > 0 ? 1 : 0;      // the second window's first key in the union
        const int off = (int)(lo - kstart);
        const float* pa = sp + qa * lds + off;
        const float* pb = sp + (qa + 1) * lds + off + d1;  // pb[k - d1]: the second query's key k of the union
        const float4* vc = sv + (size_t)off * ld4 + c4;
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
        int k = 0;
        if (d1) {
            const float pk = pa[0];
            const float4 v = vc[0];
            acc0.x = fmaf(pk, v.x, acc0.x); acc0.y = fmaf(pk, v.y, acc0.y);
            acc0.z = fmaf(pk, v.z, acc0.z); acc0.w = fmaf(pk, v.w, acc0.w);
            k = 1;
        }
        if (two) {
            for (; k < n0; k++) {
                const float4 v = vc[(size_t)k * ld4];
                const float pk = pa[k], qk = pb[k - d1];
                acc0.x = fmaf(pk, v.x, acc0.x); acc0.y = fmaf(pk, v.y, acc0.y);
                acc0.z = fmaf(pk, v.z, acc0.z); acc0.w = fmaf(pk, v.w, acc0.w);
                acc1.x = fmaf(qk, v.x, acc1.x); acc1.y = fmaf(qk, v.y, acc1.y);
                acc1.z = fmaf(qk, v.z, acc1.z); acc1.w = fmaf(qk, v.w, acc1.w);
            }
            const float4 v = vc[(size_t)n0 * ld4];
            const float qk = pb[n0 - d1];
            acc1.x = fmaf(qk, v.x, acc1.x); acc1.y = fmaf(qk, v.y, acc1.y);
            acc1.z = fmaf(qk, v.z, acc1.z); acc1.w = fmaf(qk, v.w, acc1.w);
        } else {
            for (; k < n0; k++) {
                const float4 v = vc[(size_t)k * ld4];
                const float pk = pa[k];
                acc0.x = fmaf(pk, v.x, acc0.x); acc0.y = fmaf(pk, v.y, acc0.y);
                acc0.z = fmaf(pk, v.z, acc0.z); acc0.w = fmaf(pk, v.w, acc0.w);
            }
        }
        const int ch = h * dh + 4 * c4;
        for (int e = 0; e < (two ? 2 : 1); e++) {
            const float4 acc = e ? acc1 : acc0;
            const float iz = sz[qa + e];
            const float4 y = make_float4(acc.x * iz, acc.y * iz, acc.z * iz, acc.w * iz);
            if (planes) plane_store4(planes, planes_il, row0 + qa + e, d, ch, y);
            else *reinterpret_cast<float4*>(o + (row0 + qa + e) * d + ch) = y;
        }
    }
}

size_t swa_smem_bytes(int dh, int window)
{
    const size_t maxk = (size_t)kSwaQueries + window - 1;
    const size_t ld4 = (size_t)dh / 4 + 1;
    return 16 * (2 * maxk * ld4 + (size_t)kSwaQueries * ld4) + 4 * ((size_t)kSwaQueries * (maxk + 1) + kSwaQueries);
}

cudaError_t launch_swa(const float* q, float* o, const float* kring, const float* vring, int d,
                       int heads, int window, int ring_R, int pos_r, PlanView plan, const int* qcum, int n_qblocks,
                       cudaStream_t s, void* planes, int planes_il, bool tensor_cores)
{
    if (n_qblocks <= 0) return cudaSuccess;
    if (planes && (d % 32 != 0)) return cudaErrorInvalidValue;
    const int dh = d / heads;
    if (dh > kSwaMaxDh || dh % 4 != 0 || window > kSwaMaxW) return cudaErrorInvalidValue;
    if (tensor_cores && swa_mma_eligible(dh, window))
        return launch_swa_mma(q, o, kring, vring, d, heads, window, ring_R, pos_r, plan, qcum, n_qblocks, s, planes,
                              planes_il);
    const size_t smem = swa_smem_bytes(dh, window);
    if (smem > (size_t)kSwaMaxSmem) return cudaErrorInvalidValue;
    launch_pdl(swa_kernel, dim3(n_qblocks, heads), dim3(kSwaThreads), smem, s, q, o, kring, vring, d, heads,
               window, ring_R, pos_r, plan, qcum, planes, planes_il);
    return cudaGetLastError();
}

// ------------------------------------------------ final Snake-conv-tanh --
// y[t] = tanh(b + sum_j p_j[t - (k-1) + j]), p_j[r] = sum_c w[j][c] snake(x[r][c]),
// C -> 1.  One thread per input row computes that row's k partial dot
// products (its channels read once, Snake applied once per element) into
// shared memory; each warp brings its 32 rows' channels through shared
// memory 32 at a time with coalesced 128-bit loads.  Then one thread per
// output row sums its k partials in tap order.  A block covers 128 output rows and
// the k-1 history rows before them.  One input row in, one sample out
// (blixt/phonon "Open work": a direct kernel for the last convolution with 1
// output channel); with C Snakes per sample its cost is the sine, so this
// kernel takes it as a Cody-Waite reduction of a x to [-pi, pi] (2 pi split
// into a float and its remainder) and the hardware sine there (absolute error
// a few 1e-7, against about 1e-7 for sinf), and forms x + sin^2 / a with one
// fused multiply-add; nothing else reads this Snake.
constexpr int kFinalTile = 128;
constexpr int kFinalWarps = kFinalTile / 32 + 1;   // four for the tile's rows, one for the k - 1 before them
constexpr int kFinalMaxK = 16;
constexpr int kFinalMaxSmem = (int)kFinalSmemMax;

// The Snake of two channels' values at once, in packed fp32 operations (each
// half rounds as the scalar operation would).
__device__ __forceinline__ float2 snake_final2(float2 x, float2 a, float2 inv_a)
{
    const float2 y = __fmul2_rn(a, x);
    const float2 t = __fmul2_rn(y, make_float2(0.159154943091895336f, 0.159154943091895336f));
    const float2 nk = make_float2(-rintf(t.x), -rintf(t.y));     // -(y / (2 pi)), nearest integer
    float2 r = __ffma2_rn(nk, make_float2(6.28318548202514648f, 6.28318548202514648f), y);   // 2 pi as a float
    r = __ffma2_rn(nk, make_float2(-1.7484555314695172e-7f, -1.7484555314695172e-7f), r);   // and the rest
    const float2 sn = make_float2(__sinf(r.x), __sinf(r.y));
    return __ffma2_rn(__fmul2_rn(sn, sn), inv_a, x);
}

// KP: taps padded to 8 or 16.  The weights sit in shared memory as [C][KP]
// (zero beyond k) and are read as float4s, the Snake parameters of a channel
// pair as one float4 (a_c, a_c+1, 1/a_c, 1/a_c+1).  Snake runs on channel
// pairs and the tap partials on tap pairs in packed fp32 (one instruction per
// two roundings, each the one the scalar code makes), so a channel costs half
// a Snake, KP/2 packed FMAs and KP/4 + 1/2 shared loads.
// One warp's rows r0 .. r0 + 31 (those below `rows`) of the tile: their
// channels come through shared memory 32 at a time, loaded by the whole warp
// (each load instruction covers whole 128-byte row segments), and each lane
// then takes its own row's 32 channels: Snake, then the KP tap partials in
// channel order.
template <int KP>
__device__ __forceinline__ void final_rows(const float* __restrict__ x, long long base, int C, int rows, int r0,
                                           const float4* sw, const float4* sa, float4* stg, int lane, float2* part)
{
    constexpr int kPitch = 9;                                   // float4s per staged row (8 + 1 pad)
#pragma unroll
    for (int j = 0; j < KP / 2; j++) part[j] = make_float2(0.f, 0.f);
    for (int c0 = 0; c0 < C; c0 += 32) {
        const int nq = min(32, C - c0) >> 2;                    // float4s of this chunk per row
        __syncwarp();
        for (int i = lane; i < 32 * nq; i += 32) {
            const int rr = i / nq, q = i - rr * nq;
            if (r0 + rr < rows)
                stg[rr * kPitch + q] = __ldg(reinterpret_cast<const float4*>(x + (base + r0 + rr) * C + c0) + q);
        }
        __syncwarp();
        if (r0 + lane < rows) {
            for (int q = 0; q < nq; q++) {
                const float4 v = stg[lane * kPitch + q];
                const int cb = c0 + 4 * q;
                const float4 p0 = sa[cb >> 1], p1 = sa[(cb >> 1) + 1];
                const float2 s01 = snake_final2(make_float2(v.x, v.y), make_float2(p0.x, p0.y), make_float2(p0.z, p0.w));
                const float2 s23 = snake_final2(make_float2(v.z, v.w), make_float2(p1.x, p1.y), make_float2(p1.z, p1.w));
                const float sn[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float2 s2 = make_float2(sn[u], sn[u]);
#pragma unroll
                    for (int g = 0; g < KP / 4; g++) {
                        const float4 wq = sw[(cb + u) * (KP / 4) + g];
                        part[2 * g] = __ffma2_rn(make_float2(wq.x, wq.y), s2, part[2 * g]);
                        part[2 * g + 1] = __ffma2_rn(make_float2(wq.z, wq.w), s2, part[2 * g + 1]);
                    }
                }
            }
        }
    }
}

template <int KP>
__global__ void __launch_bounds__(kFinalWarps * 32) final_conv_kernel(
    const float* __restrict__ x, Layout xl, int C, const float* __restrict__ w,
    const float* __restrict__ bias, const float* __restrict__ alpha,
    const float* __restrict__ inv_alpha, int k, float* __restrict__ audio,
    float* __restrict__ pre_tanh, long long audio_ld, int spf, PlanView plan, const int* __restrict__ bidx,
    const int* __restrict__ tcum)
{
    pdl_wait();
    pdl_launch();
    extern __shared__ float4 sm4[];
    float4* sw = sm4;                                                   // [C][KP / 4]
    float4* sa = sm4 + (size_t)C * (KP / 4);                            // [C / 2] channel-pair Snake parameters
    float4* stg = sa + C / 2 + (threadIdx.x >> 5) * 32 * 9;             // per warp [32][9]
    float* sp = reinterpret_cast<float*>(sa + C / 2 + kFinalWarps * 32 * 9);
    // sp: [kFinalTile + k - 1][k] partials
    const int tile = blockIdx.x;
    const int b = find_seg(tcum, plan.B, tile);
    const int seg_rows = (__ldg(plan.cf + b + 1) - __ldg(plan.cf + b)) * xl.r;
    const int t0 = (tile - __ldg(tcum + b)) * kFinalTile;
    const int nrows = min(kFinalTile, seg_rows - t0);
    const long long base = seg_base(xl, plan.cf, b) + t0 - (k - 1);
    float* swf = reinterpret_cast<float*>(sw);
    for (int i = threadIdx.x; i < KP * C; i += blockDim.x) {
        const int c = i / KP, j = i - c * KP;
        swf[i] = j < k ? __ldg(w + (size_t)j * C + c) : 0.f;
    }
    for (int i = threadIdx.x; i < C / 2; i += blockDim.x)
        sa[i] = make_float4(__ldg(alpha + 2 * i), __ldg(alpha + 2 * i + 1), __ldg(inv_alpha + 2 * i),
                            __ldg(inv_alpha + 2 * i + 1));
    __syncthreads();
    const int rows = nrows + k - 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2 part[KP / 2];
    // warp w takes rows 32 w .. 32 w + 31: the tile's k - 1 history rows and
    // its first rows, ..., the last warp the tile's last k - 1 rows (all at once,
    // not a second pass of one warp)
    for (int r0 = 32 * warp; r0 < rows; r0 += 32 * kFinalWarps) {
        final_rows<KP>(x, base, C, rows, r0, sw, sa, stg, lane, part);
        const int r = r0 + lane;
        if (r < rows) {
#pragma unroll
            for (int j = 0; j < KP; j++)
                if (j < k) sp[r * k + j] = (j & 1) ? part[j >> 1].y : part[j >> 1].x;
        }
    }
    __syncthreads();
    const int m = threadIdx.x;
    // the first skip[b] frames' samples (recompute mode's left context) are
    // computed but not written; the rest land from the start of the row
    const long long drop = plan.skip ? (long long)__ldg(plan.skip + b) * spf : 0;
    if (m < nrows && t0 + m >= drop) {
        float acc = __ldg(bias);
        for (int j = 0; j < k; j++) acc += sp[(m + j) * k + j];
        const long long idx = (long long)__ldg(bidx + b) * audio_ld + t0 + m - drop;
        audio[idx] = tanhf(acc);
        if (pre_tanh) pre_tanh[idx] = acc;
    }
}

size_t final_conv_smem_bytes(int C, int k)
{
    const int KP = k <= 8 ? 8 : 16;
    return sizeof(float) * ((size_t)KP * C + 2 * (size_t)C + (size_t)kFinalWarps * 32 * 9 * 4 +
                            (size_t)(kFinalTile + k - 1) * k);
}

cudaError_t launch_final_conv(const float* x, Layout xl, int C, const float* w, const float* bias,
                              const float* alpha, const float* inv_alpha, int k, float* audio,
                              float* pre_tanh, long long audio_ld, int spf, PlanView plan, const int* tcum,
                              int n_row_tiles, cudaStream_t s)
{
    if (n_row_tiles <= 0) return cudaSuccess;
    if (k > kFinalMaxK || C % 4 != 0) return cudaErrorInvalidValue;
    const int KP = k <= 8 ? 8 : 16;
    const size_t smem = final_conv_smem_bytes(C, k);
    if (smem > (size_t)kFinalMaxSmem) return cudaErrorInvalidValue;
    if (KP == 8)
        launch_pdl(final_conv_kernel<8>, dim3(n_row_tiles), dim3(kFinalWarps * 32), smem, s, x, xl, C, w, bias, alpha,
                   inv_alpha, k, audio, pre_tanh, audio_ld, spf, plan, plan.bidx, tcum);
    else
        launch_pdl(final_conv_kernel<16>, dim3(n_row_tiles), dim3(kFinalWarps * 32), smem, s, x, xl, C, w, bias, alpha,
                   inv_alpha, k, audio, pre_tanh, audio_ld, spf, plan, plan.bidx, tcum);
    return cudaGetLastError();
}

// ------------------------------------------------------------ MRF sum --
// y = ((y + y1) + y2) * scale (y2 may be null: (y + y1) * scale), rounded at
// each step, over the chunk rows of every segment of a prefixed level: the
// multi-receptive-field average of resblocks whose last convs wrote separate
// buffers, in the same order and with the same roundings as the chained MRF
// epilogues (first, add, last) of the GEMM.
__global__ void __launch_bounds__(256) mrf_sum_kernel(float* __restrict__ y, const float* __restrict__ y1,
                                                      const float* __restrict__ y2, Layout l, int C, float scale,
                                                      PlanView plan, long long total_rows)
{
    pdl_wait();
    pdl_launch();
    const int C4 = C >> 2;
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= total_rows * C4) return;
    const long long row = i / C4;
    const int c4 = (int)(i - row * C4);
    const int b = find_seg_r(plan.cf, plan.B, row, l.r);
    const long long t = row - (long long)__ldg(plan.cf + b) * l.r;
    const long long at = (seg_base(l, plan.cf, b) + t) * C4 + c4;
    float4 v = reinterpret_cast<float4*>(y)[at];
    const float4 a = reinterpret_cast<const float4*>(y1)[at];
    v = make_float4(__fadd_rn(v.x, a.x), __fadd_rn(v.y, a.y), __fadd_rn(v.z, a.z), __fadd_rn(v.w, a.w));
    if (y2) {
        const float4 e = reinterpret_cast<const float4*>(y2)[at];
        v = make_float4(__fadd_rn(v.x, e.x), __fadd_rn(v.y, e.y), __fadd_rn(v.z, e.z), __fadd_rn(v.w, e.w));
    }
    reinterpret_cast<float4*>(y)[at] =
        make_float4(__fmul_rn(v.x, scale), __fmul_rn(v.y, scale), __fmul_rn(v.z, scale), __fmul_rn(v.w, scale));
}

cudaError_t launch_mrf_sum(float* y, const float* y1, const float* y2, Layout l, int C, float scale, PlanView plan,
                           long long total_rows, cudaStream_t s)
{
    if (total_rows <= 0) return cudaSuccess;
    if (C % 4 != 0) return cudaErrorInvalidValue;
    const long long n = total_rows * (C / 4);
    launch_pdl(mrf_sum_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, y, y1, y2, l, C, scale, plan,
               total_rows);
    return cudaGetLastError();
}

// ------------------------------------------------------ history bookkeeping --
// Fill: the H history rows in front of segment b <- the slot's carried rows.
// Commit: the slot's carried rows <- the last H rows of [history | chunk]
// (blixt/phonon "Speed" item 7: after each chunk a small kernel moves each
// stage's last rows to its front).  One block per (tensor, batch entry).
__global__ void hist_fill_kernel(const HistDesc* __restrict__ dsc, PlanView plan)
{
    pdl_wait();
    pdl_launch();
    const HistDesc h = dsc[blockIdx.x];
    const int b = blockIdx.y;
    if (h.H == 0) return;
    const long long dst_row = seg_base(h.l, plan.cf, b) - h.H;
    const float4* src = reinterpret_cast<const float4*>(h.state + (long long)__ldg(plan.slot + b) * h.H * h.C);
    float4* dst = reinterpret_cast<float4*>(h.buf + dst_row * h.C);
    const int n4 = (h.H * h.C) >> 2;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
}

__global__ void hist_commit_kernel(const HistDesc* __restrict__ dsc, PlanView plan,
                                   long long* __restrict__ frames)
{
    pdl_wait();
    pdl_launch();
    const HistDesc h = dsc[blockIdx.x];
    const int b = blockIdx.y;
    const int n = __ldg(plan.cf + b + 1) - __ldg(plan.cf + b);
    if (blockIdx.x == 0 && threadIdx.x == 0) frames[__ldg(plan.slot + b)] += n;
    if (h.H == 0) return;
    const long long src_row = seg_base(h.l, plan.cf, b) + (long long)n * h.l.r - h.H;
    const float4* src = reinterpret_cast<const float4*>(h.buf + src_row * h.C);
    float4* dst = reinterpret_cast<float4*>(h.state + (long long)__ldg(plan.slot + b) * h.H * h.C);
    const int n4 = (h.H * h.C) >> 2;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
}

__global__ void state_reset_kernel(const HistDesc* __restrict__ dsc, int nd, const int* __restrict__ slots,
                                   long long* __restrict__ frames, unsigned* __restrict__ err_words)
{
    pdl_wait();
    pdl_launch();
    const int slot = slots[blockIdx.y];
    if ((int)blockIdx.x == nd) {
        if (threadIdx.x == 0) { frames[slot] = 0; err_words[slot] = 0u; }
        return;
    }
    const HistDesc h = dsc[blockIdx.x];
    float4* dst = reinterpret_cast<float4*>(h.state + (long long)slot * h.H * h.C);
    const int n4 = (h.H * h.C) >> 2;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_hist_fill(const HistDesc* d, int nd, PlanView plan, cudaStream_t s)
{
    if (nd <= 0 || plan.B <= 0) return cudaSuccess;
    launch_pdl(hist_fill_kernel, dim3(nd, plan.B), dim3(256), 0, s, d, plan);
    return cudaGetLastError();
}

cudaError_t launch_hist_commit(const HistDesc* d, int nd, PlanView plan, const int* /*n_frames*/,
                               long long* frames, cudaStream_t s)
{
    if (nd <= 0 || plan.B <= 0) return cudaSuccess;
    launch_pdl(hist_commit_kernel, dim3(nd, plan.B), dim3(256), 0, s, d, plan, frames);
    return cudaGetLastError();
}

cudaError_t launch_state_reset(const HistDesc* d, int nd, const int* slots, int n_slots,
                               long long* frames, unsigned* err_words, cudaStream_t s)
{
    if (n_slots <= 0) return cudaSuccess;
    state_reset_kernel<<<dim3(nd + 1, n_slots), 256, 0, s>>>(d, nd, slots, frames, err_words);
    return cudaGetLastError();
}

cudaError_t configure_simt_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(swa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSwaMaxSmem);
    if (e != cudaSuccess) return e;
    e = configure_swa_mma();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(final_conv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinalMaxSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(final_conv_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinalMaxSmem);
}

}  // namespace codec
