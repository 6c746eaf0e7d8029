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
// design", section 1.3: RVQ embedding sum).  One block per frame row, one
// float4 of channels per thread: every load is a 128-bit load of a codebook
// row.  A code outside [0, V) zeroes the row and sets the slot's sticky bit.
__global__ void __launch_bounds__(128) rvq_gather_kernel(
    const float* __restrict__ cb, int Q, int V, int E, const int* __restrict__ codes, int T_max,
    PlanView plan, const int* __restrict__ bidx, float* __restrict__ e, Layout el,
    unsigned* __restrict__ err_words)
{
    pdl_wait();
    pdl_launch();
    __shared__ int sc[64];
    __shared__ int sbad;
    const int row = blockIdx.x;
    const int b = find_seg(plan.cf, plan.B, row);
    const int t = row - __ldg(plan.cf + b);
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
                              int total_rows, cudaStream_t s)
{
    if (total_rows <= 0) return cudaSuccess;
    launch_pdl(rvq_gather_kernel, dim3(total_rows), dim3(128), 0, s, cb, Q, V, E, codes, T_max, plan, plan.bidx,
               e, el, err_words);
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
    dim3 grid(n_row_tiles, (a.N + SB_N - 1) / SB_N);
    launch_pdl(gemm_simt_kernel, dim3(grid), dim3(256), 0, s, a, plan);
    return cudaGetLastError();
}

// --------------------------------------------------------------- RMSNorm --
// y = x / sqrt(mean(x^2) + eps) * g, one warp per row; the row's sum of
// squares runs lane-strided then through a fixed butterfly.
// planes set: the normalised row goes straight into a tensor-core GEMM's
// operand planes (row of layout yl) instead of y.
__global__ void rms_norm_kernel(const float* __restrict__ x, Layout xl, const float* __restrict__ g,
                                float eps, float* __restrict__ y, Layout yl, int d, PlanView plan,
                                int total_rows, void* planes, int planes_il)
{
    pdl_wait();
    pdl_launch();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= total_rows) return;
    const int b = find_seg(plan.cf, plan.B, row);
    const int t = row - __ldg(plan.cf + b);
    const float4* xr = reinterpret_cast<const float4*>(x + (seg_base(xl, plan.cf, b) + t) * d);
    const long long yrow = seg_base(yl, plan.cf, b) + t;
    float4* yr = reinterpret_cast<float4*>(y + yrow * d);
    const int d4 = d >> 2;
    float ss = 0.f;
    for (int c = lane; c < d4; c += 32) {
        const float4 v = xr[c];
        ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss); ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / (float)d + eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int c = lane; c < d4; c += 32) {
        const float4 v = xr[c], w = __ldg(g4 + c);
        const float4 o = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
        if (planes) plane_store4(planes, planes_il, yrow, d, 4 * c, o);
        else yr[c] = o;
    }
}

cudaError_t launch_rms_norm(const float* x, Layout xl, const float* g, float eps, float* y, Layout yl,
                            int d, PlanView plan, int total_rows, cudaStream_t s, void* planes, int planes_il)
{
    if (planes && (d % 32 != 0)) return cudaErrorInvalidValue;
    if (total_rows <= 0) return cudaSuccess;
    const int threads = 256, rows_per_block = threads / 32;
    launch_pdl(rms_norm_kernel, dim3((total_rows + rows_per_block - 1) / rows_per_block), dim3(threads), 0, s,
               x, xl, g, eps, y, yl, d, plan, total_rows, planes, planes_il);
    return cudaGetLastError();
}

// ---------------------------------------------- sliding-window attention --
// A block takes up to 16 consecutive queries of one stream and one head,
// stages the keys and values of every position they can see (at most
// 16 + W - 1 rows, read from the stream's ring: position p lives in ring row
// p mod R) in shared memory, and gives each warp two queries.  Query at
// absolute position p attends positions max(0, p - W + 1) .. p.  Lane i
// scores keys lo + i, lo + 32 + i, ...; max and denominator go through a
// fixed butterfly and the value sum runs over the keys in position order, so
// a query's result depends only on its position and the keys, never on the
// chunking (blixt/phonon "Speed" item 7: ring of keys and values; item 11:
// softmax with max subtraction).
constexpr int kSwaMaxW = 128;
constexpr int kSwaMaxDh = 128;
constexpr int kSwaQ = 16;           // queries per block
constexpr int kSwaWarps = 8;
constexpr int kSwaMaxSmem = 160 * 1024;

// planes set: the attention output goes straight into the out-projection's
// tensor-core operand planes (dense rows) instead of o.
__global__ void __launch_bounds__(kSwaWarps * 32) swa_kernel(
    const float* __restrict__ q, float* __restrict__ o, const float* __restrict__ kring,
    const float* __restrict__ vring, int d, int heads, int W, int R, PlanView plan,
    const int* __restrict__ qcum, void* planes, int planes_il)
{
    pdl_wait();
    pdl_launch();
    extern __shared__ float sm[];
    const int dh = d / heads;
    const int ld = dh + 1;                              // padded row: conflict-free column reads
    const int maxk = kSwaQ + W - 1;
    float* sk = sm;                                     // [maxk][dh + 1]
    float* sv = sk + maxk * ld;                         // [maxk][dh + 1]
    float* sq = sv + maxk * ld;                         // [kSwaWarps][dh]
    float* sp = sq + kSwaWarps * dh;                    // [kSwaWarps][W]
    const int h = blockIdx.y;
    const int blk = blockIdx.x;
    const int b = find_seg(qcum, plan.B, blk);
    const int n = __ldg(plan.cf + b + 1) - __ldg(plan.cf + b);
    const int tq0 = (blk - __ldg(qcum + b)) * kSwaQ;
    const int nq = min(kSwaQ, n - tq0);
    const long long p0 = __ldg(plan.pos0 + b) + tq0;   // position of the block's first query
    const long long kstart = p0 - W + 1 > 0 ? p0 - W + 1 : 0;
    const int nk = (int)(p0 + nq - kstart);             // keys the block's queries can see
    const long long slot_base = (long long)__ldg(plan.slot + b) * R;
    for (int i = threadIdx.x; i < nk * dh; i += blockDim.x) {
        const int r = i / dh, c = i - r * dh;
        const long long row = (slot_base + ((kstart + r) & (R - 1))) * d + h * dh + c;
        sk[r * ld + c] = __ldg(kring + row);
        sv[r * ld + c] = __ldg(vring + row);
    }
    __syncthreads();
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale = 1.0f / sqrtf((float)dh);
    const long long row0 = (long long)__ldg(plan.cf + b) + tq0;
    for (int qi = wib; qi < nq; qi += kSwaWarps) {
        const long long pos = p0 + qi;
        const long long lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
        const int nkq = (int)(pos - lo + 1);
        const int off = (int)(lo - kstart);             // smem row of key lo
        const float* qr = q + (row0 + qi) * d + h * dh;
        for (int c = lane; c < dh; c += 32) sq[wib * dh + c] = qr[c];
        __syncwarp();
        float sc[kSwaMaxW / 32];
        float m = -INFINITY;
#pragma unroll
        for (int u = 0; u < kSwaMaxW / 32; u++) {
            const int i = lane + 32 * u;
            sc[u] = -INFINITY;
            if (i < nkq) {
                const float* kr = sk + (off + i) * ld;
                float dot = 0.f;
                for (int c = 0; c < dh; c++) dot = fmaf(sq[wib * dh + c], kr[c], dot);
                sc[u] = dot * scale;
                m = fmaxf(m, sc[u]);
            }
        }
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
        float z = 0.f;
#pragma unroll
        for (int u = 0; u < kSwaMaxW / 32; u++) {
            const int i = lane + 32 * u;
            if (i < nkq) {
                const float pe = expf(sc[u] - m);
                sp[wib * W + i] = pe;
                z += pe;
            }
        }
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) z += __shfl_xor_sync(0xffffffffu, z, sh);
        __syncwarp();
        const float inv_z = 1.0f / z;
        for (int c = lane; c < dh; c += 32) {
            float acc = 0.f;
            for (int i = 0; i < nkq; i++) acc = fmaf(sp[wib * W + i], sv[(off + i) * ld + c], acc);
            if (planes) plane_store1(planes, planes_il, row0 + qi, d, h * dh + c, acc * inv_z);
            else o[(row0 + qi) * d + h * dh + c] = acc * inv_z;
        }
        __syncwarp();
    }
}

cudaError_t launch_swa(const float* q, float* o, const float* kring, const float* vring, int d,
                       int heads, int window, int ring_R, PlanView plan, const int* qcum, int n_qblocks,
                       cudaStream_t s, void* planes, int planes_il)
{
    if (n_qblocks <= 0) return cudaSuccess;
    if (planes && (d % 32 != 0)) return cudaErrorInvalidValue;
    const int dh = d / heads;
    if (dh > kSwaMaxDh || window > kSwaMaxW) return cudaErrorInvalidValue;
    const int maxk = kSwaQ + window - 1;
    const size_t smem = sizeof(float) * (2 * (size_t)maxk * (dh + 1) + (size_t)kSwaWarps * dh + (size_t)kSwaWarps * window);
    if (smem > (size_t)kSwaMaxSmem) return cudaErrorInvalidValue;
    launch_pdl(swa_kernel, dim3(n_qblocks, heads), dim3(kSwaWarps * 32), smem, s, q, o, kring, vring, d, heads,
               window, ring_R, plan, qcum, planes, planes_il);
    return cudaGetLastError();
}

// ------------------------------------------------ final Snake-conv-tanh --
// y[t] = tanh(b + sum_j p_j[t - (k-1) + j]), p_j[r] = sum_c w[j][c] snake(x[r][c]),
// C -> 1.  One thread per input row computes that row's k partial dot
// products (its channels read once, Snake applied once per element) into
// shared memory; then one thread per output row sums its k partials in tap
// order.  A block covers 128 output rows and the k-1 history rows before
// them.  Bandwidth-bound: one input row in, one sample out (blixt/phonon
// "Open work": a direct kernel for the last convolution with 1 output
// channel).
constexpr int kFinalTile = 128;
constexpr int kFinalMaxK = 16;
constexpr int kFinalMaxSmem = 160 * 1024;

// KP: taps padded to 8 or 16.  The weights sit in shared memory as [C][KP]
// (zero beyond k) and are read as float4s, the Snake parameters as float2s,
// so a channel costs its Snake, KP/4 + 1 shared loads and KP FMAs.
template <int KP>
__global__ void __launch_bounds__(kFinalTile) final_conv_kernel(
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
    float2* sa = reinterpret_cast<float2*>(sm4 + (size_t)C * (KP / 4)); // [C] (alpha, 1/alpha)
    float* sp = reinterpret_cast<float*>(sa + C);                       // [kFinalTile + k - 1][k] partials
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
    for (int i = threadIdx.x; i < C; i += blockDim.x) sa[i] = make_float2(__ldg(alpha + i), __ldg(inv_alpha + i));
    __syncthreads();
    const int rows = nrows + k - 1;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        float part[KP];
#pragma unroll
        for (int j = 0; j < KP; j++) part[j] = 0.f;
        const float4* xr = reinterpret_cast<const float4*>(x + (base + r) * C);
        for (int c4 = 0; c4 < (C >> 2); c4++) {
            const float4 v = __ldg(xr + c4);
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int c = 4 * c4 + u;
                const float2 al = sa[c];
                const float sn = snake_f(e[u], al.x, al.y);
#pragma unroll
                for (int q = 0; q < KP / 4; q++) {
                    const float4 wq = sw[c * (KP / 4) + q];
                    part[4 * q] = fmaf(wq.x, sn, part[4 * q]);
                    part[4 * q + 1] = fmaf(wq.y, sn, part[4 * q + 1]);
                    part[4 * q + 2] = fmaf(wq.z, sn, part[4 * q + 2]);
                    part[4 * q + 3] = fmaf(wq.w, sn, part[4 * q + 3]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < KP; j++)
            if (j < k) sp[r * k + j] = part[j];
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

cudaError_t launch_final_conv(const float* x, Layout xl, int C, const float* w, const float* bias,
                              const float* alpha, const float* inv_alpha, int k, float* audio,
                              float* pre_tanh, long long audio_ld, int spf, PlanView plan, const int* tcum,
                              int n_row_tiles, cudaStream_t s)
{
    if (n_row_tiles <= 0) return cudaSuccess;
    if (k > kFinalMaxK) return cudaErrorInvalidValue;
    const int KP = k <= 8 ? 8 : 16;
    const size_t smem = sizeof(float) * ((size_t)KP * C + 2 * (size_t)C + (size_t)(kFinalTile + k - 1) * k);
    if (smem > (size_t)kFinalMaxSmem) return cudaErrorInvalidValue;
    if (KP == 8)
        launch_pdl(final_conv_kernel<8>, dim3(n_row_tiles), dim3(kFinalTile), smem, s, x, xl, C, w, bias, alpha,
                   inv_alpha, k, audio, pre_tanh, audio_ld, spf, plan, plan.bidx, tcum);
    else
        launch_pdl(final_conv_kernel<16>, dim3(n_row_tiles), dim3(kFinalTile), smem, s, x, xl, C, w, bias, alpha,
                   inv_alpha, k, audio, pre_tanh, audio_ld, spf, plan, plan.bidx, tcum);
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
    e = cudaFuncSetAttribute(final_conv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinalMaxSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(final_conv_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinalMaxSmem);
}

}  // namespace codec
