// FFT of one frame in shared memory by a team of threads, used by the iSTFT
// head and the analysis STFT.  A block may hold several teams (frames); every
// thread of the block calls it with the same n (the stages end in block-wide
// barriers), and it ends with every team's result complete and visible.
#pragma once

#include <cuda_runtime.h>

namespace codec {

__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// Stockham FFT of n = 2^k points: one radix-2 stage first when k is odd, then
// radix-4 stages.  A stage that has transforms of length Ls maps thread j =
// g Ls + k's inputs in[j + q n / r] (q < r), each times the twiddle
// exp(sign 2 pi i q k / (r Ls)), through an r-point DFT to out[r g Ls + k +
// p Ls], p < r.  tw[j] = exp(+2 pi i j / n); forward conjugates it (sign -).
// a and b are the team's two n-point buffers; tid / nthr: the thread's index
// in its team and the team's size.  Returns the buffer holding the transform
// (unnormalised).
__device__ __forceinline__ float2* fft_stockham(float2* a, float2* b, const float2* tw, int n, bool forward,
                                                int tid, int nthr)
{
    float2* in = a;
    float2* o = b;
    int log2n = 0;
    while ((1 << log2n) < n) log2n++;
    int Ls = 1;
    if (log2n & 1) {
        const int half = n / 2;
        for (int j = tid; j < half; j += nthr) {
            const int k = j & (Ls - 1);
            float2 w = tw[k * (half / Ls)];
            if (forward) w.y = -w.y;
            const float2 u = in[j];
            const float2 v = cmul(in[j + half], w);
            const int d = 2 * (j - k) + k;
            o[d] = make_float2(u.x + v.x, u.y + v.y);
            o[d + Ls] = make_float2(u.x - v.x, u.y - v.y);
        }
        __syncthreads();
        float2* tmp = in;
        in = o;
        o = tmp;
        Ls = 2;
    }
    const int q = n / 4;
    for (; Ls < n; Ls <<= 2) {
        const int step = q / Ls;                 // n / (4 Ls)
        for (int j = tid; j < q; j += nthr) {
            const int k = j & (Ls - 1);
            float2 w1 = tw[k * step], w2 = tw[(2 * k * step) & (n - 1)], w3 = tw[(3 * k * step) & (n - 1)];
            if (forward) {
                w1.y = -w1.y;
                w2.y = -w2.y;
                w3.y = -w3.y;
            }
            const float2 x0 = in[j];
            const float2 x1 = cmul(in[j + q], w1);
            const float2 x2 = cmul(in[j + 2 * q], w2);
            const float2 x3 = cmul(in[j + 3 * q], w3);
            const float2 t0 = make_float2(x0.x + x2.x, x0.y + x2.y);
            const float2 t1 = make_float2(x0.x - x2.x, x0.y - x2.y);
            const float2 t2 = make_float2(x1.x + x3.x, x1.y + x3.y);
            const float2 dd = make_float2(x1.x - x3.x, x1.y - x3.y);
            // t3 = (x1 - x3) * (sign i): i (a + ib) = -b + ia
            const float2 t3 = forward ? make_float2(dd.y, -dd.x) : make_float2(-dd.y, dd.x);
            const int d = 4 * (j - k) + k;
            o[d] = make_float2(t0.x + t2.x, t0.y + t2.y);
            o[d + Ls] = make_float2(t1.x + t3.x, t1.y + t3.y);
            o[d + 2 * Ls] = make_float2(t0.x - t2.x, t0.y - t2.y);
            o[d + 3 * Ls] = make_float2(t1.x - t3.x, t1.y - t3.y);
        }
        __syncthreads();
        float2* tmp = in;
        in = o;
        o = tmp;
    }
    return in;
}

// Threads per frame: a power of two, one radix-4 butterfly (or, for a direct
// DFT, one output) each where possible, at most 256.
inline int fft_team_threads(int n)
{
    int t = 1;
    while (t < n / 4 && t < 256) t <<= 1;          // one radix-4 butterfly per thread
    if ((n & (n - 1)) != 0)            // direct DFT: one output (or bin) per thread
        while (t < n && t < 256) t <<= 1;
    return t;
}

}  // namespace codec
