// FFT of one frame in shared memory by a team of threads, used by the iSTFT
// head and the analysis STFT.  A block may hold several teams (frames); every
// thread of the block calls it with the same n (the stages end in block-wide
// barriers), and it ends with every team's result complete and visible.
#pragma once

#include <cuda_runtime.h>

namespace codec {

// Radix-2 Stockham FFT of n = 2^k points: stage with half-length Ls maps
// in[j], in[j + n/2] (j = g Ls + k) to out[2 g Ls + k], out[2 g Ls + k + Ls]
// with the twiddle exp(sign i pi k / Ls) = tw[k n / (2 Ls)] (conjugated when
// sign < 0); tw[j] = exp(+2 pi i j / n).  a and b are the two n-point
// buffers of this team; tid / nthr: the thread's index in its team and the
// team's size.  Returns the buffer holding the transform (unnormalised).
__device__ __forceinline__ float2* fft_stockham(float2* a, float2* b, const float2* tw, int n, bool forward,
                                                int tid, int nthr)
{
    float2* in = a;
    float2* o = b;
    const int half = n / 2;
    for (int Ls = 1; Ls < n; Ls <<= 1) {
        const int tstep = half / Ls;
        for (int j = tid; j < half; j += nthr) {
            const int k = j & (Ls - 1);
            const float2 u = in[j];
            const float2 v0 = in[j + half];
            float2 w = tw[k * tstep];
            if (forward) w.y = -w.y;
            const float2 v = make_float2(v0.x * w.x - v0.y * w.y, v0.x * w.y + v0.y * w.x);
            const int d = 2 * (j - k) + k;
            o[d] = make_float2(u.x + v.x, u.y + v.y);
            o[d + Ls] = make_float2(u.x - v.x, u.y - v.y);
        }
        __syncthreads();
        float2* tmp = in;
        in = o;
        o = tmp;
    }
    return in;
}

// Threads per frame (a power of two, one butterfly or one output each where
// possible) and frames per block of at most 256 threads.
inline int fft_team_threads(int n)
{
    int t = 1;
    while (t < n / 2 && t < 256) t <<= 1;
    if ((n & (n - 1)) != 0)            // direct DFT: one output (or bin) per thread
        while (t < n && t < 256) t <<= 1;
    return t;
}

}  // namespace codec
