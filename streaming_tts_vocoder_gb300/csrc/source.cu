// The excitation path of the iSTFT-head vocoders: a harmonic sine source
// driven by per-frame F0 with an exact integer phase carried per stream, and
// a causal analysis STFT with the last n_fft - hop input samples carried per
// stream.  Both take ragged multi-stream batches packed back to back, as the
// decoder and the iSTFT head do.
//
// Sine source, two launches per call:
//   sine_scan_kernel  one warp per batch entry: each frame's phase at its
//                     start and its increment (a warp prefix sum over the
//                     frames), and the slot's phase after the chunk
//   sine_out_kernel   one thread per output sample: phase = start + (r + 1)
//                     increment (unsigned 32-bit wrap = modulo one cycle), the
//                     harmonics' sines
// Analysis STFT, two launches per call:
//   stft_frame_kernel   one block per frame: n_fft input samples (the carried
//                       history for those before the chunk), Hann window,
//                       forward FFT in shared memory (radix-4 Stockham, or a
//                       direct DFT for other sizes), n_fft / 2 + 1 bins out
//   stft_commit_kernel  the new history, into the slot's other buffer
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "codec.h"
#include "common.cuh"
#include "fft_smem.cuh"

namespace codec {

namespace {

constexpr int kSrcMaxFft = 4096;
constexpr int kSrcPlanRing = 8;
constexpr int kMaxHarmonics = 16;

struct SrcPlan {
    int B;              // batch entries with frames
    const int* cf;      // [B + 1] cumulative frames
    const int* slot;    // [B]
    const int* bidx;    // [B] row in the caller's arrays
    const int* cur;     // [B] current history buffer (analysis STFT)
};

// One warp per batch entry: the frames' increments D, 32 frames at a time,
// and an inclusive warp prefix sum of upp D (unsigned, so modulo one cycle,
// and exact: the order of the additions cannot change a bit) give each
// frame's phase at its start; lane 0 stores the slot's phase after the chunk
// (every lane read the old one first).
__global__ void sine_scan_kernel(const float* __restrict__ f0, SrcPlan plan, int T_max, double scale,
                                 double f0_max, int upp, unsigned* __restrict__ phase,
                                 unsigned* __restrict__ pstart, unsigned* __restrict__ dinc)
{
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (b >= plan.B) return;                    // whole warps
    const int c0 = __ldg(plan.cf + b), n = __ldg(plan.cf + b + 1) - c0;
    const float* row = f0 + (size_t)__ldg(plan.bidx + b) * T_max;
    const int sl = __ldg(plan.slot + b);
    unsigned P = phase[sl];
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        unsigned D = 0u;
        if (i < n) {
            const double f = fmin(fmax((double)__ldg(row + i), 0.0), f0_max);
            D = (unsigned)__double2ull_rn(__dmul_rn(f, scale));
        }
        const unsigned own = (unsigned)upp * D;
        unsigned incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (i < n) {
            pstart[c0 + i] = P + (incl - own);
            dinc[c0 + i] = D;
        }
        P += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) phase[sl] = P;
}

__global__ void sine_out_kernel(const float* __restrict__ f0, SrcPlan plan, int T_max, int upp, int H,
                                float amplitude, float threshold, const unsigned* __restrict__ pstart,
                                const unsigned* __restrict__ dinc, long long total_samples, float* __restrict__ out)
{
    const long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (u >= total_samples) return;
    const int fg = (int)(u / upp);
    const int r = (int)(u - (long long)fg * upp);
    const int seg = find_seg(plan.cf, plan.B, fg);
    const int t = fg - __ldg(plan.cf + seg);
    const int bi = __ldg(plan.bidx + seg);
    const bool voiced = __ldg(f0 + (size_t)bi * T_max + t) > threshold;
    const unsigned P = __ldg(pstart + fg) + (unsigned)(r + 1) * __ldg(dinc + fg);
    float* o = out + ((size_t)bi * T_max * upp + (size_t)t * upp + r) * H;
    for (int h = 1; h <= H; h++) {
        // the phase h P mod 2^32 as a signed fraction of half a cycle: sin(pi x)
        const float x = (float)(int)(P * (unsigned)h) * 4.656612873077392578125e-10f;   // 2^-31
        o[h - 1] = voiced ? amplitude * sinpif(x) : 0.f;
    }
}

// Frames of the call, fpb per block, one team of tpf threads each.  Shared
// memory: the twiddles exp(+2 pi i j / n_fft), then two n_fft complex buffers
// per team.  Every thread reaches every barrier; a team past the last frame
// does no work.
__global__ void stft_frame_kernel(const float* __restrict__ x, const float* __restrict__ hist,
                                  const float2* __restrict__ twiddles, SrcPlan plan, int total, int T_max,
                                  int n_fft, int hop, int log2n, int tpf, long long hist_per_buf,
                                  float* __restrict__ spec)
{
    extern __shared__ float2 sh[];
    float2* tw = sh;
    const int team = threadIdx.x / tpf, tid = threadIdx.x - team * tpf;
    float2* a = sh + n_fft + (size_t)team * 2 * n_fft;
    float2* b = a + n_fft;
    const int f = blockIdx.x * (blockDim.x / tpf) + team;
    const bool valid = f < total;
    for (int j = threadIdx.x; j < n_fft; j += blockDim.x) tw[j] = __ldg(twiddles + j);
    const int L = n_fft - hop;
    int seg = 0, t = 0, bi = 0;
    if (valid) {
        seg = find_seg(plan.cf, plan.B, f);
        t = f - __ldg(plan.cf + seg);
        bi = __ldg(plan.bidx + seg);
        const float* xr = x + (size_t)bi * T_max * hop;
        const float* hr = hist + __ldg(plan.cur + seg) * hist_per_buf + (size_t)__ldg(plan.slot + seg) * L;
        for (int m = tid; m < n_fft; m += tpf) {
            const int j = t * hop + m;              // position in [history | chunk]
            const float v = j < L ? __ldg(hr + j) : __ldg(xr + (j - L));
            const float sv = sinpif((float)m / (float)n_fft);
            a[m] = make_float2(v * (sv * sv), 0.f);
        }
    }
    __syncthreads();
    const int nb = n_fft / 2 + 1;
    const float2* X;
    if (log2n > 0) {
        X = fft_stockham(a, b, tw, n_fft, true, tid, tpf);
    } else {
        // direct DFT of the bins kept: X[k] = sum_m a[m] exp(-2 pi i k m / n)
        if (valid) {
            for (int k = tid; k < nb; k += tpf) {
                float re = 0.f, im = 0.f;
                int km = 0;
                for (int m = 0; m < n_fft; m++) {
                    const float v = a[m].x;
                    const float2 w = tw[km];
                    re = fmaf(v, w.x, re);
                    im = fmaf(-v, w.y, im);
                    km += k;
                    if (km >= n_fft) km -= n_fft;
                }
                b[k] = make_float2(re, im);
            }
        }
        __syncthreads();
        X = b;
    }
    if (!valid) return;
    float* dst = spec + ((size_t)bi * T_max + t) * (size_t)(2 * nb);
    for (int k = tid; k < nb; k += tpf) {
        dst[k] = X[k].x;
        dst[nb + k] = X[k].y;
    }
}

// Element (segment, j) of the new history: sample n hop + j of [old history |
// chunk] (n the entry's hops), into the slot's other buffer.
__global__ void stft_commit_kernel(const float* __restrict__ x, float* __restrict__ hist, SrcPlan plan, int T_max,
                                   int n_fft, int hop, long long hist_per_buf)
{
    const int L = n_fft - hop;
    const long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (u >= (long long)plan.B * L) return;
    const int seg = (int)(u / L);
    const int j = (int)(u - (long long)seg * L);
    const int n = __ldg(plan.cf + seg + 1) - __ldg(plan.cf + seg);
    const int c = __ldg(plan.cur + seg);
    const size_t slot_off = (size_t)__ldg(plan.slot + seg) * L;
    const int src = n * hop + j;
    const float v = src < L ? hist[c * hist_per_buf + slot_off + src]
                            : x[(size_t)__ldg(plan.bidx + seg) * T_max * hop + (src - L)];
    hist[(1 - c) * hist_per_buf + slot_off + j] = v;
}

__global__ void src_zero_kernel(float* __restrict__ buf, const int* __restrict__ slots, int per_slot,
                                long long per_buf, int n_bufs)
{
    for (int k = 0; k < n_bufs; k++) {
        float* s = buf + k * per_buf + (size_t)__ldg(slots + blockIdx.x) * per_slot;
        for (int m = threadIdx.x; m < per_slot; m += blockDim.x) s[m] = 0.f;
    }
}

__global__ void src_zero_u32_kernel(unsigned* __restrict__ v, const int* __restrict__ slots, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) v[__ldg(slots + i)] = 0u;
}

// Per-call plan (cumulative frames, slots, caller rows, current buffers)
// staged through a ring of page-locked buffers and uploaded on the call's
// stream.
struct SrcPlanRing {
    int S = 0, ints = 0, next = 0;
    int* dev = nullptr;
    int* host[kSrcPlanRing] = {};
    cudaEvent_t ev[kSrcPlanRing] = {};

    bool init(int slots, std::vector<void*>& allocs)
    {
        S = slots;
        ints = 4 * S + 1;
        if (cudaMalloc(&dev, sizeof(int) * ints) != cudaSuccess) return false;
        allocs.push_back(dev);
        for (int i = 0; i < kSrcPlanRing; i++) {
            if (cudaMallocHost(&host[i], sizeof(int) * ints) != cudaSuccess) return false;
            if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) return false;
        }
        return true;
    }
    void release()
    {
        for (int i = 0; i < kSrcPlanRing; i++) {
            if (host[i]) cudaFreeHost(host[i]);
            if (ev[i]) cudaEventDestroy(ev[i]);
        }
    }
    // Validates the batch and enqueues its plan; *Bc = 0 when no entry has frames.
    codec_status build(const int32_t* n_frames, const int32_t* ids, int32_t B, int32_t T_max, int max_chunk,
                       const std::vector<int>* cur, cudaStream_t cs, SrcPlan* plan, int* Bc, int* total,
                       std::vector<int>* slots_out)
    {
        if (B < 1 || T_max < 1) return CODEC_ERR_ARG;
        if (B > S || T_max > max_chunk) return CODEC_ERR_CAPACITY;
        std::vector<char> seen(S, 0);
        for (int b = 0; b < B; b++) {
            const int id = ids ? ids[b] : b;
            if (id < 0 || id >= S || seen[id]) return CODEC_ERR_ARG;
            seen[id] = 1;
            if (n_frames[b] < 0 || n_frames[b] > T_max) return CODEC_ERR_ARG;
        }
        const int i = next;
        next = (i + 1) % kSrcPlanRing;
        if (cudaEventSynchronize(ev[i]) != cudaSuccess) return CODEC_ERR_CUDA;
        int* cf = host[i];
        int* slot = cf + S + 1;
        int* bidx = slot + S;
        int* cb = bidx + S;
        int n = 0;
        cf[0] = 0;
        slots_out->clear();
        for (int b = 0; b < B; b++) {
            if (n_frames[b] == 0) continue;
            slot[n] = ids ? ids[b] : b;
            bidx[n] = b;
            cb[n] = cur ? (*cur)[slot[n]] : 0;
            cf[n + 1] = cf[n] + n_frames[b];
            slots_out->push_back(slot[n]);
            n++;
        }
        *Bc = n;
        *total = cf[n];
        if (n == 0) return CODEC_OK;
        if (cudaMemcpyAsync(dev, cf, sizeof(int) * ints, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
            cudaEventRecord(ev[i], cs) != cudaSuccess)
            return CODEC_ERR_CUDA;
        *plan = SrcPlan{n, dev, dev + S + 1, dev + 2 * S + 1, dev + 3 * S + 1};
        return CODEC_OK;
    }
    // Uploads a list of slot ids (for a reset) into dev; returns false on a CUDA error.
    bool upload_ids(const std::vector<int>& list, cudaStream_t cs)
    {
        const int i = next;
        next = (i + 1) % kSrcPlanRing;
        if (cudaEventSynchronize(ev[i]) != cudaSuccess) return false;
        std::memcpy(host[i], list.data(), sizeof(int) * list.size());
        return cudaMemcpyAsync(dev, host[i], sizeof(int) * list.size(), cudaMemcpyHostToDevice, cs) == cudaSuccess &&
               cudaEventRecord(ev[i], cs) == cudaSuccess;
    }
};

codec_status id_list(const int32_t* ids, int32_t n, int S, std::vector<int>* list)
{
    list->clear();
    if (!ids) {
        for (int i = 0; i < S; i++) list->push_back(i);
        return CODEC_OK;
    }
    if (n < 0 || n > S) return CODEC_ERR_ARG;
    std::vector<char> seen(S, 0);
    for (int i = 0; i < n; i++) {
        if (ids[i] < 0 || ids[i] >= S || seen[ids[i]]) return CODEC_ERR_ARG;
        seen[ids[i]] = 1;
        list->push_back(ids[i]);
    }
    return CODEC_OK;
}

bool sm100_or_newer()
{
    int dev = 0, major = 0;
    return cudaGetDevice(&dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess && major >= 10;
}

}  // namespace

}  // namespace codec

using namespace codec;

struct codec_sine_s {
    codec_sine_config cfg{};
    unsigned* phase = nullptr;     // [slots]
    unsigned* pstart = nullptr;    // [max_streams * max_chunk_frames]
    unsigned* dinc = nullptr;
    SrcPlanRing ring;
    std::vector<void*> allocs;
};

struct codec_stft_s {
    codec_stft_config cfg{};
    int log2n = 0, tpf = 0, fpb = 0;   // threads per frame, frames per block
    size_t smem = 0;
    float* hist = nullptr;         // [2][slots][n_fft - hop]
    float2* twiddles = nullptr;
    std::vector<int> cur;
    SrcPlanRing ring;
    std::vector<void*> allocs;
};

namespace {

template <class T>
void src_free(T* s)
{
    s->ring.release();
    for (void* p : s->allocs) cudaFree(p);
    delete s;
}

template <class T, class U>
U* src_alloc(T* s, size_t n, bool& ok)
{
    void* p = nullptr;
    if (!ok || cudaMalloc(&p, std::max<size_t>(n, 1) * sizeof(U)) != cudaSuccess) {
        ok = false;
        return nullptr;
    }
    s->allocs.push_back(p);
    return static_cast<U*>(p);
}

}  // namespace

codec_status codec_sine_create(const codec_sine_config* cfg, codec_sine_t** out)
{
    if (!cfg || !out) return CODEC_ERR_NULL;
    *out = nullptr;
    const codec_sine_config& c = *cfg;
    if (c.upp < 1 || c.upp > 65536 || c.harmonics < 1 || c.harmonics > kMaxHarmonics || !(c.sample_rate > 0.f) ||
        c.max_streams < 1 || c.max_chunk_frames < 1 ||
        (long long)c.max_streams * c.max_chunk_frames * c.upp > (1LL << 31))
        return CODEC_ERR_CONFIG;
    if (!sm100_or_newer()) return CODEC_ERR_NO_DEVICE;
    codec_sine_s* s = new codec_sine_s();
    s->cfg = c;
    bool ok = true;
    const size_t S = (size_t)c.max_streams;
    s->phase = src_alloc<codec_sine_s, unsigned>(s, S, ok);
    s->pstart = src_alloc<codec_sine_s, unsigned>(s, S * c.max_chunk_frames, ok);
    s->dinc = src_alloc<codec_sine_s, unsigned>(s, S * c.max_chunk_frames, ok);
    if (!ok || !s->ring.init(c.max_streams, s->allocs)) {
        src_free(s);
        return CODEC_ERR_OOM;
    }
    if (cudaMemset(s->phase, 0, sizeof(unsigned) * S) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        src_free(s);
        return CODEC_ERR_CUDA;
    }
    *out = s;
    return CODEC_OK;
}

void codec_sine_destroy(codec_sine_t* s)
{
    if (!s) return;
    cudaDeviceSynchronize();
    src_free(s);
}

codec_status codec_sine_reset(codec_sine_t* s, const int32_t* ids, int32_t n, void* stream)
{
    if (!s) return CODEC_ERR_NULL;
    std::vector<int> list;
    const codec_status st = id_list(ids, n, s->cfg.max_streams, &list);
    if (st != CODEC_OK) return st;
    if (list.empty()) return CODEC_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!s->ring.upload_ids(list, cs)) return CODEC_ERR_CUDA;
    src_zero_u32_kernel<<<((unsigned)list.size() + 255) / 256, 256, 0, cs>>>(s->phase, s->ring.dev, (int)list.size());
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}

codec_status codec_sine_decode(codec_sine_t* s, const float* f0, const int32_t* n_frames, const int32_t* ids,
                               int32_t B, int32_t T_max, float* out, void* stream)
{
    if (!s || !f0 || !n_frames || !out) return CODEC_ERR_NULL;
    const codec_sine_config& c = s->cfg;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    SrcPlan plan{};
    int Bc = 0, total = 0;
    std::vector<int> slots;
    const codec_status st = s->ring.build(n_frames, ids, B, T_max, c.max_chunk_frames, nullptr, cs, &plan, &Bc,
                                          &total, &slots);
    if (st != CODEC_OK || Bc == 0) return st;
    const double fs = (double)c.sample_rate;
    sine_scan_kernel<<<(Bc + 3) / 4, 128, 0, cs>>>(f0, plan, T_max, 4294967296.0 / fs, fs / 2, c.upp, s->phase,
                                                   s->pstart, s->dinc);
    const long long samples = (long long)total * c.upp;
    sine_out_kernel<<<(unsigned)((samples + 255) / 256), 256, 0, cs>>>(f0, plan, T_max, c.upp, c.harmonics,
                                                                     c.amplitude, c.voiced_threshold, s->pstart,
                                                                     s->dinc, samples, out);
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}

codec_status codec_stft_create(const codec_stft_config* cfg, codec_stft_t** out)
{
    if (!cfg || !out) return CODEC_ERR_NULL;
    *out = nullptr;
    const codec_stft_config& c = *cfg;
    if (c.n_fft < 4 || c.n_fft > kSrcMaxFft || (c.n_fft & 1) || c.hop < 1 || c.n_fft % c.hop != 0 ||
        c.max_streams < 1 || c.max_chunk_frames < 1 || (long long)c.max_streams * c.max_chunk_frames > (1LL << 24))
        return CODEC_ERR_CONFIG;
    if (!sm100_or_newer()) return CODEC_ERR_NO_DEVICE;
    codec_stft_s* s = new codec_stft_s();
    s->cfg = c;
    if ((c.n_fft & (c.n_fft - 1)) == 0)
        while ((1 << s->log2n) < c.n_fft) s->log2n++;
    s->tpf = fft_team_threads(c.n_fft);
    s->fpb = std::max(1, 256 / s->tpf);
    s->smem = sizeof(float2) * (1 + 2 * (size_t)s->fpb) * (size_t)c.n_fft;
    if (cudaFuncSetAttribute(stft_frame_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s->smem) !=
        cudaSuccess) {
        src_free(s);
        return CODEC_ERR_CUDA;
    }
    bool ok = true;
    const size_t S = (size_t)c.max_streams, L = (size_t)(c.n_fft - c.hop);
    s->hist = src_alloc<codec_stft_s, float>(s, 2 * S * L, ok);
    s->twiddles = src_alloc<codec_stft_s, float2>(s, c.n_fft, ok);
    s->cur.assign(S, 0);
    if (!ok || !s->ring.init(c.max_streams, s->allocs)) {
        src_free(s);
        return CODEC_ERR_OOM;
    }
    std::vector<float2> tw(c.n_fft);
    for (int j = 0; j < c.n_fft; j++) {
        const double a = 2.0 * M_PI * (double)j / (double)c.n_fft;
        tw[j] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
    if (cudaMemcpy(s->twiddles, tw.data(), sizeof(float2) * c.n_fft, cudaMemcpyHostToDevice) != cudaSuccess ||
        (L > 0 && cudaMemset(s->hist, 0, sizeof(float) * 2 * S * L) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        src_free(s);
        return CODEC_ERR_CUDA;
    }
    *out = s;
    return CODEC_OK;
}

void codec_stft_destroy(codec_stft_t* s)
{
    if (!s) return;
    cudaDeviceSynchronize();
    src_free(s);
}

codec_status codec_stft_reset(codec_stft_t* s, const int32_t* ids, int32_t n, void* stream)
{
    if (!s) return CODEC_ERR_NULL;
    std::vector<int> list;
    const codec_status st = id_list(ids, n, s->cfg.max_streams, &list);
    if (st != CODEC_OK) return st;
    const int L = s->cfg.n_fft - s->cfg.hop;
    if (list.empty() || L == 0) return CODEC_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!s->ring.upload_ids(list, cs)) return CODEC_ERR_CUDA;
    src_zero_kernel<<<(unsigned)list.size(), 256, 0, cs>>>(s->hist, s->ring.dev, L,
                                                           (long long)s->cfg.max_streams * L, 2);
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}

codec_status codec_stft_decode(codec_stft_t* s, const float* x, const int32_t* n_frames, const int32_t* ids,
                               int32_t B, int32_t T_max, float* spec, void* stream)
{
    if (!s || !x || !n_frames || !spec) return CODEC_ERR_NULL;
    const codec_stft_config& c = s->cfg;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    SrcPlan plan{};
    int Bc = 0, total = 0;
    std::vector<int> slots;
    const codec_status st = s->ring.build(n_frames, ids, B, T_max, c.max_chunk_frames, &s->cur, cs, &plan, &Bc,
                                          &total, &slots);
    if (st != CODEC_OK || Bc == 0) return st;
    const long long L = c.n_fft - c.hop;
    const long long per_buf = (long long)c.max_streams * L;
    stft_frame_kernel<<<(total + s->fpb - 1) / s->fpb, s->fpb * s->tpf, s->smem, cs>>>(
        x, s->hist, s->twiddles, plan, total, T_max, c.n_fft, c.hop, s->log2n, s->tpf, per_buf, spec);
    if (L > 0) {
        const long long work = (long long)Bc * L;
        stft_commit_kernel<<<(unsigned)((work + 255) / 256), 256, 0, cs>>>(x, s->hist, plan, T_max, c.n_fft, c.hop,
                                                                         per_buf);
        for (int sl : slots) s->cur[sl] ^= 1;
    }
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}
