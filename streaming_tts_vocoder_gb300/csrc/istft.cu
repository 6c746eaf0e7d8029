// Streaming iSTFT head (the last step of the iSTFT-head vocoders: Vocos,
// HiFT, iSTFTNet): log-magnitude / phase frames -> inverse real DFT -> periodic
// Hann window -> overlap-add at hop -> division by the stationary
// window-square envelope, causal, with each stream's last n_fft / hop - 1
// windowed frames carried between calls.
//
// Two kernels per call, over the call's packed frames (stream segments back
// to back, as the decoder packs them):
//   istft_frame_kernel   one block per frame: spectrum in shared memory,
//                        Hermitian completion, inverse FFT (radix-4 Stockham
//                        for power-of-two n_fft, a direct DFT otherwise),
//                        window; the windowed frame goes to a scratch row
//   istft_ola_kernel     y = 0: one thread per output sample, the n_fft / hop
//                        frames covering it (scratch rows, or carried frames
//                        for frames before the chunk), newest first, over the
//                        envelope; y = 1: the last n_fft / hop - 1 windowed
//                        frames become the carried frames
// The carried frames of a slot live in two buffers used in turn (the host
// keeps which one is current), so the same launch can read the old ones and
// write the new ones.
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

constexpr int kMaxFft = 4096;
constexpr int kPlanRing = 8;

struct IstftPlan {
    int B;              // batch entries with frames
    const int* cf;      // [B + 1] cumulative frames
    const int* slot;    // [B]
    const int* bidx;    // [B] row in the caller's spec / audio arrays
    const int* cur;     // [B] the slot's current carried-frame buffer (0 or 1)
};

// Frames of the call (global index over all segments), fpb per block, one
// team of tpf threads each.  Shared memory: the n_fft twiddles exp(+2 pi i j
// / n_fft), copied from the table made at create, then two n_fft complex
// buffers per team.  Every thread reaches every barrier; a team past the last
// frame does no work.
__global__ void istft_frame_kernel(const float* __restrict__ spec, const float2* __restrict__ twiddles,
                                   IstftPlan plan, int total, int T_max, int n_fft, int log2n, int tpf,
                                   float mag_clip, float* __restrict__ frames)
{
    extern __shared__ float2 sh[];
    float2* tw = sh;
    const int team = threadIdx.x / tpf, tid = threadIdx.x - team * tpf;
    float2* a = sh + n_fft + (size_t)team * 2 * n_fft;
    float2* b = a + n_fft;
    const int f = blockIdx.x * (blockDim.x / tpf) + team;
    const bool valid = f < total;
    for (int j = threadIdx.x; j < n_fft; j += blockDim.x) tw[j] = __ldg(twiddles + j);
    const int nb = n_fft / 2 + 1;
    if (valid) {
        const int seg = find_seg(plan.cf, plan.B, f);
        const int t = f - __ldg(plan.cf + seg);
        const float* row = spec + ((size_t)__ldg(plan.bidx + seg) * T_max + t) * (size_t)(2 * nb);
        // X[k] for k <= n_fft / 2 and its Hermitian mirror; the imaginary parts of
        // the DC and Nyquist bins do not enter the real inverse transform
        for (int k = tid; k < nb; k += tpf) {
            float mag = expf(__ldg(row + k));
            if (mag_clip > 0.f) mag = fminf(mag, mag_clip);
            float sn, cs;
            sincosf(__ldg(row + nb + k), &sn, &cs);
            float2 x = make_float2(mag * cs, mag * sn);
            if (k == 0 || 2 * k == n_fft) x.y = 0.f;
            a[k] = x;
            if (k > 0 && 2 * k < n_fft) a[n_fft - k] = make_float2(x.x, -x.y);
        }
    }
    __syncthreads();
    float2* out = a;
    if (log2n > 0) {
        out = fft_stockham(a, b, tw, n_fft, false, tid, tpf);
    } else {
        // direct inverse DFT: x[m] = sum_k X[k] exp(2 pi i k m / n)
        if (valid) {
            for (int m = tid; m < n_fft; m += tpf) {
                float re = 0.f;
                int km = 0;
                for (int k = 0; k < n_fft; k++) {
                    const float2 x = a[k], w = tw[km];
                    re = fmaf(x.x, w.x, re);
                    re = fmaf(-x.y, w.y, re);
                    km += m;
                    if (km >= n_fft) km -= n_fft;
                }
                b[m].x = re;
            }
        }
        __syncthreads();
        out = b;
    }
    if (!valid) return;
    float* dst = frames + (size_t)f * n_fft;
    const float inv_n = 1.0f / (float)n_fft;
    for (int m = tid; m < n_fft; m += tpf) {
        const float sv = sinpif((float)m / (float)n_fft);
        dst[m] = out[m].x * inv_n * (sv * sv);
    }
}

// blockIdx.y == 0: output sample u of the call (global over all segments'
// samples).  blockIdx.y == 1: element (segment, i, m) of the new carried
// frames, carried frame i = frame n - (taps - 1) + i of the chunk (n its
// frames), from the scratch rows or, for a chunk shorter than that, from the
// old carried frames; written to the slot's other buffer.
__global__ void istft_ola_kernel(const float* __restrict__ frames, float* __restrict__ state,
                                 const float* __restrict__ env, IstftPlan plan, int n_fft, int hop, int T_max,
                                 long long total_samples, long long state_per_buf, float* __restrict__ audio)
{
    const long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const int taps = n_fft / hop;
    const long long per_slot = (long long)(taps - 1) * n_fft;
    if (blockIdx.y == 0) {
        if (u >= total_samples) return;
        const int fg = (int)(u / hop);
        const int p = (int)(u - (long long)fg * hop);
        const int seg = find_seg(plan.cf, plan.B, fg);
        const int f0 = __ldg(plan.cf + seg);
        const int t = fg - f0;
        const float* carried = state + __ldg(plan.cur + seg) * state_per_buf + __ldg(plan.slot + seg) * per_slot;
        float y = 0.f;
        for (int j = 0; j < taps; j++) {
            const int tj = t - j;
            const float* fr = tj >= 0 ? frames + (size_t)(f0 + tj) * n_fft : carried + (size_t)(tj + taps - 1) * n_fft;
            y += fr[p + j * hop];
        }
        audio[((size_t)__ldg(plan.bidx + seg) * T_max + t) * hop + p] = __fdiv_rn(y, __ldg(env + p));
    } else {
        if (u >= (long long)plan.B * per_slot) return;
        const int seg = (int)(u / per_slot);
        const long long e = u - (long long)seg * per_slot;
        const int i = (int)(e / n_fft), m = (int)(e - (long long)i * n_fft);
        const int f0 = __ldg(plan.cf + seg);
        const int n = __ldg(plan.cf + seg + 1) - f0;
        const int c = __ldg(plan.cur + seg);
        const long long slot_off = __ldg(plan.slot + seg) * per_slot;
        const int tj = n - (taps - 1) + i;
        const float v = tj >= 0 ? frames[(size_t)(f0 + tj) * n_fft + m]
                                : state[c * state_per_buf + slot_off + (long long)(tj + taps - 1) * n_fft + m];
        state[(1 - c) * state_per_buf + slot_off + e] = v;
    }
}

// Both carried-frame buffers of the listed slots (blockIdx.y: the buffer).
__global__ void istft_reset_kernel(float* __restrict__ state, const int* __restrict__ slots, int per_slot,
                                   long long state_per_buf)
{
    float* s = state + blockIdx.y * state_per_buf + (size_t)__ldg(slots + blockIdx.x) * per_slot;
    for (int m = threadIdx.x; m < per_slot; m += blockDim.x) s[m] = 0.f;
}

}  // namespace

}  // namespace codec

using namespace codec;

struct codec_istft_s {
    codec_istft_config cfg{};
    int taps = 0, nb = 0, log2n = 0, tpf = 0, fpb = 0;   // threads per frame, frames per block
    size_t smem = 0;
    float* state = nullptr;     // [2][slots][taps - 1][n_fft]: two buffers used in turn
    std::vector<int> cur;       // per slot: the buffer holding its current carried frames
    float2* twiddles = nullptr; // [n_fft] exp(+2 pi i j / n_fft)
    float* frames = nullptr;    // [max_streams * max_chunk_frames][n_fft]
    float* env = nullptr;       // [hop]
    int* slots_d = nullptr;     // reset list
    int* plan_d = nullptr;      // cf [S + 1], slot [S], bidx [S]
    int* plan_h[kPlanRing] = {};
    cudaEvent_t plan_ev[kPlanRing] = {};
    int plan_next = 0;
    int plan_ints = 0;
    std::vector<void*> allocs;
};

namespace {

void istft_free(codec_istft_s* s)
{
    for (int i = 0; i < kPlanRing; i++) {
        if (s->plan_h[i]) cudaFreeHost(s->plan_h[i]);
        if (s->plan_ev[i]) cudaEventDestroy(s->plan_ev[i]);
    }
    for (void* p : s->allocs) cudaFree(p);
    delete s;
}

template <class T>
T* istft_alloc(codec_istft_s* s, size_t n, bool& ok)
{
    void* p = nullptr;
    if (!ok || cudaMalloc(&p, std::max<size_t>(n, 1) * sizeof(T)) != cudaSuccess) {
        ok = false;
        return nullptr;
    }
    s->allocs.push_back(p);
    return static_cast<T*>(p);
}

}  // namespace

codec_status codec_istft_create(const codec_istft_config* cfg, codec_istft_t** out)
{
    if (!cfg || !out) return CODEC_ERR_NULL;
    *out = nullptr;
    const codec_istft_config& c = *cfg;
    if (c.n_fft < 4 || c.n_fft > kMaxFft || (c.n_fft & 1) || c.hop < 1 || c.n_fft % c.hop != 0 ||
        c.max_streams < 1 || c.max_chunk_frames < 1 ||
        (long long)c.max_streams * c.max_chunk_frames > (1LL << 24))
        return CODEC_ERR_CONFIG;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major < 10)
        return CODEC_ERR_NO_DEVICE;
    codec_istft_s* s = new codec_istft_s();
    s->cfg = c;
    s->taps = c.n_fft / c.hop;
    s->nb = c.n_fft / 2 + 1;
    s->log2n = 0;
    if ((c.n_fft & (c.n_fft - 1)) == 0)
        while ((1 << s->log2n) < c.n_fft) s->log2n++;
    s->tpf = fft_team_threads(c.n_fft);
    s->fpb = std::max(1, 256 / s->tpf);
    s->smem = sizeof(float2) * (1 + 2 * (size_t)s->fpb) * (size_t)c.n_fft;
    if (cudaFuncSetAttribute(istft_frame_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s->smem) !=
        cudaSuccess) {
        istft_free(s);
        return CODEC_ERR_CUDA;
    }
    bool ok = true;
    const size_t S = (size_t)c.max_streams;
    s->state = istft_alloc<float>(s, 2 * S * (s->taps - 1) * c.n_fft, ok);
    s->twiddles = istft_alloc<float2>(s, c.n_fft, ok);
    s->cur.assign(S, 0);
    s->frames = istft_alloc<float>(s, S * c.max_chunk_frames * c.n_fft, ok);
    s->env = istft_alloc<float>(s, c.hop, ok);
    s->slots_d = istft_alloc<int>(s, S, ok);
    s->plan_ints = (int)(4 * S + 1);
    s->plan_d = istft_alloc<int>(s, s->plan_ints, ok);
    for (int i = 0; i < kPlanRing && ok; i++) {
        if (cudaMallocHost(&s->plan_h[i], sizeof(int) * s->plan_ints) != cudaSuccess) ok = false;
        else if (cudaEventCreateWithFlags(&s->plan_ev[i], cudaEventDisableTiming) != cudaSuccess) ok = false;
    }
    if (!ok) {
        istft_free(s);
        return CODEC_ERR_OOM;
    }
    // envelope E[p] = sum_j w[p + j hop]^2 in double, rounded once
    std::vector<float> env(c.hop);
    for (int p = 0; p < c.hop; p++) {
        double e = 0.0;
        for (int j = 0; j < s->taps; j++) {
            const double w = std::sin(M_PI * (double)(p + j * c.hop) / (double)c.n_fft);
            e += w * w * w * w;
        }
        env[p] = (float)e;
    }
    std::vector<float2> tw(c.n_fft);
    for (int j = 0; j < c.n_fft; j++) {
        const double a = 2.0 * M_PI * (double)j / (double)c.n_fft;
        tw[j] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
    if (cudaMemcpy(s->env, env.data(), sizeof(float) * c.hop, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(s->twiddles, tw.data(), sizeof(float2) * c.n_fft, cudaMemcpyHostToDevice) != cudaSuccess ||
        (s->taps > 1 && cudaMemset(s->state, 0, sizeof(float) * 2 * S * (s->taps - 1) * c.n_fft) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        istft_free(s);
        return CODEC_ERR_CUDA;
    }
    *out = s;
    return CODEC_OK;
}

void codec_istft_destroy(codec_istft_t* s)
{
    if (!s) return;
    cudaDeviceSynchronize();
    istft_free(s);
}

codec_status codec_istft_reset(codec_istft_t* s, const int32_t* ids, int32_t n, void* stream)
{
    if (!s) return CODEC_ERR_NULL;
    const int S = s->cfg.max_streams;
    if (ids && (n < 0 || n > S)) return CODEC_ERR_ARG;
    std::vector<int> list;
    if (ids) {
        std::vector<char> seen(S, 0);
        for (int i = 0; i < n; i++) {
            if (ids[i] < 0 || ids[i] >= S || seen[ids[i]]) return CODEC_ERR_ARG;
            seen[ids[i]] = 1;
            list.push_back(ids[i]);
        }
    } else {
        for (int i = 0; i < S; i++) list.push_back(i);
    }
    const int per_slot = (s->taps - 1) * s->cfg.n_fft;
    if (list.empty() || per_slot == 0) return CODEC_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the id list rides in a plan staging buffer (page-locked, ring-guarded)
    const int i = s->plan_next;
    s->plan_next = (i + 1) % kPlanRing;
    if (cudaEventSynchronize(s->plan_ev[i]) != cudaSuccess) return CODEC_ERR_CUDA;
    std::memcpy(s->plan_h[i], list.data(), sizeof(int) * list.size());
    if (cudaMemcpyAsync(s->slots_d, s->plan_h[i], sizeof(int) * list.size(), cudaMemcpyHostToDevice, cs) !=
            cudaSuccess ||
        cudaEventRecord(s->plan_ev[i], cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    istft_reset_kernel<<<dim3((unsigned)list.size(), 2), 256, 0, cs>>>(s->state, s->slots_d, per_slot,
                                                                        (long long)S * per_slot);
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}

codec_status codec_istft_decode(codec_istft_t* s, const float* spec, const int32_t* n_frames,
                                const int32_t* ids, int32_t B, int32_t T_max, float* audio, void* stream)
{
    if (!s || !spec || !n_frames || !audio) return CODEC_ERR_NULL;
    const codec_istft_config& c = s->cfg;
    const int S = c.max_streams;
    if (B < 1 || T_max < 1) return CODEC_ERR_ARG;
    if (B > S || T_max > c.max_chunk_frames) return CODEC_ERR_CAPACITY;
    std::vector<char> seen(S, 0);
    for (int b = 0; b < B; b++) {
        const int id = ids ? ids[b] : b;
        if (id < 0 || id >= S || seen[id]) return CODEC_ERR_ARG;
        seen[id] = 1;
        if (n_frames[b] < 0 || n_frames[b] > T_max) return CODEC_ERR_ARG;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int i = s->plan_next;
    s->plan_next = (i + 1) % kPlanRing;
    if (cudaEventSynchronize(s->plan_ev[i]) != cudaSuccess) return CODEC_ERR_CUDA;
    int* cf = s->plan_h[i];
    int* slot = cf + S + 1;
    int* bidx = slot + S;
    int* cur = bidx + S;
    int Bc = 0;
    cf[0] = 0;
    for (int b = 0; b < B; b++) {
        if (n_frames[b] == 0) continue;
        slot[Bc] = ids ? ids[b] : b;
        bidx[Bc] = b;
        cur[Bc] = s->cur[slot[Bc]];
        cf[Bc + 1] = cf[Bc] + n_frames[b];
        Bc++;
    }
    if (Bc == 0) return CODEC_OK;
    const int total = cf[Bc];
    if (cudaMemcpyAsync(s->plan_d, cf, sizeof(int) * s->plan_ints, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaEventRecord(s->plan_ev[i], cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    const IstftPlan plan{Bc, s->plan_d, s->plan_d + S + 1, s->plan_d + 2 * S + 1, s->plan_d + 3 * S + 1};
    istft_frame_kernel<<<(total + s->fpb - 1) / s->fpb, s->fpb * s->tpf, s->smem, cs>>>(
        spec, s->twiddles, plan, total, T_max, c.n_fft, s->log2n, s->tpf, c.mag_clip, s->frames);
    const long long samples = (long long)total * c.hop;
    const long long per_slot = (long long)(s->taps - 1) * c.n_fft;
    const long long work = std::max(samples, (long long)Bc * per_slot);
    istft_ola_kernel<<<dim3((unsigned)((work + 255) / 256), s->taps > 1 ? 2 : 1), 256, 0, cs>>>(
        s->frames, s->state, s->env, plan, c.n_fft, c.hop, T_max, samples, (long long)S * per_slot, audio);
    // the new carried frames are in the other buffer from here on
    for (int b = 0; b < Bc; b++) s->cur[slot[b]] ^= 1;
    return cudaGetLastError() == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}
