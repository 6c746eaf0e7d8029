// Streaming Vocos-style generator in front of the iSTFT head (vox: F5-TTS's
// "Vocos -> iSTFT"), causal for streaming like the decoder:
//   mel -> causal conv k (embedding) -> LayerNorm
//       -> L x [ causal depthwise conv k -> LayerNorm -> W1 + b1 -> GELU -> W2 + b2,
//                times the layer scale, plus the block input ]
//       -> LayerNorm -> linear head to n_bins log-magnitudes and n_bins phases
//       -> the streaming iSTFT head (codec_istft_*).
// Carried per stream: the embedding conv's last k - 1 mel rows, each block's
// last k - 1 input rows, and the iSTFT head's frames, so a stream decoded in
// chunks of any sizes gives the same samples as one full decode.
//
// Launch sequence of a call (many streams' ragged chunks packed back to back,
// as in the decoder): history fill; mel rows into the prefixed buffer; the
// embedding conv (implicit GEMM); LayerNorm; per block the fused depthwise
// conv + LayerNorm kernel (a warp per row) and the two pointwise GEMMs (on the
// tcgen05 fp16x3 path where the channel counts allow: the layer scale is
// folded into W2 and b2, the residual added in the GEMM epilogue); the final
// LayerNorm; the head GEMM; the spectra scattered to the head's batch layout;
// the iSTFT head's own launches; history commit.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "codec.h"
#include "kernels.h"
#include "tc_gemm.h"

using namespace codec;

namespace {

constexpr int kPlanRing = 8;

// One contraction (conv or linear) in implicit-GEMM form: K = ntaps * Cin.
struct VContraction {
    float* w = nullptr;            // fp32 [K][N] (CUDA-core path)
    TcWeights tc;
    bool use_tc = false;
    float* bias = nullptr;
    int Cin = 0, N = 0, K = 0, ntaps = 0;
    int shift[kMaxTaps] = {};
};

struct VBlock {
    float* dw_w = nullptr;         // [k][d] (tap-major)
    float* dw_b = nullptr;
    float* ln_g = nullptr;
    float* ln_b = nullptr;
    VContraction pw1, pw2;
};

// LayerNorm over the d channels of each row (biased variance, eps inside the
// root), optionally after a causal depthwise conv of k taps over the rows of
// a prefixed buffer:  y[c] = b_dw[c] + sum_j w[j][c] x[row - (k - 1) + j][c].
// A warp per row; lane l takes the four-channel groups l, l + 32, ... (128-bit
// loads and stores), each row sum runs over a lane's channels in ascending
// order and then through a fixed butterfly, so a row's result does not depend
// on the batch it came in.  KT: the tap count when fixed at compile time
// (every load of a row's taps then in flight at once), 0 for the runtime k;
// PG: the groups per lane the registers hold (d <= 128 PG).  planes set: the
// result goes straight into the next linear's tensor-core operand planes
// (layout planes_il), split as the prep kernel would, instead of y.
template <int KT, int PG>
__global__ void __launch_bounds__(256) vocos_ln_kernel(const float* __restrict__ x, Layout xl,
                                                       const float* __restrict__ dw_w,
                                                       const float* __restrict__ dw_b, int k,
                                                       const float* __restrict__ g, const float* __restrict__ b,
                                                       float eps, int d, float* __restrict__ y, Layout yl,
                                                       PlanView plan, int total_rows, void* planes, int planes_il)
{
    pdl_wait();
    pdl_launch();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= total_rows) return;
    const int seg = find_seg(plan.cf, plan.B, row);
    const int t = row - __ldg(plan.cf + seg);
    const long long xr = seg_base(xl, plan.cf, seg) + t;
    const int d4 = d >> 2;
    auto f4 = [](const float* p, int i) { return reinterpret_cast<const float4*>(p)[i]; };
    auto fma4 = [](float4 w, float4 v, float4 a) {
        return make_float4(fmaf(w.x, v.x, a.x), fmaf(w.y, v.y, a.y), fmaf(w.z, v.z, a.z), fmaf(w.w, v.w, a.w));
    };
    float4 v[PG];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < PG; i++) {
        const int c4 = lane + 32 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c4 < d4) {
            float4 a;
            if (dw_w && KT > 0) {
                float4 xs[KT > 0 ? KT : 1], ws[KT > 0 ? KT : 1];
#pragma unroll
                for (int j = 0; j < KT; j++) {
                    xs[j] = f4(x + (xr - (KT - 1) + j) * d, c4);
                    ws[j] = __ldg(reinterpret_cast<const float4*>(dw_w + (size_t)j * d) + c4);
                }
                a = __ldg(reinterpret_cast<const float4*>(dw_b) + c4);
#pragma unroll
                for (int j = 0; j < KT; j++) a = fma4(ws[j], xs[j], a);
            } else if (dw_w) {
                a = __ldg(reinterpret_cast<const float4*>(dw_b) + c4);
                for (int j = 0; j < k; j++)
                    a = fma4(__ldg(reinterpret_cast<const float4*>(dw_w + (size_t)j * d) + c4),
                             f4(x + (xr - (k - 1) + j) * d, c4), a);
            } else {
                a = f4(x + xr * d, c4);
            }
            v[i] = a;
            s += a.x;
            s += a.y;
            s += a.z;
            s += a.w;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / (float)d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < PG; i++) {
        if (lane + 32 * i < d4) {
            const float ex = v[i].x - mean, ey = v[i].y - mean, ez = v[i].z - mean, ew = v[i].w - mean;
            q = fmaf(ex, ex, q);
            q = fmaf(ey, ey, q);
            q = fmaf(ez, ez, q);
            q = fmaf(ew, ew, q);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float r = rsqrtf(q / (float)d + eps);
    const long long yr = seg_base(yl, plan.cf, seg) + t;
#pragma unroll
    for (int i = 0; i < PG; i++) {
        const int c4 = lane + 32 * i;
        if (c4 < d4) {
            const float4 gg = __ldg(reinterpret_cast<const float4*>(g) + c4);
            const float4 bb = __ldg(reinterpret_cast<const float4*>(b) + c4);
            const float4 o =
                make_float4(fmaf((v[i].x - mean) * r, gg.x, bb.x), fmaf((v[i].y - mean) * r, gg.y, bb.y),
                            fmaf((v[i].z - mean) * r, gg.z, bb.z), fmaf((v[i].w - mean) * r, gg.w, bb.w));
            if (planes) plane_store4(planes, planes_il, yr, d, 4 * c4, o);
            else reinterpret_cast<float4*>(y + yr * d)[c4] = o;
        }
    }
}

// spec rows of the call (packed, pitch `pitch`) -> [B][T_max][width] at each
// entry's row in the caller's batch, the layout the iSTFT head reads.
__global__ void vocos_scatter_kernel(const float* __restrict__ spec, int pitch, int width, int T_max, PlanView plan,
                                     int total_rows, float* __restrict__ out)
{
    pdl_wait();
    pdl_launch();
    const int row = blockIdx.x;
    if (row >= total_rows) return;
    const int seg = find_seg(plan.cf, plan.B, row);
    const int t = row - __ldg(plan.cf + seg);
    const float* src = spec + (size_t)row * pitch;
    float* dst = out + ((size_t)__ldg(plan.bidx + seg) * T_max + t) * width;
    for (int c = threadIdx.x; c < width; c += blockDim.x) dst[c] = src[c];
}

}  // namespace

struct codec_vocos_s {
    codec_vocos_config cfg{};
    int num_sms = 0;
    int P = 0;                       // history rows in front of each segment (k - 1, at least 1)
    VContraction embed, head;        // head: N padded to Hp = n_fft + 2 rounded up to 16 (zero columns)
    int Mp = 0;                      // mel channels padded to a multiple of 32 (zero channels): the
                                     // embedding conv's input width, so that it runs on the tensor cores
    int Hp = 0;
    float *norm_g = nullptr, *norm_b = nullptr, *final_g = nullptr, *final_b = nullptr;
    std::vector<VBlock> blocks;
    float* zeros = nullptr;          // [n_mels] / ones: the mel copy's identity affine
    float* ones = nullptr;
    // activations
    float* mel = nullptr;            // prefixed [rows][Mp], channels n_mels .. Mp - 1 zero
    std::vector<float*> xb;          // block inputs x_0 .. x_L, prefixed [rows][d]
    float* emb = nullptr;            // dense [rows][d]
    float* u = nullptr;              // dense [rows][d]
    float* f = nullptr;              // dense [rows][ffn]
    float* spec = nullptr;           // dense [rows][n_fft + 2]
    float* spec_b = nullptr;         // [S][max_chunk][n_fft + 2]
    TcScratch tc;
    std::vector<HistDesc> hist;
    HistDesc* hist_d = nullptr;
    long long* frames_d = nullptr;
    unsigned* err_d = nullptr;
    codec_istft_t* istft = nullptr;
    // plan: cf [S + 1], slot [S], pos0 [2 S] (8-byte), bidx [S], t64 [S + 1], t128 [S + 1]
    int plan_ints = 0, off_pos0 = 0, off_cf = 0, off_slot = 0, off_bidx = 0, off_t64 = 0, off_t128 = 0;
    int* plan_d = nullptr;
    int* plan_h[kPlanRing] = {};
    cudaEvent_t plan_ev[kPlanRing] = {};
    int plan_next = 0;
    int* slots_d = nullptr;
    std::vector<long long> frames_h;
    std::vector<void*> allocs;
    int last_launches = 0;
};

namespace {

bool vcfg_valid(const codec_vocos_config* c)
{
    auto m4 = [](int v) { return v > 0 && v % 4 == 0; };
    if (!m4(c->n_mels) || !m4(c->d) || c->d > 1024 || !m4(c->ffn) || c->layers < 0 || c->layers > 64) return false;
    if (c->k < 1 || c->k > kMaxTaps) return false;
    if (c->n_fft < 4 || c->n_fft > 4096 || (c->n_fft & 1) || c->hop < 1 || c->n_fft % c->hop) return false;
    if (!(c->ln_eps > 0.f)) return false;
    if (c->max_streams < 1 || c->max_chunk_frames < 1 || c->max_batch_frames < c->max_chunk_frames) return false;
    if ((long long)c->max_batch_frames * std::max(c->ffn, c->n_fft + 2) > (1LL << 31)) return false;
    if (c->precision != CODEC_PRECISION_FP32 && c->precision != CODEC_PRECISION_FP16X3 &&
        c->precision != CODEC_PRECISION_FP16)
        return false;
    return true;
}

long long vblob_floats(const codec_vocos_config* c)
{
    const long long d = c->d, F = c->ffn, H = c->n_fft + 2;
    long long n = d * c->n_mels * c->k + d + 2 * d;
    n += (long long)c->layers * (d * c->k + d + 2 * d + F * d + F + d * F + d + d);
    n += 2 * d + H * d + H;
    return n;
}

template <class T>
T* valloc(codec_vocos_s* s, size_t n, codec_status& st, bool zero = false)
{
    if (st != CODEC_OK) return nullptr;
    void* p = nullptr;
    if (cudaMalloc(&p, std::max<size_t>(n, 1) * sizeof(T)) != cudaSuccess) {
        st = CODEC_ERR_OOM;
        return nullptr;
    }
    s->allocs.push_back(p);
    if (zero && cudaMemset(p, 0, std::max<size_t>(n, 1) * sizeof(T)) != cudaSuccess) st = CODEC_ERR_CUDA;
    return static_cast<T*>(p);
}

template <class T>
T* vupload(codec_vocos_s* s, const T* src, size_t n, codec_status& st)
{
    T* p = valloc<T>(s, n, st);
    if (p && cudaMemcpy(p, src, n * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess) st = CODEC_ERR_CUDA;
    return p;
}

// wkn: [K][N] fp32 host, K = ntaps * Cin tap-major.
void vfinish(codec_vocos_s* s, VContraction& C, const std::vector<float>& wkn, const float* bias,
             codec_status& st)
{
    C.K = C.ntaps * C.Cin;
    C.w = vupload(s, wkn.data(), wkn.size(), st);
    if (bias) C.bias = vupload(s, bias, (size_t)C.N, st);
    C.use_tc = s->cfg.precision != CODEC_PRECISION_FP32 && tc_eligible(C.Cin, C.N);
    if (C.use_tc && st == CODEC_OK) {
        const int passes = s->cfg.precision == CODEC_PRECISION_FP16 ? 1 : 3;
        if (!tc_pack_weights(wkn.data(), C.ntaps, C.Cin, C.N, passes, &C.tc, s->allocs)) st = CODEC_ERR_OOM;
    }
}

// Linear [N][K] (times a per-output scale when given) -> [K][N].
void vlinear(codec_vocos_s* s, VContraction& C, const float* w, const float* b, const float* scale, int K, int N,
             codec_status& st)
{
    C.Cin = K; C.N = N; C.ntaps = 1; C.shift[0] = 0;
    std::vector<float> p((size_t)K * N), bias(N);
    for (int o = 0; o < N; o++) {
        const double sc = scale ? (double)scale[o] : 1.0;
        for (int i = 0; i < K; i++) p[(size_t)i * N + o] = (float)((double)w[(size_t)o * K + i] * sc);
        bias[o] = (float)((double)b[o] * sc);
    }
    vfinish(s, C, p, bias.data(), st);
}

void vfree(codec_vocos_s* s)
{
    for (int i = 0; i < kPlanRing; i++) {
        if (s->plan_h[i]) cudaFreeHost(s->plan_h[i]);
        if (s->plan_ev[i]) cudaEventDestroy(s->plan_ev[i]);
    }
    if (s->istft) codec_istft_destroy(s->istft);
    for (void* p : s->allocs) cudaFree(p);
    delete s;
}

}  // namespace

extern "C" {

int64_t codec_vocos_weight_floats(const codec_vocos_config* cfg)
{
    if (!cfg || !vcfg_valid(cfg)) return -1;
    return vblob_floats(cfg);
}

codec_status codec_vocos_create(const codec_vocos_config* cfg, const float* weights, int64_t n_floats,
                                codec_vocos_t** out)
{
    if (!out) return CODEC_ERR_NULL;
    *out = nullptr;
    if (!cfg || !weights) return CODEC_ERR_NULL;
    if (!vcfg_valid(cfg)) return CODEC_ERR_CONFIG;
    if (n_floats != vblob_floats(cfg)) return CODEC_ERR_WEIGHTS;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return CODEC_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return CODEC_ERR_NO_DEVICE;
    codec_vocos_s* s = new codec_vocos_s();
    s->cfg = *cfg;
    s->num_sms = prop.multiProcessorCount;
    const codec_vocos_config& g = s->cfg;
    codec_status st = CODEC_OK;
    const int d = g.d, k = g.k, S = g.max_streams, H = g.n_fft + 2;
    s->P = std::max(k - 1, 1);

    const float* p = weights;
    auto take = [&](long long n) { const float* r = p; p += n; return r; };
    {   // embedding conv [d][n_mels][k] -> [k Mp][d] (zero rows for the pad
        // channels, which add exact zeros), tap j reads row t - (k - 1 - j)
        const float* w = take((long long)d * g.n_mels * k);
        const float* b = take(d);
        s->Mp = (g.n_mels + 31) / 32 * 32;
        const int Mp = s->Mp;
        VContraction& C = s->embed;
        C.Cin = Mp; C.N = d; C.ntaps = k;
        for (int j = 0; j < k; j++) C.shift[j] = k - 1 - j;
        std::vector<float> wkn((size_t)k * Mp * d, 0.f);
        for (int co = 0; co < d; co++)
            for (int ci = 0; ci < g.n_mels; ci++)
                for (int j = 0; j < k; j++) wkn[((size_t)j * Mp + ci) * d + co] = w[((size_t)co * g.n_mels + ci) * k + j];
        vfinish(s, C, wkn, b, st);
    }
    s->norm_g = vupload(s, take(d), d, st);
    s->norm_b = vupload(s, take(d), d, st);
    s->blocks.resize(g.layers);
    for (int l = 0; l < g.layers; l++) {
        VBlock& B = s->blocks[l];
        const float* dw = take((long long)d * k);
        std::vector<float> dwt((size_t)k * d);
        for (int c = 0; c < d; c++)
            for (int j = 0; j < k; j++) dwt[(size_t)j * d + c] = dw[(size_t)c * k + j];
        B.dw_w = vupload(s, dwt.data(), dwt.size(), st);
        B.dw_b = vupload(s, take(d), d, st);
        B.ln_g = vupload(s, take(d), d, st);
        B.ln_b = vupload(s, take(d), d, st);
        const float* w1 = take((long long)g.ffn * d);
        const float* b1 = take(g.ffn);
        const float* w2 = take((long long)d * g.ffn);
        const float* b2 = take(d);
        const float* gamma = take(d);
        vlinear(s, B.pw1, w1, b1, nullptr, d, g.ffn, st);
        // the layer scale folded into the second layer (blixt/phonon "Weights"
        // does the same with the codec transformer's layer scales)
        vlinear(s, B.pw2, w2, b2, gamma, g.ffn, d, st);
    }
    s->final_g = vupload(s, take(d), d, st);
    s->final_b = vupload(s, take(d), d, st);
    {
        // the head's n_fft + 2 outputs padded with zero columns to a multiple
        // of 16 (the GEMMs read weight rows in 16-byte units; the tensor-core
        // path takes N in multiples of 16); the pad columns are never read
        const float* w = take((long long)H * d);
        const float* b = take(H);
        s->Hp = (H + 15) / 16 * 16;
        std::vector<float> wp((size_t)s->Hp * d, 0.f), bp(s->Hp, 0.f);
        std::memcpy(wp.data(), w, sizeof(float) * (size_t)H * d);
        std::memcpy(bp.data(), b, sizeof(float) * H);
        vlinear(s, s->head, wp.data(), bp.data(), nullptr, d, s->Hp, st);
    }
    {
        std::vector<float> z(g.n_mels, 0.f), o(g.n_mels, 1.f);
        s->zeros = vupload(s, z.data(), z.size(), st);
        s->ones = vupload(s, o.data(), o.size(), st);
    }
    // activations: chunk rows of every stream plus P history rows per stream
    const size_t R = (size_t)g.max_batch_frames, RP = R + (size_t)S * s->P;
    s->mel = valloc<float>(s, RP * s->Mp, st, true);
    s->xb.resize(g.layers + 1);
    for (int l = 0; l <= g.layers; l++) s->xb[l] = valloc<float>(s, RP * d, st);
    s->emb = valloc<float>(s, R * d, st);
    s->u = valloc<float>(s, R * d, st);
    s->f = valloc<float>(s, R * g.ffn, st);
    s->spec = valloc<float>(s, R * s->Hp, st);
    s->spec_b = valloc<float>(s, (size_t)S * g.max_chunk_frames * H, st);
    // carried rows: the embedding conv's mel rows, each block's input rows
    auto add_hist = [&](float* buf, int C) {
        if (k <= 1) return;
        HistDesc h;
        h.buf = buf; h.C = C; h.H = k - 1; h.l = Layout{1, s->P};
        h.state = valloc<float>(s, (size_t)S * (k - 1) * C, st, true);
        s->hist.push_back(h);
    };
    add_hist(s->mel, s->Mp);
    for (int l = 0; l < g.layers; l++) add_hist(s->xb[l], d);
    if (!s->hist.empty()) s->hist_d = vupload(s, s->hist.data(), s->hist.size(), st);
    s->frames_d = valloc<long long>(s, S, st, true);
    s->err_d = valloc<unsigned>(s, S, st, true);
    s->frames_h.assign(S, 0);
    if (st == CODEC_OK && g.precision != CODEC_PRECISION_FP32) {
        size_t elems = 4;
        auto need = [&](const VContraction& C, size_t rows) {
            if (C.use_tc) elems = std::max(elems, rows * (size_t)C.Cin);
        };
        need(s->embed, RP);
        for (const VBlock& B : s->blocks) {
            need(B.pw1, R);
            need(B.pw2, R);
        }
        need(s->head, R);
        if (!tc_scratch_alloc(&s->tc, elems, 1, 0, s->allocs)) st = CODEC_ERR_OOM;
    }
    s->off_pos0 = 0;
    s->off_cf = 2 * S;
    s->off_slot = s->off_cf + S + 1;
    s->off_bidx = s->off_slot + S;
    s->off_t64 = s->off_bidx + S;
    s->off_t128 = s->off_t64 + S + 1;
    s->plan_ints = s->off_t128 + S + 1;
    s->plan_d = valloc<int>(s, s->plan_ints, st, true);
    s->slots_d = valloc<int>(s, S, st);
    for (int i = 0; i < kPlanRing && st == CODEC_OK; i++) {
        if (cudaMallocHost(&s->plan_h[i], sizeof(int) * s->plan_ints) != cudaSuccess) st = CODEC_ERR_OOM;
        else if (cudaEventCreateWithFlags(&s->plan_ev[i], cudaEventDisableTiming) != cudaSuccess) st = CODEC_ERR_CUDA;
    }
    if (st == CODEC_OK) {
        codec_istft_config ic{g.n_fft, g.hop, g.mag_clip, S, g.max_chunk_frames};
        st = codec_istft_create(&ic, &s->istft);
    }
    if (st == CODEC_OK && (configure_simt_kernels() != cudaSuccess || tc_configure() != cudaSuccess))
        st = CODEC_ERR_CUDA;
    if (st == CODEC_OK && cudaDeviceSynchronize() != cudaSuccess) st = CODEC_ERR_CUDA;
    if (st != CODEC_OK) {
        vfree(s);
        return st;
    }
    *out = s;
    return CODEC_OK;
}

void codec_vocos_destroy(codec_vocos_t* s)
{
    if (!s) return;
    cudaDeviceSynchronize();
    vfree(s);
}

codec_status codec_vocos_reset(codec_vocos_t* s, const int32_t* ids, int32_t n, void* stream)
{
    if (!s) return CODEC_ERR_NULL;
    const int S = s->cfg.max_streams;
    std::vector<int> list;
    if (ids) {
        if (n < 0 || n > S) return CODEC_ERR_ARG;
        std::vector<char> seen(S, 0);
        for (int i = 0; i < n; i++) {
            if (ids[i] < 0 || ids[i] >= S || seen[ids[i]]) return CODEC_ERR_ARG;
            seen[ids[i]] = 1;
            list.push_back(ids[i]);
        }
    } else {
        for (int i = 0; i < S; i++) list.push_back(i);
    }
    if (list.empty()) return CODEC_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int i = s->plan_next;
    s->plan_next = (i + 1) % kPlanRing;
    if (cudaEventSynchronize(s->plan_ev[i]) != cudaSuccess) return CODEC_ERR_CUDA;
    std::memcpy(s->plan_h[i], list.data(), sizeof(int) * list.size());
    if (cudaMemcpyAsync(s->slots_d, s->plan_h[i], sizeof(int) * list.size(), cudaMemcpyHostToDevice, cs) !=
            cudaSuccess ||
        cudaEventRecord(s->plan_ev[i], cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    if (launch_state_reset(s->hist_d, (int)s->hist.size(), s->slots_d, (int)list.size(), s->frames_d, s->err_d,
                           cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    const codec_status r = codec_istft_reset(s->istft, list.data(), (int32_t)list.size(), stream);
    if (r != CODEC_OK) return r;
    for (int id : list) s->frames_h[id] = 0;
    return CODEC_OK;
}

codec_status codec_vocos_decode(codec_vocos_t* s, const float* mel, const int32_t* n_frames, const int32_t* ids,
                                int32_t B, int32_t T_max, float* audio, void* stream)
{
    if (!s || !mel || !n_frames || !audio) return CODEC_ERR_NULL;
    const codec_vocos_config& g = s->cfg;
    const int S = g.max_streams;
    if (B < 1 || T_max < 1) return CODEC_ERR_ARG;
    if (B > S) return CODEC_ERR_CAPACITY;
    std::vector<char> seen(S, 0);
    long long total = 0;
    for (int b = 0; b < B; b++) {
        const int id = ids ? ids[b] : b;
        if (id < 0 || id >= S || seen[id]) return CODEC_ERR_ARG;
        seen[id] = 1;
        if (n_frames[b] < 0 || n_frames[b] > T_max) return CODEC_ERR_ARG;
        if (n_frames[b] > g.max_chunk_frames) return CODEC_ERR_CAPACITY;
        total += n_frames[b];
    }
    if (T_max > g.max_chunk_frames) return CODEC_ERR_CAPACITY;
    if (total > g.max_batch_frames) return CODEC_ERR_CAPACITY;
    s->last_launches = 0;
    if (total == 0) return CODEC_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    // plan
    const int pi = s->plan_next;
    s->plan_next = (pi + 1) % kPlanRing;
    if (cudaEventSynchronize(s->plan_ev[pi]) != cudaSuccess) return CODEC_ERR_CUDA;
    int* P = s->plan_h[pi];
    long long* pos0 = reinterpret_cast<long long*>(P + s->off_pos0);
    int* cf = P + s->off_cf;
    int* slot = P + s->off_slot;
    int* bidx = P + s->off_bidx;
    int* t64 = P + s->off_t64;
    int* t128 = P + s->off_t128;
    int Bc = 0;
    cf[0] = t64[0] = t128[0] = 0;
    std::vector<int> slot_h, n_h;
    for (int b = 0; b < B; b++) {
        if (n_frames[b] == 0) continue;
        const int id = ids ? ids[b] : b;
        slot[Bc] = id;
        bidx[Bc] = b;
        pos0[Bc] = s->frames_h[id];
        cf[Bc + 1] = cf[Bc] + n_frames[b];
        t64[Bc + 1] = t64[Bc] + (n_frames[b] + 63) / 64;
        t128[Bc + 1] = t128[Bc] + (n_frames[b] + 127) / 128;
        slot_h.push_back(id);
        n_h.push_back(n_frames[b]);
        Bc++;
    }
    if (cudaMemcpyAsync(s->plan_d, P, sizeof(int) * s->plan_ints, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaEventRecord(s->plan_ev[pi], cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    const int* D = s->plan_d;
    const PlanView pv{Bc, D + s->off_cf, D + s->off_slot, reinterpret_cast<const long long*>(D + s->off_pos0),
                      D + s->off_bidx, nullptr};
    const int rows = (int)total;
    const int n64 = t64[Bc], n128 = t128[Bc];
    const Layout Lp{1, s->P}, Ld{1, 0};
    const int d = g.d, H = g.n_fft + 2;
    cudaError_t err = cudaSuccess;
    int launches = 0;
    auto ok = [&](cudaError_t e) {
        launches++;
        if (e != cudaSuccess && err == cudaSuccess) err = e;
        return err == cudaSuccess;
    };
    // from_producer: the LayerNorm before the linear already wrote its operand planes
    auto gemm = [&](const VContraction& C, const float* in, Layout il, float* out, Layout ol, const float* res,
                    int epi, bool from_producer = false, bool a_gelu = false) {
        if (err != cudaSuccess) return;
        GemmArgs a{};
        a.in = in; a.in_l = il; a.Cin = C.Cin; a.ntaps = C.ntaps;
        for (int j = 0; j < C.ntaps; j++) a.shift[j] = C.shift[j];
        a.N = C.N; a.K = C.K; a.w = C.w;
        a.bias = C.bias; a.bias_mod = C.N;
        a.out = out; a.out_l = ol; a.out_C = C.N; a.out_step = 1;
        a.res = res; a.epi = epi; a.scale = 1.f; a.pos_r = 1;
        if (C.use_tc) {
            a.tcum = D + s->off_t128;
            a.bm = 128;
            a.dense = (il.P == 0 && ol.P == 0 && C.ntaps == 1) ? 1 : 0;
            const int tiles = a.dense ? (rows + 127) / 128 : n128;
            const long long arows = rows + (long long)Bc * il.P;
            if (!from_producer)
                ok(launch_tc_prep(in, nullptr, nullptr, arows, C.Cin, &s->tc, C.tc.passes == 3, cs, a_gelu));
            int extra = 0;
            ok(launch_tc_gemm(a, C.tc, pv, tiles, &s->tc, arows, s->num_sms, cs, &extra));
            launches += extra > 1 ? extra - 1 : 0;
        } else {
            a.tcum = D + s->off_t64;
            a.bm = 64;
            ok(launch_gemm_simt(a, pv, n64, cs));
        }
    };
    // to: the linear that reads y next; when it runs on the tensor cores the
    // LayerNorm writes its operand planes instead of y (returns true)
    auto ln = [&](const float* x, Layout xl, const float* dw, const float* dwb, const float* gg, const float* bb,
                  float* y, Layout yl, const VContraction* to = nullptr) {
        if (err != cudaSuccess) return false;
        void* pl = (to && to->use_tc && yl.P == 0) ? s->tc.a_hi : nullptr;
        const int il = to && to->tc.passes == 3 ? 1 : 0;
        const dim3 grid((rows + 7) / 8), blk(256);
        if (d <= 512 && dw && g.k == 7)
            launch_pdl(vocos_ln_kernel<7, 4>, grid, blk, 0, cs, x, xl, dw, dwb, g.k, gg, bb, g.ln_eps, d, y, yl, pv,
                       rows, pl, il);
        else if (d <= 512)
            launch_pdl(vocos_ln_kernel<0, 4>, grid, blk, 0, cs, x, xl, dw, dwb, g.k, gg, bb, g.ln_eps, d, y, yl, pv,
                       rows, pl, il);
        else
            launch_pdl(vocos_ln_kernel<0, 8>, grid, blk, 0, cs, x, xl, dw, dwb, g.k, gg, bb, g.ln_eps, d, y, yl, pv,
                       rows, pl, il);
        ok(cudaGetLastError());
        return pl != nullptr;
    };

    if (!s->hist.empty()) ok(launch_hist_fill(s->hist_d, (int)s->hist.size(), pv, cs));
    ok(launch_latent_fill(mel, g.n_mels, T_max, pv, s->zeros, s->ones, s->mel, Lp, rows, cs, s->Mp));
    gemm(s->embed, s->mel, Lp, s->emb, Ld, nullptr, EPI_STORE);
    ln(s->emb, Ld, nullptr, nullptr, s->norm_g, s->norm_b, s->xb[0], Lp);
    for (int l = 0; l < g.layers; l++) {
        const VBlock& Bk = s->blocks[l];
        const bool p1 = ln(s->xb[l], Lp, Bk.dw_w, Bk.dw_b, Bk.ln_g, Bk.ln_b, s->u, Ld, &Bk.pw1);
        // the GELU in the second linear's operand prep on the tensor cores (same bits)
        const bool gp = Bk.pw1.use_tc && Bk.pw2.use_tc;
        gemm(Bk.pw1, s->u, Ld, s->f, Ld, nullptr, gp ? EPI_STORE : EPI_GELU, p1);
        gemm(Bk.pw2, s->f, Ld, s->xb[l + 1], Lp, s->xb[l], EPI_RESID, false, gp);
    }
    const bool ph = ln(s->xb[g.layers], Lp, nullptr, nullptr, s->final_g, s->final_b, s->u, Ld, &s->head);
    gemm(s->head, s->u, Ld, s->spec, Ld, nullptr, EPI_STORE, ph);
    if (err == cudaSuccess) {
        launch_pdl(vocos_scatter_kernel, dim3(rows), dim3(256), 0, cs, (const float*)s->spec, s->Hp, H, T_max, pv,
                   rows, s->spec_b);
        ok(cudaGetLastError());
    }
    if (!s->hist.empty()) ok(launch_hist_commit(s->hist_d, (int)s->hist.size(), pv, nullptr, s->frames_d, cs));
    if (err != cudaSuccess) return CODEC_ERR_CUDA;
    const codec_status r = codec_istft_decode(s->istft, s->spec_b, n_frames, ids, B, T_max, audio, stream);
    if (r != CODEC_OK) return r;
    for (size_t b = 0; b < slot_h.size(); b++) s->frames_h[slot_h[b]] += n_h[b];
    s->last_launches = launches + 2;
    return CODEC_OK;
}

}  // extern "C"
