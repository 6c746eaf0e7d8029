// Host runtime and C ABI of the decoder: configuration checks, weight repack
// and upload, stream-slot state, per-call planning of ragged multi-stream
// batches, and the launch sequence.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "codec.h"
#include "kernels.h"
#include "tc_gemm.h"

using namespace codec;

namespace {

// Weights of one contraction (conv, transposed conv or linear) in the packed
// implicit-GEMM form: K = ntaps * Cin rows (tap-major), N columns.
struct Contraction {
    float* w = nullptr;            // fp32 [K][N] (CUDA-core path)
    TcWeights tc;                  // fp16 hi/lo planes [N][K] (tensor-core path)
    bool use_tc = false;
    float* bias = nullptr;
    int bias_mod = 1;
    float* alpha = nullptr;        // Snake on the input, or null
    float* inv_alpha = nullptr;
    int Cin = 0, N = 0, K = 0, ntaps = 0;
    int shift[kMaxTaps] = {};
};

struct LayerW {
    float* n1 = nullptr;
    float* n2 = nullptr;
    Contraction qkv, o, w1, w2;
};

bool debug_sync()
{
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("CODEC_DEBUG_SYNC");
        v = (e && *e && *e != '0') ? 1 : 0;
    }
    return v == 1;
}

struct GraphEntry {
    std::vector<long long> key;
    cudaGraphExec_t exec;
    int launches;
    unsigned long long used;
};

struct ProfRec {
    int kind;
    double flops, bytes;
    double ms;
};

int next_pow2(int x)
{
    int r = 1;
    while (r < x) r <<= 1;
    return r;
}

}  // namespace

struct codec_s {
    codec_config cfg{};
    int device = 0;
    int spf = 0;
    int n_levels = 0;
    int level_r[16] = {};
    int num_sms = 0;
    int lvl_tf = 0;                // level of the transformer rows: 0 (code input) or 1 (latent input)
    int r_tf = 1;                  // transformer rows (positions) per frame
    float* cb = nullptr;
    Contraction pre;               // code input: the causal pre-conv; latent input: the folded
                                   // projection + depthwise upsampling phase GEMM
    float* lat_mu = nullptr;       // latent input: denormalisation
    float* lat_sigma = nullptr;
    std::vector<LayerW> layers;
    float* tf_norm = nullptr;
    Contraction up[4];
    Contraction st[8];
    std::vector<Contraction> rb;   // [stage][resblock][dilation]
    float* out_w = nullptr;        // [final_k][C_n]
    float* out_b = nullptr;
    float* out_alpha = nullptr;
    float* out_inv_alpha = nullptr;
    std::vector<void*> allocs;
    int rb_index(int s, int j, int i) const { return (s * cfg.n_rb + j) * cfg.n_dil + i; }
};

struct codec_state_s {
    codec_s* c = nullptr;
    int n_slots = 0;
    int R = 0;
    float* kring = nullptr;
    float* vring = nullptr;
    long long* frames_d = nullptr;
    unsigned* err_d = nullptr;
    std::vector<long long> frames_h;
    std::vector<HistDesc> hist;
    HistDesc* hist_d = nullptr;
    int P[16] = {};
    float *e = nullptr, *h = nullptr, *u = nullptr, *q = nullptr, *o = nullptr, *f = nullptr, *hf = nullptr;
    float* up_out[4] = {};
    float* x0[8] = {};
    float* rbuf[8][4][4] = {};
    float* y[8] = {};
    // small calls: resblocks 1 and 2's own outputs before the MRF sum
    static constexpr int kMrfSmallFrames = 8;
    float* ymrf[8][4] = {};
    TcScratch tc_scratch;
    // Resblock chains 1 and 2 of an MRF run their convs before the last one on
    // side streams, each with its own operand planes and split-K partials
    // (chain 0 uses tc_scratch on the caller's stream).
    static constexpr int kChains = 3;
    TcScratch tc_chain[kChains - 1];
    cudaStream_t side[kChains - 1] = {};
    cudaEvent_t fork_ev = nullptr;
    cudaEvent_t done_ev[kChains - 1] = {};
    // plan: device copy and a ring of page-locked host staging copies
    int plan_ints = 0;
    int off_pos0 = 0, off_cf = 0, off_slot = 0, off_bidx = 0, off_tc64 = 0, off_tc128 = 0, off_q16 = 0, off_skip = 0;
    int* plan_d = nullptr;
    static constexpr int kPlanRing = 8;
    int* plan_h[kPlanRing] = {};
    cudaEvent_t plan_ev[kPlanRing] = {};
    int plan_next = 0;
    int* slots_d = nullptr;
    int* slots_h = nullptr;
    cudaEvent_t slots_ev = nullptr;
    int* codes_d = nullptr;        // host-buffer entry point staging
    float* audio_d = nullptr;
    int last_launches = 0;
    double hist_floats_per_slot = 0.0;
    // captured launch sequences, keyed by call shape and buffers
    static constexpr size_t kMaxGraphs = 32;
    bool graphs_on = true;
    cudaStream_t cap_stream = nullptr;
    std::vector<GraphEntry> graphs;
    std::vector<std::vector<long long>> seen;
    unsigned long long graph_clock = 0;
    // per-launch timing (codec_profile_begin / _end)
    bool prof_on = false;
    int prof_n = 0, prof_max = 0, prof_done = 0;
    std::vector<cudaEvent_t> prof_ev;
    std::vector<ProfRec> prof_rec;
    std::vector<void*> allocs;
};

// ------------------------------------------------------------- helpers ----

namespace {

bool cfg_valid(const codec_config* c)
{
    auto m4 = [](int v) { return v > 0 && v % 4 == 0; };
    const bool latent = c->latent_dim != 0;
    if (latent) {
        if (!m4(c->latent_dim) || c->tf_up < 1 || c->tf_up > 64) return false;
    } else {
        if (c->Q < 1 || c->Q > 64 || c->V < 1 || !m4(c->E)) return false;
        if (c->pre_k < 1 || c->pre_k > kMaxTaps) return false;
    }
    if (!m4(c->d) || c->heads < 1 || c->d % c->heads || c->d / c->heads > 128) return false;
    if (!m4(c->ffn) || c->layers < 0 || c->layers > 64 || c->window < 1 || c->window > kSwaWindowMax) return false;
    if (swa_smem_bytes(c->d / c->heads, c->window) > kSwaSmemMax) return false;
    if (c->n_up < (latent ? 0 : 1) || c->n_up > 4 || c->up_s < 1 || c->up_k != 2 * c->up_s) return false;
    for (int u = 0; u < c->n_up; u++) if (!m4(c->up_ch[u])) return false;
    if (c->n_stages < 1 || c->n_stages > 8) return false;
    for (int s = 0; s < c->n_stages; s++) if (c->strides[s] < 1 || !m4(c->ch[s])) return false;
    if (c->n_rb < 1 || c->n_rb > 3 || c->n_dil < 1 || c->n_dil > 4) return false;
    for (int j = 0; j < c->n_rb; j++) if (c->rb_k[j] < 1 || c->rb_k[j] > kMaxTaps) return false;
    for (int i = 0; i < c->n_dil; i++) if (c->dil[i] < 1 || c->dil[i] > 64) return false;
    if (c->final_k < 1 || c->final_k > kMaxTaps) return false;
    if (c->n_stages >= 1 && c->n_stages <= 8 &&
        final_conv_smem_bytes(c->ch[c->n_stages - 1], c->final_k) > kFinalSmemMax)
        return false;
    if (!(c->rms_eps > 0.f)) return false;
    if (c->max_streams < 1 || c->max_chunk_frames < 1 || c->max_batch_frames < c->max_chunk_frames) return false;
    if (c->precision != CODEC_PRECISION_FP32 && c->precision != CODEC_PRECISION_FP16X3 &&
        c->precision != CODEC_PRECISION_FP16)
        return false;
    long long spf = latent ? c->tf_up : 1;
    for (int u = 0; u < c->n_up; u++) spf *= c->up_s;
    for (int s = 0; s < c->n_stages; s++) spf *= c->strides[s];
    if (spf > (1 << 20)) return false;
    if ((long long)c->max_batch_frames * spf > (1LL << 30)) return false;
    return true;
}

long long blob_floats(const codec_config* c)
{
    long long n;
    if (c->latent_dim)   // mu, sigma, projection [d][L], depthwise taps [d][1][2 tf_up], bias [d]
        n = 2LL * c->latent_dim + (long long)c->d * c->latent_dim + (long long)c->d * 2 * c->tf_up + c->d;
    else
        n = (long long)c->Q * c->V * c->E + (long long)c->d * c->E * c->pre_k + c->d;
    n += (long long)c->layers * (2LL * c->d + 4LL * c->d * c->d + 2LL * c->ffn * c->d);
    n += c->d;
    long long cin = c->d;
    for (int u = 0; u < c->n_up; u++) {
        n += cin * c->up_ch[u] * c->up_k + c->up_ch[u];
        cin = c->up_ch[u];
    }
    for (int s = 0; s < c->n_stages; s++) {
        const long long co = c->ch[s];
        n += cin + cin * co * 2 * c->strides[s] + co;
        for (int j = 0; j < c->n_rb; j++) n += (long long)c->n_dil * (co + co * co * c->rb_k[j] + co);
        cin = co;
    }
    n += cin + cin * c->final_k + 1;
    return n;
}

template <class T>
T* dev_upload(std::vector<void*>& allocs, const T* src, size_t n, codec_status& st)
{
    if (st != CODEC_OK) return nullptr;
    T* p = nullptr;
    if (cudaMalloc(&p, sizeof(T) * (n ? n : 1)) != cudaSuccess) { st = CODEC_ERR_OOM; return nullptr; }
    allocs.push_back(p);
    if (n && cudaMemcpy(p, src, sizeof(T) * n, cudaMemcpyHostToDevice) != cudaSuccess) {
        st = CODEC_ERR_CUDA;
        return nullptr;
    }
    return p;
}

template <class T>
T* dev_alloc(std::vector<void*>& allocs, size_t n, codec_status& st, bool zero = false)
{
    if (st != CODEC_OK) return nullptr;
    T* p = nullptr;
    if (cudaMalloc(&p, sizeof(T) * (n ? n : 1)) != cudaSuccess) { st = CODEC_ERR_OOM; return nullptr; }
    allocs.push_back(p);
    if (zero && cudaMemset(p, 0, sizeof(T) * (n ? n : 1)) != cudaSuccess) st = CODEC_ERR_CUDA;
    return p;
}

// Fill a Contraction from packed host weights [K][N] and upload it.
void finish_contraction(codec_s* c, Contraction& C, const std::vector<float>& wkn,
                        const float* bias, int bias_mod, const float* alpha, codec_status& st)
{
    C.K = C.ntaps * C.Cin;
    C.w = dev_upload(c->allocs, wkn.data(), wkn.size(), st);
    C.bias_mod = bias_mod;
    if (bias) C.bias = dev_upload(c->allocs, bias, (size_t)bias_mod, st);
    if (alpha) {
        std::vector<float> inv(C.Cin);
        for (int i = 0; i < C.Cin; i++) inv[i] = 1.0f / alpha[i];
        C.alpha = dev_upload(c->allocs, alpha, (size_t)C.Cin, st);
        C.inv_alpha = dev_upload(c->allocs, inv.data(), inv.size(), st);
    }
    C.use_tc = c->cfg.precision != CODEC_PRECISION_FP32 && tc_eligible(C.Cin, C.N);
    if (C.use_tc && st == CODEC_OK) {
        const int passes = c->cfg.precision == CODEC_PRECISION_FP16 ? 1 : 3;
        if (!tc_pack_weights(wkn.data(), C.ntaps, C.Cin, C.N, passes, &C.tc, c->allocs)) st = CODEC_ERR_OOM;
    }
}

// Conv1d weight [Cout][Cin][k] -> [k Cin][Cout]; tap j reads row t - (k-1-j) dil.
void make_conv(codec_s* c, Contraction& C, const float* w, const float* b, const float* alpha,
               int Cin, int Cout, int k, int dil, codec_status& st)
{
    C.Cin = Cin; C.N = Cout; C.ntaps = k;
    for (int j = 0; j < k; j++) C.shift[j] = (k - 1 - j) * dil;
    std::vector<float> p((size_t)k * Cin * Cout);
    for (int co = 0; co < Cout; co++)
        for (int ci = 0; ci < Cin; ci++)
            for (int j = 0; j < k; j++)
                p[((size_t)j * Cin + ci) * Cout + co] = w[((size_t)co * Cin + ci) * k + j];
    finish_contraction(c, C, p, b, Cout, alpha, st);
}

// ConvTranspose1d weight [Cin][Cout][2s] -> phase GEMM [2 Cin][s Cout]:
// output column p Cout + co of input row n is row n s + p of the upsampled
// signal; tap 0 reads a[n-1] with W[:, :, p+s], tap 1 reads a[n] with
// W[:, :, p] (blixt/phonon "Weights": one GEMM per output phase, gathering
// its inputs, never scattering).
void make_convt(codec_s* c, Contraction& C, const float* w, const float* b, const float* alpha,
                int Cin, int Cout, int s, codec_status& st)
{
    C.Cin = Cin; C.N = s * Cout; C.ntaps = 2;
    C.shift[0] = 1;
    C.shift[1] = 0;
    const int k = 2 * s;
    std::vector<float> p((size_t)2 * Cin * s * Cout);
    for (int ci = 0; ci < Cin; ci++)
        for (int co = 0; co < Cout; co++)
            for (int ph = 0; ph < s; ph++) {
                const size_t n = (size_t)ph * Cout + co;
                p[(size_t)ci * C.N + n] = w[((size_t)ci * Cout + co) * k + ph + s];
                p[((size_t)Cin + ci) * C.N + n] = w[((size_t)ci * Cout + co) * k + ph];
            }
    finish_contraction(c, C, p, b, Cout, alpha, st);
}

// Latent front end: the 1x1 projection Wp [d][L] folded into the causal
// depthwise transposed conv u [d][1][2s] (blixt/phonon "Weights": the
// projection merged into the upsampling weights), as one phase GEMM
// [2 L][s d] over [z[n-1] | z[n]] (z = the denormalised latents):
//   y[n s + p][c] = b[c] + sum_l u[c][p+s] Wp[c][l] z[n-1][l] + u[c][p] Wp[c][l] z[n][l].
// The folded products are formed in double and rounded once.
void make_front(codec_s* c, Contraction& C, const float* Wp, const float* u, const float* b, int L, int d, int s,
                codec_status& st)
{
    C.Cin = L; C.N = s * d; C.ntaps = 2;
    C.shift[0] = 1;
    C.shift[1] = 0;
    std::vector<float> p((size_t)2 * L * s * d);
    for (int l = 0; l < L; l++)
        for (int ph = 0; ph < s; ph++)
            for (int ch = 0; ch < d; ch++) {
                const size_t n = (size_t)ph * d + ch;
                const double w = Wp[(size_t)ch * L + l];
                p[(size_t)l * C.N + n] = (float)((double)u[(size_t)ch * 2 * s + ph + s] * w);
                p[((size_t)L + l) * C.N + n] = (float)((double)u[(size_t)ch * 2 * s + ph] * w);
            }
    finish_contraction(c, C, p, b, d, nullptr, st);
}

// Linear weights [Cout][Cin] (several concatenated along Cout) -> [Cin][sum Cout].
void make_linear(codec_s* c, Contraction& C, std::vector<const float*> ws, int Cin, int Cout_each,
                 codec_status& st)
{
    const int N = Cout_each * (int)ws.size();
    C.Cin = Cin; C.N = N; C.ntaps = 1; C.shift[0] = 0;
    std::vector<float> p((size_t)Cin * N);
    for (size_t m = 0; m < ws.size(); m++)
        for (int o = 0; o < Cout_each; o++)
            for (int i = 0; i < Cin; i++)
                p[(size_t)i * N + m * Cout_each + o] = ws[m][(size_t)o * Cin + i];
    finish_contraction(c, C, p, nullptr, 1, nullptr, st);
}

void free_all(std::vector<void*>& v)
{
    for (void* p : v) cudaFree(p);
    v.clear();
}

}  // namespace

// ------------------------------------------------------------ C ABI -------

extern "C" {

const char* codec_status_string(codec_status s)
{
    switch (s) {
    case CODEC_OK: return "ok";
    case CODEC_ERR_NULL: return "a required pointer is NULL";
    case CODEC_ERR_CONFIG: return "invalid or unsupported configuration";
    case CODEC_ERR_WEIGHTS: return "weight blob length does not match the configuration";
    case CODEC_ERR_ARG: return "argument out of range or repeated stream id";
    case CODEC_ERR_CAPACITY: return "request exceeds the configured capacity";
    case CODEC_ERR_OOM: return "device allocation failed";
    case CODEC_ERR_CUDA: return "CUDA call failed";
    case CODEC_ERR_NO_DEVICE: return "no usable sm_103 device";
    }
    return "unknown status";
}

int64_t codec_weight_floats(const codec_config* cfg)
{
    if (!cfg || !cfg_valid(cfg)) return -1;
    return blob_floats(cfg);
}

int32_t codec_samples_per_frame(const codec_t* c) { return c ? c->spf : 0; }

codec_status codec_create(const codec_config* cfg, const float* weights, int64_t n_floats, codec_t** out)
{
    if (!out) return CODEC_ERR_NULL;
    *out = nullptr;
    if (!cfg || !weights) return CODEC_ERR_NULL;
    if (!cfg_valid(cfg)) return CODEC_ERR_CONFIG;
    if (n_floats != blob_floats(cfg)) return CODEC_ERR_WEIGHTS;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return CODEC_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return CODEC_ERR_NO_DEVICE;

    codec_s* c = new codec_s();
    c->cfg = *cfg;
    c->device = dev;
    c->num_sms = prop.multiProcessorCount;
    const codec_config& g = c->cfg;
    codec_status st = CODEC_OK;
    c->spf = 1;
    c->level_r[0] = 1;
    c->n_levels = 1;
    if (g.latent_dim) {
        c->lvl_tf = 1;
        c->r_tf = g.tf_up;
        c->spf = g.tf_up;
        c->level_r[c->n_levels++] = c->spf;
    }
    for (int u = 0; u < g.n_up; u++) { c->spf *= g.up_s; c->level_r[c->n_levels++] = c->spf; }
    for (int s = 0; s < g.n_stages; s++) { c->spf *= g.strides[s]; c->level_r[c->n_levels++] = c->spf; }

    const float* p = weights;
    auto take = [&](long long n) { const float* r = p; p += n; return r; };
    if (g.latent_dim) {
        const int L = g.latent_dim;
        c->lat_mu = dev_upload(c->allocs, take(L), (size_t)L, st);
        c->lat_sigma = dev_upload(c->allocs, take(L), (size_t)L, st);
        const float* wp = take((long long)g.d * L);
        const float* u = take((long long)g.d * 2 * g.tf_up);
        const float* b = take(g.d);
        make_front(c, c->pre, wp, u, b, L, g.d, g.tf_up, st);
    } else {
        c->cb = dev_upload(c->allocs, take((long long)g.Q * g.V * g.E), (size_t)g.Q * g.V * g.E, st);
        const float* w = take((long long)g.d * g.E * g.pre_k);
        const float* b = take(g.d);
        make_conv(c, c->pre, w, b, nullptr, g.E, g.d, g.pre_k, 1, st);
    }
    c->layers.resize(g.layers);
    for (int l = 0; l < g.layers; l++) {
        LayerW& L = c->layers[l];
        const long long dd = (long long)g.d * g.d;
        L.n1 = dev_upload(c->allocs, take(g.d), g.d, st);
        const float* wq = take(dd);
        const float* wk = take(dd);
        const float* wv = take(dd);
        const float* wo = take(dd);
        make_linear(c, L.qkv, {wq, wk, wv}, g.d, g.d, st);
        make_linear(c, L.o, {wo}, g.d, g.d, st);
        L.n2 = dev_upload(c->allocs, take(g.d), g.d, st);
        const float* w1 = take((long long)g.ffn * g.d);
        const float* w2 = take((long long)g.d * g.ffn);
        make_linear(c, L.w1, {w1}, g.d, g.ffn, st);
        make_linear(c, L.w2, {w2}, g.ffn, g.d, st);
    }
    c->tf_norm = dev_upload(c->allocs, take(g.d), g.d, st);
    int cin = g.d;
    for (int u = 0; u < g.n_up; u++) {
        const int co = g.up_ch[u];
        const float* w = take((long long)cin * co * g.up_k);
        const float* b = take(co);
        make_convt(c, c->up[u], w, b, nullptr, cin, co, g.up_s, st);
        cin = co;
    }
    c->rb.resize((size_t)g.n_stages * g.n_rb * g.n_dil);
    for (int s = 0; s < g.n_stages; s++) {
        const int co = g.ch[s];
        const float* alpha = take(cin);
        const float* w = take((long long)cin * co * 2 * g.strides[s]);
        const float* b = take(co);
        make_convt(c, c->st[s], w, b, alpha, cin, co, g.strides[s], st);
        for (int j = 0; j < g.n_rb; j++)
            for (int i = 0; i < g.n_dil; i++) {
                const float* a2 = take(co);
                const float* w2 = take((long long)co * co * g.rb_k[j]);
                const float* b2 = take(co);
                make_conv(c, c->rb[c->rb_index(s, j, i)], w2, b2, a2, co, co, g.rb_k[j], g.dil[i], st);
            }
        cin = co;
    }
    {
        const float* alpha = take(cin);
        const float* w = take((long long)cin * g.final_k);
        const float* b = take(1);
        std::vector<float> wt((size_t)g.final_k * cin), inv(cin);
        for (int ci = 0; ci < cin; ci++) {
            inv[ci] = 1.0f / alpha[ci];
            for (int j = 0; j < g.final_k; j++) wt[(size_t)j * cin + ci] = w[(size_t)ci * g.final_k + j];
        }
        c->out_w = dev_upload(c->allocs, wt.data(), wt.size(), st);
        c->out_b = dev_upload(c->allocs, b, 1, st);
        c->out_alpha = dev_upload(c->allocs, alpha, (size_t)cin, st);
        c->out_inv_alpha = dev_upload(c->allocs, inv.data(), inv.size(), st);
    }
    // kernel attributes (shared-memory carve-outs) are set once here, never
    // while a call's launches are being captured into a graph
    if (st == CODEC_OK && (configure_simt_kernels() != cudaSuccess || tc_configure() != cudaSuccess))
        st = CODEC_ERR_CUDA;
    if (st == CODEC_OK && cudaDeviceSynchronize() != cudaSuccess) st = CODEC_ERR_CUDA;
    if (st != CODEC_OK) {
        free_all(c->allocs);
        delete c;
        return st;
    }
    *out = c;
    return CODEC_OK;
}

void codec_destroy(codec_t* c)
{
    if (!c) return;
    cudaDeviceSynchronize();
    free_all(c->allocs);
    delete c;
}

codec_status codec_state_create(codec_t* c, int32_t n_streams, codec_state_t** out)
{
    if (!out) return CODEC_ERR_NULL;
    *out = nullptr;
    if (!c) return CODEC_ERR_NULL;
    const codec_config& g = c->cfg;
    if (n_streams < 0 || n_streams > (1 << 16)) return CODEC_ERR_ARG;
    codec_state_s* s = new codec_state_s();
    s->c = c;
    s->n_slots = n_streams ? n_streams : g.max_streams;
    const int S = s->n_slots;
    codec_status st = CODEC_OK;

    // per-level history rows in front of every segment; the transformer's
    // level (0, or 1 behind the latent front end) feeds the first ConvT
    const int last = c->n_levels - 1;
    const int lt = c->lvl_tf;
    s->P[0] = g.latent_dim ? 1 : std::max(g.pre_k - 1, 1);
    s->P[lt] = std::max(s->P[lt], 1);
    for (int u = 0; u < g.n_up; u++) s->P[lt + 1 + u] = 1;
    for (int si = 0; si < g.n_stages; si++) {
        int P = 1;
        for (int j = 0; j < g.n_rb; j++)
            for (int i = 0; i < g.n_dil; i++) P = std::max(P, (g.rb_k[j] - 1) * g.dil[i]);
        if (si == g.n_stages - 1) P = std::max(P, g.final_k - 1);
        s->P[lt + g.n_up + 1 + si] = P;
    }
    auto rows = [&](int lvl, bool pref) {
        return (size_t)g.max_batch_frames * c->level_r[lvl] + (pref ? (size_t)S * s->P[lvl] : 0);
    };
    auto& A = s->allocs;
    const size_t r0 = rows(lt, false);
    s->e = dev_alloc<float>(A, rows(0, true) * (g.latent_dim ? g.latent_dim : g.E), st);
    s->h = dev_alloc<float>(A, r0 * g.d, st);
    s->u = dev_alloc<float>(A, r0 * g.d, st);
    s->q = dev_alloc<float>(A, r0 * g.d, st);
    s->o = dev_alloc<float>(A, r0 * g.d, st);
    s->f = dev_alloc<float>(A, r0 * g.ffn, st);
    s->hf = dev_alloc<float>(A, rows(lt, true) * g.d, st);
    for (int u = 0; u < g.n_up; u++) s->up_out[u] = dev_alloc<float>(A, rows(lt + 1 + u, true) * g.up_ch[u], st);
    for (int si = 0; si < g.n_stages; si++) {
        const int lvl = lt + g.n_up + 1 + si;
        const size_t n = rows(lvl, true) * g.ch[si];
        s->x0[si] = dev_alloc<float>(A, n, st);
        for (int j = 0; j < g.n_rb; j++)
            for (int i = 1; i < g.n_dil; i++) s->rbuf[si][j][i] = dev_alloc<float>(A, n, st);
        s->y[si] = dev_alloc<float>(A, n, st);
    }
    (void)last;

    // carried state: histories, ring KV, counters
    auto add_hist = [&](float* buf, int C, int H, int lvl) {
        if (H <= 0) return;
        HistDesc d;
        d.buf = buf; d.C = C; d.H = H; d.l = Layout{c->level_r[lvl], s->P[lvl]};
        d.state = dev_alloc<float>(A, (size_t)S * H * C, st, true);
        s->hist.push_back(d);
        s->hist_floats_per_slot += (double)H * C;
    };
    if (g.latent_dim) add_hist(s->e, g.latent_dim, 1, 0);      // the front phase GEMM's z[n-1]
    else add_hist(s->e, g.E, g.pre_k - 1, 0);
    add_hist(s->hf, g.d, 1, lt);
    for (int u = 0; u < g.n_up; u++) add_hist(s->up_out[u], g.up_ch[u], 1, lt + 1 + u);
    for (int si = 0; si < g.n_stages; si++) {
        const int lvl = lt + g.n_up + 1 + si;
        int h0 = 0;
        for (int j = 0; j < g.n_rb; j++) h0 = std::max(h0, (g.rb_k[j] - 1) * g.dil[0]);
        add_hist(s->x0[si], g.ch[si], h0, lvl);
        for (int j = 0; j < g.n_rb; j++)
            for (int i = 1; i < g.n_dil; i++) add_hist(s->rbuf[si][j][i], g.ch[si], (g.rb_k[j] - 1) * g.dil[i], lvl);
        add_hist(s->y[si], g.ch[si], si == g.n_stages - 1 ? g.final_k - 1 : 1, lvl);
    }
    s->hist_d = dev_upload(A, s->hist.data(), s->hist.size(), st);
    s->R = next_pow2(g.max_chunk_frames * c->r_tf + g.window - 1);
    const size_t ring = (size_t)std::max(g.layers, 1) * S * s->R * g.d;
    s->kring = dev_alloc<float>(A, ring, st, true);
    s->vring = dev_alloc<float>(A, ring, st, true);
    s->frames_d = dev_alloc<long long>(A, S, st, true);
    s->err_d = dev_alloc<unsigned>(A, S, st, true);
    s->frames_h.assign(S, 0);

    // plan layout (ints); pos0 first for 8-byte alignment
    s->off_pos0 = 0;
    s->off_cf = 2 * S;
    s->off_slot = s->off_cf + S + 1;
    s->off_bidx = s->off_slot + S;
    s->off_tc64 = s->off_bidx + S;
    s->off_tc128 = s->off_tc64 + c->n_levels * (S + 1);
    s->off_q16 = s->off_tc128 + c->n_levels * (S + 1);
    s->off_skip = s->off_q16 + (S + 1);
    s->plan_ints = s->off_skip + S;
    s->plan_d = dev_alloc<int>(A, s->plan_ints, st, true);
    for (int i = 0; i < codec_state_s::kPlanRing && st == CODEC_OK; i++) {
        if (cudaMallocHost(&s->plan_h[i], sizeof(int) * s->plan_ints) != cudaSuccess) st = CODEC_ERR_OOM;
        else if (cudaEventCreateWithFlags(&s->plan_ev[i], cudaEventDisableTiming) != cudaSuccess) st = CODEC_ERR_CUDA;
    }
    if (st == CODEC_OK && cudaStreamCreateWithFlags(&s->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
        st = CODEC_ERR_CUDA;
    s->slots_d = dev_alloc<int>(A, S, st);
    if (st == CODEC_OK) {
        if (cudaMallocHost(&s->slots_h, sizeof(int) * S) != cudaSuccess) st = CODEC_ERR_OOM;
        else if (cudaEventCreateWithFlags(&s->slots_ev, cudaEventDisableTiming) != cudaSuccess) st = CODEC_ERR_CUDA;
    }
    s->codes_d = dev_alloc<int>(A, (size_t)S * std::max(g.Q, 1) * g.max_chunk_frames, st);
    s->audio_d = dev_alloc<float>(A, (size_t)S * g.max_chunk_frames * c->spf, st);
    if (st == CODEC_OK && g.precision != CODEC_PRECISION_FP32) {
        // operand planes for the widest tensor-core input: (contraction, input level, prefixed?)
        size_t elems = 0, b_elems = 0;
        auto need = [&](const Contraction& C, int lvl, bool pref) {
            if (C.use_tc) {
                elems = std::max(elems, rows(lvl, pref) * (size_t)C.Cin);
                b_elems = std::max(b_elems, (size_t)C.K * C.N);
            }
        };
        need(c->pre, 0, true);
        for (const LayerW& L : c->layers) {
            need(L.qkv, lt, false);
            need(L.o, lt, false);
            need(L.w1, lt, false);
            need(L.w2, lt, false);
        }
        for (int u = 0; u < g.n_up; u++) need(c->up[u], lt + u, true);
        for (int si = 0; si < g.n_stages; si++) {
            need(c->st[si], lt + g.n_up + si, true);
            for (int j = 0; j < g.n_rb; j++)
                for (int i = 0; i < g.n_dil; i++) need(c->rb[c->rb_index(si, j, i)], lt + g.n_up + 1 + si, true);
        }
        // split-GEMM partials: 64 M floats (256 MB)
        if (!tc_scratch_alloc(&s->tc_scratch, std::max<size_t>(elems, 4), b_elems, size_t(64) << 20, A))
            st = CODEC_ERR_OOM;
        // the side chains' planes, sized for the stages' inputs, and partials
        if (st == CODEC_OK && g.n_rb > 1) {
            size_t st_elems = 4;
            for (int si = 0; si < g.n_stages; si++)
                for (int j = 1; j < g.n_rb; j++)
                    for (int i = 0; i < g.n_dil; i++) {
                        const Contraction& C = c->rb[c->rb_index(si, j, i)];
                        if (C.use_tc) st_elems = std::max(st_elems, rows(lt + g.n_up + 1 + si, true) * (size_t)C.Cin);
                    }
            for (int j = 0; j < std::min(g.n_rb, (int)codec_state_s::kChains) - 1 && st == CODEC_OK; j++) {
                if (!tc_scratch_alloc(&s->tc_chain[j], st_elems, 1, size_t(64) << 20, A)) st = CODEC_ERR_OOM;
                s->tc_chain[j].err = s->tc_scratch.err;      // one timeout flag for the state
            }
        }
    }
    if (st == CODEC_OK && g.n_rb > 1) {
        for (int si = 0; si < g.n_stages; si++) {
            const int lvl = lt + g.n_up + 1 + si;
            const size_t n = ((size_t)codec_state_s::kMrfSmallFrames * c->level_r[lvl] +
                              (size_t)std::min(S, codec_state_s::kMrfSmallFrames) * s->P[lvl]) * g.ch[si];
            for (int j = 1; j < g.n_rb; j++) s->ymrf[si][j] = dev_alloc<float>(A, n, st);
        }
        for (int j = 0; j < codec_state_s::kChains - 1 && st == CODEC_OK; j++)
            if (cudaStreamCreateWithFlags(&s->side[j], cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&s->done_ev[j], cudaEventDisableTiming) != cudaSuccess)
                st = CODEC_ERR_CUDA;
        if (st == CODEC_OK && cudaEventCreateWithFlags(&s->fork_ev, cudaEventDisableTiming) != cudaSuccess)
            st = CODEC_ERR_CUDA;
    }
    if (st == CODEC_OK && cudaDeviceSynchronize() != cudaSuccess) st = CODEC_ERR_CUDA;
    if (st != CODEC_OK) {
        for (int i = 0; i < codec_state_s::kPlanRing; i++) {
            if (s->plan_h[i]) cudaFreeHost(s->plan_h[i]);
            if (s->plan_ev[i]) cudaEventDestroy(s->plan_ev[i]);
        }
        if (s->slots_h) cudaFreeHost(s->slots_h);
        if (s->slots_ev) cudaEventDestroy(s->slots_ev);
        if (s->cap_stream) cudaStreamDestroy(s->cap_stream);
        for (int j = 0; j < codec_state_s::kChains - 1; j++) {
            if (s->side[j]) cudaStreamDestroy(s->side[j]);
            if (s->done_ev[j]) cudaEventDestroy(s->done_ev[j]);
        }
        if (s->fork_ev) cudaEventDestroy(s->fork_ev);
        free_all(A);
        delete s;
        return st;
    }
    *out = s;
    return CODEC_OK;
}

void codec_state_destroy(codec_state_t* s)
{
    if (!s) return;
    cudaDeviceSynchronize();
    for (int i = 0; i < codec_state_s::kPlanRing; i++) {
        if (s->plan_h[i]) cudaFreeHost(s->plan_h[i]);
        if (s->plan_ev[i]) cudaEventDestroy(s->plan_ev[i]);
    }
    if (s->slots_h) cudaFreeHost(s->slots_h);
    if (s->slots_ev) cudaEventDestroy(s->slots_ev);
    for (cudaEvent_t e : s->prof_ev) cudaEventDestroy(e);
    for (GraphEntry& e : s->graphs) cudaGraphExecDestroy(e.exec);
    if (s->cap_stream) cudaStreamDestroy(s->cap_stream);
    for (int j = 0; j < codec_state_s::kChains - 1; j++) {
        if (s->side[j]) cudaStreamDestroy(s->side[j]);
        if (s->done_ev[j]) cudaEventDestroy(s->done_ev[j]);
    }
    if (s->fork_ev) cudaEventDestroy(s->fork_ev);
    free_all(s->allocs);
    delete s;
}

codec_status codec_state_set_graphs(codec_state_t* s, int32_t enable)
{
    if (!s) return CODEC_ERR_NULL;
    s->graphs_on = enable != 0;
    if (!s->graphs_on) {
        if (cudaDeviceSynchronize() != cudaSuccess) return CODEC_ERR_CUDA;
        for (GraphEntry& e : s->graphs) cudaGraphExecDestroy(e.exec);
        s->graphs.clear();
        s->seen.clear();
    }
    return CODEC_OK;
}

codec_status codec_state_set_wait_limit(codec_state_t* s, uint32_t polls, int32_t unarrived_wait)
{
    if (!s) return CODEC_ERR_NULL;
    TcWaitLimit wl;
    wl.polls = polls ? polls : kDefaultWaitPolls;
    wl.unarrived_wait = unarrived_wait ? 1 : 0;
    // captured graphs hold the old limits in their kernel arguments
    if (cudaDeviceSynchronize() != cudaSuccess) return CODEC_ERR_CUDA;
    for (GraphEntry& e : s->graphs) cudaGraphExecDestroy(e.exec);
    s->graphs.clear();
    s->seen.clear();
    s->tc_scratch.wait = wl;
    s->tc_scratch.op.wait = wl;
    for (TcScratch& t : s->tc_chain) t.wait = wl;
    return CODEC_OK;
}

codec_status codec_profile_begin(codec_state_t* s, int32_t max_records)
{
    if (!s) return CODEC_ERR_NULL;
    if (max_records < 1 || max_records > (1 << 20)) return CODEC_ERR_ARG;
    while ((int)s->prof_ev.size() < 2 * max_records) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return CODEC_ERR_CUDA;
        s->prof_ev.push_back(e);
    }
    s->prof_rec.assign(max_records, ProfRec{0, 0.0, 0.0, 0.0});
    s->prof_done = 0;
    s->prof_max = max_records;
    s->prof_n = 0;
    s->prof_on = true;
    return CODEC_OK;
}

codec_status codec_profile_end(codec_state_t* s, codec_kernel_stats* out, void* stream)
{
    if (!s || !out) return CODEC_ERR_NULL;
    s->prof_on = false;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CODEC_ERR_CUDA;
    for (int k = 0; k < CODEC_KERNEL_KINDS; k++) out[k] = codec_kernel_stats{k, 0, 0.0, 0.0, 0.0};
    for (int i = 0; i < s->prof_n; i++) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, s->prof_ev[2 * i], s->prof_ev[2 * i + 1]) != cudaSuccess) return CODEC_ERR_CUDA;
        codec_kernel_stats& o = out[s->prof_rec[i].kind];
        o.launches++;
        o.ms += ms;
        o.flops += s->prof_rec[i].flops;
        o.bytes += s->prof_rec[i].bytes;
        s->prof_rec[i].ms = ms;
    }
    s->prof_done = s->prof_n;
    s->prof_n = 0;
    return CODEC_OK;
}

codec_status codec_profile_launches(codec_state_t* s, codec_launch_record* out, int32_t max_out, int32_t* n_out)
{
    if (!s || !out || !n_out) return CODEC_ERR_NULL;
    if (max_out < 0) return CODEC_ERR_ARG;
    const int n = std::min(max_out, s->prof_done);
    for (int i = 0; i < n; i++)
        out[i] = codec_launch_record{s->prof_rec[i].kind, 0, s->prof_rec[i].ms, s->prof_rec[i].flops,
                                     s->prof_rec[i].bytes};
    *n_out = n;
    return CODEC_OK;
}

int32_t codec_state_streams(const codec_state_t* s) { return s ? s->n_slots : 0; }
int32_t codec_state_last_launches(const codec_state_t* s) { return s ? s->last_launches : 0; }

codec_status codec_state_reset(codec_state_t* s, const int32_t* ids, int32_t n, void* stream)
{
    if (!s) return CODEC_ERR_NULL;
    const int S = s->n_slots;
    std::vector<int> list;
    if (!ids) {
        for (int i = 0; i < S; i++) list.push_back(i);
    } else {
        if (n < 0 || n > S) return CODEC_ERR_ARG;
        std::vector<char> seen(S, 0);
        for (int i = 0; i < n; i++) {
            if (ids[i] < 0 || ids[i] >= S || seen[ids[i]]) return CODEC_ERR_ARG;
            seen[ids[i]] = 1;
            list.push_back(ids[i]);
        }
    }
    if (list.empty()) return CODEC_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    if (cudaEventSynchronize(s->slots_ev) != cudaSuccess) return CODEC_ERR_CUDA;
    std::memcpy(s->slots_h, list.data(), sizeof(int) * list.size());
    if (cudaMemcpyAsync(s->slots_d, s->slots_h, sizeof(int) * list.size(), cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    if (cudaEventRecord(s->slots_ev, cs) != cudaSuccess) return CODEC_ERR_CUDA;
    if (launch_state_reset(s->hist_d, (int)s->hist.size(), s->slots_d, (int)list.size(), s->frames_d,
                           s->err_d, cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    if (!ids && s->tc_scratch.err && cudaMemsetAsync(s->tc_scratch.err, 0, sizeof(int), cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    for (int i : list) s->frames_h[i] = 0;
    return CODEC_OK;
}

codec_status codec_state_conv1d(codec_state_t* s, const float* x, int32_t T, int32_t Cin, const float* w,
                                const float* bias, const float* alpha, int32_t Cout, int32_t k, int32_t dilation,
                                float* y, void* stream)
{
    if (!s || !x || !w || !y) return CODEC_ERR_NULL;
    if (!s->tc_scratch.op.words) return CODEC_ERR_CONFIG;
    const int r = run_tc_conv1d(s->tc_scratch.op, x, T, Cin, w, bias, alpha, Cout, k, dilation, y, s->c->num_sms,
                                (cudaStream_t)stream);
    switch (r) {
    case OP_OK: return CODEC_OK;
    case OP_BAD_ARG: return CODEC_ERR_ARG;
    case OP_TOO_BIG: return CODEC_ERR_CAPACITY;
    default: return CODEC_ERR_CUDA;
    }
}

codec_status codec_state_query(codec_state_t* s, int32_t id, codec_stream_info* info, void* stream)
{
    if (!s || !info) return CODEC_ERR_NULL;
    if (id < 0 || id >= s->n_slots) return CODEC_ERR_ARG;
    cudaStream_t cs = (cudaStream_t)stream;
    long long fr = 0;
    unsigned err = 0;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return CODEC_ERR_CUDA;
    if (cudaMemcpy(&fr, s->frames_d + id, sizeof(fr), cudaMemcpyDeviceToHost) != cudaSuccess) return CODEC_ERR_CUDA;
    if (cudaMemcpy(&err, s->err_d + id, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return CODEC_ERR_CUDA;
    if (s->tc_scratch.err) {
        int te = 0;
        if (cudaMemcpy(&te, s->tc_scratch.err, sizeof(te), cudaMemcpyDeviceToHost) != cudaSuccess) return CODEC_ERR_CUDA;
        if (te) err |= CODEC_STREAM_ERR_KERNEL_TIMEOUT;
    }
    info->frames_decoded = fr;
    info->error_bits = err;
    info->reserved = 0;
    return CODEC_OK;
}

}  // extern "C"

// ------------------------------------------------------- decode call ------

namespace {

struct Launcher {
    codec_state_s* s;
    cudaStream_t cs;
    TcScratch* scr = nullptr;               // operand planes and partials of the current chain
    PlanView pv;
    const int* tc64;     // device, [levels][S + 1]
    const int* tc128;
    const int* q16;                         // device, [S + 1] attention blocks of kSwaQueries frames
    int nq16 = 0;
    std::vector<int> ntiles64, ntiles128;   // per level
    std::vector<int> slot_h, n_h;           // host copies of the compacted batch
    long long frames = 0;                   // frames in this call
    int Bc = 0;                             // streams with frames in this call
    int launches = 0;
    cudaError_t err = cudaSuccess;
    const char* where = "";

    // Enqueue one kernel through f(), with an event pair around it when the
    // state is recording, and note its algorithmic work.
    template <class F>
    bool run(int kind, double flops, double bytes, const char* what, F&& f)
    {
        if (err != cudaSuccess) return false;
        const bool rec = s->prof_on && s->prof_n < s->prof_max;
        if (rec) cudaEventRecord(s->prof_ev[2 * s->prof_n], cs);
        cudaError_t e = f();
        launches++;
        if (rec) {
            cudaEventRecord(s->prof_ev[2 * s->prof_n + 1], cs);
            s->prof_rec[s->prof_n] = ProfRec{kind, flops, bytes, 0.0};
            s->prof_n++;
        }
        if (e != cudaSuccess) { err = e; where = what; }
        if (err == cudaSuccess && debug_sync()) {
            cudaError_t e2 = cudaStreamSynchronize(cs);
            if (e2 != cudaSuccess) { err = e2; where = what; }
        }
        return err == cudaSuccess;
    }

    long long rows(int lvl) const { return frames * s->c->level_r[lvl]; }
    int max_frames() const
    {
        int m = 0;
        for (int n : n_h) m = std::max(m, n);
        return m;
    }
    long long rows_pref(int lvl, Layout l) const { return frames * s->c->level_r[lvl] + (long long)Bc * l.P; }

    // from_producer: the operand planes are already in plane block 0, written
    // by the kernel that produced `in`; otherwise the prep kernel makes them
    // (of GELU(in) when a_gelu: tensor-core path only).
    void gemm(const Contraction& C, const float* in, Layout il, int in_lvl, float* out, Layout ol,
              int out_C, int out_step, const float* res, int epi, float scale, int layer_ring,
              const char* what, bool from_producer = false, bool a_gelu = false)
    {
        if (err != cudaSuccess) return;
        const int S1 = s->n_slots + 1;
        GemmArgs a{};
        a.in = in; a.in_l = il; a.Cin = C.Cin; a.ntaps = C.ntaps;
        for (int j = 0; j < C.ntaps; j++) a.shift[j] = C.shift[j];
        a.alpha = C.alpha; a.inv_alpha = C.inv_alpha;
        a.N = C.N; a.K = C.K; a.w = C.w;
        a.bias = C.bias; a.bias_mod = C.bias_mod;
        a.out = out; a.out_l = ol; a.out_C = out_C; a.out_step = out_step;
        a.res = res; a.epi = epi; a.scale = scale;
        if (epi == EPI_QKV) {
            const size_t per_layer = (size_t)s->n_slots * s->R * s->c->cfg.d;
            a.kring = s->kring + per_layer * layer_ring;
            a.vring = s->vring + per_layer * layer_ring;
            a.ring_R = s->R;
            a.d = s->c->cfg.d;
        }
        a.pos_r = s->c->r_tf;
        const double M = (double)rows(in_lvl);
        const double flops = 2.0 * M * C.N * C.K;
        const double out_rw = (epi == EPI_RESID || epi == EPI_MRF_FIRST) ? 2.0
                              : (epi == EPI_MRF_ADD || epi == EPI_MRF_LAST) ? 3.0 : 1.0;
        const double bytes = 4.0 * ((M + (double)Bc * C.shift[0]) * C.Cin + (double)C.K * C.N + M * C.N * out_rw);
        if (C.use_tc) {
            a.tcum = tc128 + (size_t)in_lvl * S1;
            a.bm = 128;
            // dense single-tap contractions tile all streams' rows back to back
            // (the transformer linears: 1600 rows of 64 streams are 13 tiles, not 64)
            a.dense = (il.P == 0 && ol.P == 0 && C.ntaps == 1 && out_step == 1) ? 1 : 0;
            const int n_row_tiles = a.dense ? (int)((rows(in_lvl) + 127) / 128) : ntiles128[in_lvl];
            const long long arows = il.P ? rows_pref(in_lvl, il) : rows(in_lvl);
            TcScratch* sc = scr ? scr : &s->tc_scratch;
            if (!from_producer)
                run(CODEC_KERNEL_OPERAND_PREP, 0.0, 8.0 * (double)arows * C.Cin, what, [&] {
                    return launch_tc_prep(in, C.alpha, C.inv_alpha, arows, C.Cin, sc, C.tc.passes == 3, cs, a_gelu);
                });
            int extra = 0;
            run(CODEC_KERNEL_GEMM_TC, flops, bytes, what, [&] {
                return launch_tc_gemm(a, C.tc, pv, n_row_tiles, sc, arows, s->c->num_sms, cs, &extra);
            });
            launches += extra > 1 ? extra - 1 : 0;   // the split reduction, timed with its GEMM
        } else {
            a.tcum = tc64 + (size_t)in_lvl * S1;
            a.bm = 64;
            run(CODEC_KERNEL_GEMM_SIMT, flops, bytes, what, [&] { return launch_gemm_simt(a, pv, ntiles64[in_lvl], cs); });
        }
    }
};

// Validate a call's batch, build its plan (cumulative frames, slots, tile
// counts per level) in a page-locked staging buffer and enqueue the upload.
codec_status plan_call(codec_state_t* s, const int32_t* n_frames, const int32_t* ids, int32_t B,
                       int32_t T_max, cudaStream_t cs, Launcher& L, int& rows0, const int32_t* skip_h = nullptr)
{
    codec_s* c = s->c;
    const codec_config& g = c->cfg;
    const int S = s->n_slots;
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
    if (total > g.max_batch_frames) return CODEC_ERR_CAPACITY;
    rows0 = (int)total;
    if (total == 0) return CODEC_OK;

    const int i = s->plan_next;
    s->plan_next = (i + 1) % codec_state_s::kPlanRing;
    if (cudaEventSynchronize(s->plan_ev[i]) != cudaSuccess) return CODEC_ERR_CUDA;
    int* P = s->plan_h[i];
    long long* pos0 = reinterpret_cast<long long*>(P + s->off_pos0);
    int* cf = P + s->off_cf;
    int* slot = P + s->off_slot;
    int* bidx = P + s->off_bidx;
    int* skip = P + s->off_skip;
    int Bc = 0;
    cf[0] = 0;
    for (int b = 0; b < B; b++) {
        if (n_frames[b] == 0) continue;
        const int id = ids ? ids[b] : b;
        slot[Bc] = id;
        bidx[Bc] = b;
        skip[Bc] = skip_h ? skip_h[b] : 0;
        pos0[Bc] = s->frames_h[id];
        cf[Bc + 1] = cf[Bc] + n_frames[b];
        Bc++;
    }
    const int S1 = S + 1;
    L.s = s;
    L.cs = cs;
    L.ntiles64.assign(c->n_levels, 0);
    L.ntiles128.assign(c->n_levels, 0);
    for (int lvl = 0; lvl < c->n_levels; lvl++) {
        int* t64 = P + s->off_tc64 + lvl * S1;
        int* t128 = P + s->off_tc128 + lvl * S1;
        t64[0] = t128[0] = 0;
        for (int b = 0; b < Bc; b++) {
            const long long rows = (long long)(cf[b + 1] - cf[b]) * c->level_r[lvl];
            t64[b + 1] = t64[b] + (int)((rows + 63) / 64);
            t128[b + 1] = t128[b] + (int)((rows + 127) / 128);
        }
        L.ntiles64[lvl] = t64[Bc];
        L.ntiles128[lvl] = t128[Bc];
    }
    {
        int* q16 = P + s->off_q16;
        q16[0] = 0;
        for (int b = 0; b < Bc; b++)
            q16[b + 1] = q16[b] + ((cf[b + 1] - cf[b]) * c->r_tf + kSwaQueries - 1) / kSwaQueries;
        L.nq16 = q16[Bc];
    }
    if (cudaMemcpyAsync(s->plan_d, P, sizeof(int) * s->plan_ints, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    if (cudaEventRecord(s->plan_ev[i], cs) != cudaSuccess) return CODEC_ERR_CUDA;
    const int* D = s->plan_d;
    L.pv = PlanView{Bc, D + s->off_cf, D + s->off_slot,
                    reinterpret_cast<const long long*>(D + s->off_pos0), D + s->off_bidx,
                    skip_h ? D + s->off_skip : nullptr};
    L.tc64 = D + s->off_tc64;
    L.tc128 = D + s->off_tc128;
    L.q16 = D + s->off_q16;
    L.frames = total;
    L.Bc = Bc;
    L.slot_h.assign(slot, slot + Bc);
    L.n_h.resize(Bc);
    for (int b = 0; b < Bc; b++) L.n_h[b] = cf[b + 1] - cf[b];
    return CODEC_OK;
}

// The launch sequence of one decode call, enqueued on cs.  `input` is the
// codes (int32 [B][Q][T_max]) or, for a latent-input codec, the latents
// (float [B][T_max][L]).
void enqueue_decode(codec_state_t* s, Launcher& L, const void* input, int32_t T_max, float* audio,
                    float* pre_tanh, int rows0, cudaStream_t cs)
{
    codec_s* c = s->c;
    const codec_config& g = c->cfg;
    const int S = s->n_slots;
    L.cs = cs;
    const int lt = c->lvl_tf, rt = c->r_tf;
    const Layout L0p{1, s->P[0]};
    const Layout Ltd{rt, 0};                 // the transformer's dense rows
    auto lay = [&](int lvl) { return Layout{c->level_r[lvl], s->P[lvl]}; };
    const int rows_tf = rows0 * rt;

    const double hist_bytes = 8.0 * s->hist_floats_per_slot * (double)L.Bc;
    L.run(CODEC_KERNEL_HISTORY, 0.0, hist_bytes, "history fill",
          [&] { return launch_hist_fill(s->hist_d, (int)s->hist.size(), L.pv, cs); });
    if (g.latent_dim) {
        const int Lc = g.latent_dim;
        L.run(CODEC_KERNEL_GATHER, 2.0 * rows0 * Lc, 4.0 * rows0 * 2.0 * Lc, "latent fill", [&] {
            return launch_latent_fill(static_cast<const float*>(input), Lc, T_max, L.pv, c->lat_mu, c->lat_sigma,
                                      s->e, L0p, rows0, cs);
        });
        L.gemm(c->pre, s->e, L0p, 0, s->h, Ltd, g.d, g.tf_up, nullptr, EPI_STORE, 1.f, 0, "latent front");
    } else {
        L.run(CODEC_KERNEL_GATHER, (double)rows0 * g.Q * g.E, 4.0 * rows0 * ((double)g.Q * (1 + g.E) + g.E),
              "codebook gather", [&] {
                  return launch_rvq_gather(c->cb, g.Q, g.V, g.E, static_cast<const int32_t*>(input), T_max, L.pv,
                                           s->e, L0p, s->err_d, L.max_frames(), cs);
              });
        L.gemm(c->pre, s->e, L0p, 0, s->h, Ltd, g.d, 1, nullptr, EPI_STORE, 1.f, 0, "pre-conv");
    }
    const double norm_flops = 3.0 * rows_tf * g.d, norm_bytes = 8.0 * rows_tf * g.d;
    double attn_flops = 0.0, attn_bytes = 8.0 * rows_tf * g.d;
    for (size_t b = 0; b < L.n_h.size(); b++) {
        const long long p0 = s->frames_h[L.slot_h[b]] * rt;
        const long long nq = (long long)L.n_h[b] * rt;
        for (long long t = 0; t < nq; t++) attn_flops += 4.0 * g.d * (double)std::min<long long>(p0 + t + 1, g.window);
        attn_bytes += 8.0 * g.d * (double)(nq + std::min<long long>(p0, g.window - 1));
    }
    for (int l = 0; l < g.layers; l++) {
        const LayerW& W = c->layers[l];
        // the norms and the attention feed tensor-core GEMMs only: they write the
        // GEMM's operand planes themselves (the prep kernel would split the same
        // values the same way)
        void* pl = s->tc_scratch.a_hi;
        const int pil = W.qkv.tc.passes == 3 ? 1 : 0;
        L.run(CODEC_KERNEL_RMSNORM, norm_flops, norm_bytes, "rmsnorm 1", [&] {
            return launch_rms_norm(s->h, Ltd, W.n1, g.rms_eps, s->u, Ltd, g.d, L.pv, rows_tf, cs,
                                   W.qkv.use_tc ? pl : nullptr, pil);
        });
        L.gemm(W.qkv, s->u, Ltd, lt, s->q, Ltd, g.d, 1, nullptr, EPI_QKV, 1.f, l, "qkv", W.qkv.use_tc);
        const size_t per_layer = (size_t)S * s->R * g.d;
        L.run(CODEC_KERNEL_ATTENTION, attn_flops, attn_bytes, "attention", [&] {
            return launch_swa(s->q, s->o, s->kring + per_layer * l, s->vring + per_layer * l, g.d, g.heads,
                              g.window, s->R, rt, L.pv, L.q16, L.nq16, cs, W.o.use_tc ? pl : nullptr,
                              W.o.tc.passes == 3 ? 1 : 0, g.precision != CODEC_PRECISION_FP32);
        });
        L.gemm(W.o, s->o, Ltd, lt, s->h, Ltd, g.d, 1, s->h, EPI_RESID, 1.f, 0, "out-proj", W.o.use_tc);
        L.run(CODEC_KERNEL_RMSNORM, norm_flops, norm_bytes, "rmsnorm 2", [&] {
            return launch_rms_norm(s->h, Ltd, W.n2, g.rms_eps, s->u, Ltd, g.d, L.pv, rows_tf, cs,
                                   W.w1.use_tc ? pl : nullptr, W.w1.tc.passes == 3 ? 1 : 0);
        });
        // on the tensor cores the GELU moves from the first linear's epilogue to
        // the second's operand prep (the same function of the same value, so the
        // same bits; the prep runs at full occupancy, the epilogue on 8 warps)
        const bool gelu_prep = W.w1.use_tc && W.w2.use_tc;
        L.gemm(W.w1, s->u, Ltd, lt, s->f, Ltd, g.ffn, 1, nullptr, gelu_prep ? EPI_STORE : EPI_GELU, 1.f, 0, "mlp 1",
               W.w1.use_tc);
        L.gemm(W.w2, s->f, Ltd, lt, s->h, Ltd, g.d, 1, s->h, EPI_RESID, 1.f, 0, "mlp 2", false, gelu_prep);
    }
    L.run(CODEC_KERNEL_RMSNORM, norm_flops, norm_bytes, "final rmsnorm",
          [&] { return launch_rms_norm(s->h, Ltd, c->tf_norm, g.rms_eps, s->hf, lay(lt), g.d, L.pv, rows_tf, cs); });
    const float* x = s->hf;
    int xl = lt;
    for (int u = 0; u < g.n_up; u++) {
        L.gemm(c->up[u], x, lay(xl), xl, s->up_out[u], lay(xl + 1), g.up_ch[u], g.up_s, nullptr, EPI_STORE,
               1.f, 0, "latent upsample");
        x = s->up_out[u];
        xl++;
    }
    for (int si = 0; si < g.n_stages; si++) {
        const int lvl = xl + 1;
        const int C = g.ch[si];
        L.gemm(c->st[si], x, lay(xl), xl, s->x0[si], lay(lvl), C, g.strides[si], nullptr, EPI_STORE, 1.f, 0,
               "stage upsample");
        // The resblocks of an MRF are independent until their sum: every conv but
        // the last of resblock j > 0 runs on side stream j - 1 with its own
        // scratch, concurrently with resblock 0 on cs; the last convs then add
        // into y in resblock order on cs, so the sum's order (and its bits) is
        // that of a serial run.
        // (serial while per-launch timing is on: concurrent launches would
        // overlap each other's event intervals)
        const bool fork = g.n_rb > 1 && s->side[0] != nullptr && !s->prof_on;
        if (fork && L.err == cudaSuccess) {
            if (cudaEventRecord(s->fork_ev, cs) != cudaSuccess) L.err = cudaErrorUnknown;
            for (int j = 1; j < g.n_rb && L.err == cudaSuccess; j++)
                if (cudaStreamWaitEvent(s->side[j - 1], s->fork_ev, 0) != cudaSuccess) L.err = cudaErrorUnknown;
        }
        // a small call (first audio) also runs each resblock's last conv on its
        // own stream into its own buffer, and one kernel forms the MRF sum
        // with the same additions in the same order
        const bool split_mrf = fork && L.frames <= codec_state_s::kMrfSmallFrames && s->ymrf[si][1] != nullptr;
        float* last_in[4] = {};
        for (int j = 0; j < g.n_rb; j++) {
            const bool on_side = fork && j > 0;
            L.cs = on_side ? s->side[j - 1] : cs;
            L.scr = on_side ? &s->tc_chain[j - 1] : nullptr;
            const float* rin = s->x0[si];
            for (int ii = 0; ii < g.n_dil - 1; ii++) {
                float* out = s->rbuf[si][j][ii + 1];
                L.gemm(c->rb[c->rb_index(si, j, ii)], rin, lay(lvl), lvl, out, lay(lvl), C, 1, rin, EPI_RESID,
                       1.0f / (float)g.n_rb, 0, "resblock conv");
                rin = out;
            }
            last_in[j] = const_cast<float*>(rin);
            if (split_mrf) {
                float* out = j == 0 ? s->y[si] : s->ymrf[si][j];
                L.gemm(c->rb[c->rb_index(si, j, g.n_dil - 1)], rin, lay(lvl), lvl, out, lay(lvl), C, 1, rin,
                       EPI_RESID, 1.0f / (float)g.n_rb, 0, "resblock conv");
            }
            if (on_side && L.err == cudaSuccess && cudaEventRecord(s->done_ev[j - 1], L.cs) != cudaSuccess)
                L.err = cudaErrorUnknown;
        }
        L.cs = cs;
        L.scr = nullptr;
        if (split_mrf) {
            for (int j = 1; j < g.n_rb; j++)
                if (L.err == cudaSuccess && cudaStreamWaitEvent(cs, s->done_ev[j - 1], 0) != cudaSuccess)
                    L.err = cudaErrorUnknown;
            const double R = (double)L.rows(lvl);
            L.run(CODEC_KERNEL_MRF_SUM, R * C * g.n_rb, 4.0 * R * C * (g.n_rb + 1), "MRF sum", [&] {
                return launch_mrf_sum(s->y[si], s->ymrf[si][1], g.n_rb > 2 ? s->ymrf[si][2] : nullptr, lay(lvl), C,
                                      1.0f / (float)g.n_rb, L.pv, L.rows(lvl), cs);
            });
        }
        for (int j = 0; j < g.n_rb && !split_mrf; j++) {
            if (fork && j > 0 && L.err == cudaSuccess && cudaStreamWaitEvent(cs, s->done_ev[j - 1], 0) != cudaSuccess)
                L.err = cudaErrorUnknown;
            int epi = EPI_RESID;
            if (g.n_rb > 1) epi = j == 0 ? EPI_MRF_FIRST : (j == g.n_rb - 1 ? EPI_MRF_LAST : EPI_MRF_ADD);
            L.gemm(c->rb[c->rb_index(si, j, g.n_dil - 1)], last_in[j], lay(lvl), lvl, s->y[si], lay(lvl), C, 1,
                   last_in[j], epi, 1.0f / (float)g.n_rb, 0, "resblock conv");
        }
        x = s->y[si];
        xl = lvl;
    }
    {
        const int Cl = g.ch[g.n_stages - 1];
        const double R = (double)L.rows(xl);
        L.run(CODEC_KERNEL_FINAL_CONV, 2.0 * R * Cl * g.final_k, 4.0 * R * (Cl + (pre_tanh ? 2 : 1)), "final conv",
              [&] {
                  return launch_final_conv(x, lay(xl), Cl, c->out_w, c->out_b, c->out_alpha, c->out_inv_alpha,
                                           g.final_k, audio, pre_tanh, (long long)T_max * c->spf, c->spf, L.pv,
                                           L.tc128 + (size_t)xl * (S + 1), L.ntiles128[xl], cs);
              });
    }
    L.run(CODEC_KERNEL_HISTORY, 0.0, hist_bytes, "history commit",
          [&] { return launch_hist_commit(s->hist_d, (int)s->hist.size(), L.pv, nullptr, s->frames_d, cs); });
}

codec_status decode_impl(codec_state_t* s, const void* codes, const int32_t* n_frames,
                         const int32_t* ids, int32_t B, int32_t T_max, float* audio, float* pre_tanh,
                         cudaStream_t cs, const int32_t* skip = nullptr)
{
    if (!s || !codes || !n_frames || !audio) return CODEC_ERR_NULL;
    s->last_launches = 0;
    Launcher L;
    int rows0 = 0;
    codec_status pst = plan_call(s, n_frames, ids, B, T_max, cs, L, rows0, skip);
    if (pst != CODEC_OK || rows0 == 0) return pst;

    // Replay a captured graph of this call's launch sequence when one exists
    // for the same shape and buffers: the sequence reads everything that
    // changes between such calls (positions, slots) from the plan uploaded
    // above, so only the shape and the pointers baked into kernel arguments
    // select the graph.
    const bool use_graph = s->graphs_on && !s->prof_on && !debug_sync();
    if (use_graph) {
        std::vector<long long> key;
        key.reserve(L.n_h.size() + 5);
        key.push_back((long long)L.n_h.size());
        key.push_back(T_max);
        key.push_back((long long)(uintptr_t)codes);
        key.push_back((long long)(uintptr_t)audio);
        key.push_back((long long)(uintptr_t)pre_tanh);
        key.push_back(skip ? 1 : 0);
        for (int n : L.n_h) key.push_back(n);
        GraphEntry* ge = nullptr;
        for (GraphEntry& e : s->graphs)
            if (e.key == key) { ge = &e; break; }
        // capture a shape the second time it is seen; one-off shapes run directly
        bool seen = false;
        if (!ge) {
            for (const auto& k : s->seen)
                if (k == key) { seen = true; break; }
            if (!seen) {
                if (s->seen.size() >= 64) s->seen.erase(s->seen.begin());
                s->seen.push_back(key);
            }
        }
        if (!ge && seen) {
            cudaGraph_t graph = nullptr;
            cudaGraphExec_t exec = nullptr;
            bool ok = cudaStreamBeginCapture(s->cap_stream, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
            if (ok) {
                enqueue_decode(s, L, codes, T_max, audio, pre_tanh, rows0, s->cap_stream);
                const cudaError_t ce = cudaStreamEndCapture(s->cap_stream, &graph);
                ok = ce == cudaSuccess && L.err == cudaSuccess && graph != nullptr &&
                     cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
                if (graph) cudaGraphDestroy(graph);
            }
            cudaGetLastError();   // a failed capture leaves nothing behind; run the call directly
            if (ok) {
                if (s->graphs.size() >= codec_state_s::kMaxGraphs) {
                    auto lru = std::min_element(s->graphs.begin(), s->graphs.end(),
                                                [](const GraphEntry& x, const GraphEntry& y) { return x.used < y.used; });
                    cudaGraphExecDestroy(lru->exec);
                    s->graphs.erase(lru);
                }
                s->graphs.push_back(GraphEntry{key, exec, L.launches, 0});
                ge = &s->graphs.back();
            } else {
                if (exec) cudaGraphExecDestroy(exec);
                s->graphs_on = false;   // this driver or configuration cannot capture: stay direct
                Launcher L2 = L;
                L2.launches = 0;
                L2.err = cudaSuccess;
                L = L2;
            }
        }
        if (ge) {
            ge->used = ++s->graph_clock;
            if (cudaGraphLaunch(ge->exec, cs) != cudaSuccess) return CODEC_ERR_CUDA;
            s->last_launches = ge->launches;
            for (size_t b = 0; b < L.slot_h.size(); b++) s->frames_h[L.slot_h[b]] += L.n_h[b];
            return CODEC_OK;
        }
    }
    enqueue_decode(s, L, codes, T_max, audio, pre_tanh, rows0, cs);
    s->last_launches = L.launches;
    if (L.err != cudaSuccess) {
        if (debug_sync()) fprintf(stderr, "codec: %s failed: %s\n", L.where, cudaGetErrorString(L.err));
        return CODEC_ERR_CUDA;
    }
    for (size_t b = 0; b < L.slot_h.size(); b++) s->frames_h[L.slot_h[b]] += L.n_h[b];
    return CODEC_OK;
}

codec_status embed_impl(codec_state_t* s, const int32_t* codes, const int32_t* n_frames, const int32_t* ids,
                        int32_t B, int32_t T_max, float* emb, cudaStream_t cs)
{
    if (!s || !codes || !n_frames || !emb) return CODEC_ERR_NULL;
    if (s->c->cfg.latent_dim) return CODEC_ERR_CONFIG;
    const codec_config& g = s->c->cfg;
    Launcher L;
    int rows0 = 0;
    codec_status pst = plan_call(s, n_frames, ids, B, T_max, cs, L, rows0);
    if (pst != CODEC_OK || rows0 == 0) return pst;
    L.run(CODEC_KERNEL_GATHER, (double)rows0 * g.Q * g.E, 4.0 * rows0 * ((double)g.Q * (1 + g.E) + g.E),
          "codebook gather",
          [&] {
              return launch_rvq_gather(s->c->cb, g.Q, g.V, g.E, codes, T_max, L.pv, emb, Layout{1, 0}, s->err_d,
                                       L.max_frames(), cs);
          });
    s->last_launches = L.launches;
    return L.err == cudaSuccess ? CODEC_OK : CODEC_ERR_CUDA;
}

}  // namespace

extern "C" {

codec_status codec_decode_chunk(codec_state_t* s, const int32_t* codes, const int32_t* n_frames,
                                const int32_t* ids, int32_t B, int32_t T_max, float* audio, void* stream)
{
    if (s && s->c->cfg.latent_dim) return CODEC_ERR_CONFIG;
    return decode_impl(s, codes, n_frames, ids, B, T_max, audio, nullptr, (cudaStream_t)stream);
}

codec_status codec_decode_chunk_ex(codec_state_t* s, const int32_t* codes, const int32_t* n_frames,
                                   const int32_t* ids, int32_t B, int32_t T_max, float* audio,
                                   float* pre_tanh, void* stream)
{
    if (s && s->c->cfg.latent_dim) return CODEC_ERR_CONFIG;
    return decode_impl(s, codes, n_frames, ids, B, T_max, audio, pre_tanh, (cudaStream_t)stream);
}

codec_status codec_decode_latents(codec_state_t* s, const float* latents, const int32_t* n_frames,
                                  const int32_t* ids, int32_t B, int32_t T_max, float* audio, float* pre_tanh,
                                  void* stream)
{
    if (s && !s->c->cfg.latent_dim) return CODEC_ERR_CONFIG;
    return decode_impl(s, latents, n_frames, ids, B, T_max, audio, pre_tanh, (cudaStream_t)stream);
}

codec_status codec_embed_chunk(codec_state_t* s, const int32_t* codes, const int32_t* n_frames,
                               const int32_t* ids, int32_t B, int32_t T_max, float* emb, void* stream)
{
    return embed_impl(s, codes, n_frames, ids, B, T_max, emb, (cudaStream_t)stream);
}

codec_status codec_decode_recompute(codec_state_t* s, const int32_t* codes, const int32_t* n_ctx,
                                    const int32_t* n_new, const int32_t* ids, int32_t B, int32_t T_max,
                                    float* audio, float* pre_tanh, void* stream)
{
    if (!s || !codes || !n_ctx || !n_new || !audio) return CODEC_ERR_NULL;
    const codec_config& g = s->c->cfg;
    if (g.latent_dim) return CODEC_ERR_CONFIG;
    if (B < 1 || T_max < 1) return CODEC_ERR_ARG;
    if (B > s->n_slots) return CODEC_ERR_CAPACITY;
    std::vector<int32_t> n_frames(B), reset_ids;
    long long total = 0;
    for (int b = 0; b < B; b++) {
        if (n_ctx[b] < 0 || n_new[b] < 0 || (long long)n_ctx[b] + n_new[b] > T_max) return CODEC_ERR_ARG;
        if (n_ctx[b] + n_new[b] > g.max_chunk_frames) return CODEC_ERR_CAPACITY;
        // an entry with no new frames is left alone: no reset, no decode
        n_frames[b] = n_new[b] > 0 ? n_ctx[b] + n_new[b] : 0;
        total += n_frames[b];
    }
    if (total > g.max_batch_frames) return CODEC_ERR_CAPACITY;
    // the remaining argument errors (ids) are the decode's own; check them
    // before the reset enqueues anything
    {
        std::vector<char> seen(s->n_slots, 0);
        for (int b = 0; b < B; b++) {
            const int id = ids ? ids[b] : b;
            if (id < 0 || id >= s->n_slots || seen[id]) return CODEC_ERR_ARG;
            seen[id] = 1;
            if (n_frames[b] > 0) reset_ids.push_back(id);
        }
    }
    if (reset_ids.empty()) return CODEC_OK;
    const codec_status rst = codec_state_reset(s, reset_ids.data(), (int32_t)reset_ids.size(), stream);
    if (rst != CODEC_OK) return rst;
    return decode_impl(s, codes, n_frames.data(), ids, B, T_max, audio, pre_tanh, (cudaStream_t)stream, n_ctx);
}

int32_t codec_chunk_frames(const codec_chunk_schedule* sch, int32_t index, int64_t frames_delivered)
{
    if (!sch || index < 0 || frames_delivered < 0 || sch->first < 1 || sch->steady < 1) return 0;
    switch (sch->kind) {
    case CODEC_SCHEDULE_FIXED:
        return index == 0 ? sch->first : sch->steady;
    case CODEC_SCHEDULE_RAMP:
        if (sch->n_ramp < 0 || sch->n_ramp > 8) return 0;
        return index < sch->n_ramp ? std::max(1, sch->ramp[index]) : sch->steady;
    case CODEC_SCHEDULE_ADAPTIVE:
        if (index == 0) return std::min(sch->first, sch->steady);
        return (int32_t)std::min<int64_t>(sch->steady, std::max<int64_t>(1, frames_delivered));
    default:
        return 0;
    }
}

codec_status codec_decode_chunk_host(codec_state_t* s, const int32_t* codes_host, const int32_t* n_frames,
                                     const int32_t* ids, int32_t B, int32_t T_max, float* audio_host,
                                     void* stream)
{
    if (!s || !codes_host || !n_frames || !audio_host) return CODEC_ERR_NULL;
    const codec_config& g = s->c->cfg;
    if (g.latent_dim) return CODEC_ERR_CONFIG;
    if (B < 1 || T_max < 1) return CODEC_ERR_ARG;
    if (B > s->n_slots || T_max > g.max_chunk_frames) return CODEC_ERR_CAPACITY;
    cudaStream_t cs = (cudaStream_t)stream;
    if (cudaMemcpyAsync(s->codes_d, codes_host, sizeof(int32_t) * (size_t)B * g.Q * T_max,
                        cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return CODEC_ERR_CUDA;
    codec_status st = decode_impl(s, s->codes_d, n_frames, ids, B, T_max, s->audio_d, nullptr, cs);
    if (st != CODEC_OK) return st;
    const size_t ld = (size_t)T_max * s->c->spf;
    for (int b = 0; b < B; b++) {
        if (n_frames[b] <= 0) continue;
        if (cudaMemcpyAsync(audio_host + b * ld, s->audio_d + b * ld, sizeof(float) * (size_t)n_frames[b] * s->c->spf,
                            cudaMemcpyDeviceToHost, cs) != cudaSuccess)
            return CODEC_ERR_CUDA;
    }
    if (cudaStreamSynchronize(cs) != cudaSuccess) return CODEC_ERR_CUDA;
    return CODEC_OK;
}

}  // extern "C"
