// The blixt/phonon "Weights" storage format for a decoder weight blob, read
// on the GPU: every tensor of 16,384 values or more is int8 with one f16
// scale per 32 values along the rows of its converted layout; every other
// tensor is f16.  codec_create_q8 uploads such a file, expands it to the fp32
// blob (PyTorch layouts) with one kernel per tensor, and builds the codec
// from that.  int8 x f16 products have at most 18 significant bits, so the
// expanded values are exact in fp32 and the decode sees exactly the
// dequantised weights.
//
// File layout, tensor by tensor in blob order, each part starting on a
// 4-byte boundary (the page's shaders read the file as 32-bit words):
//   quantised tensor: int8 q [R][L], then f16 scale [R][ceil(L / 32)];
//                     value (r, c) = q[r][c] * scale[r][c / 32]
//   other tensor:     f16 values in the blob layout
// Converted rows (R x L): linear / codebook [out][in]; conv [out][tap][in]
// (PyTorch [out][in][tap]); transposed conv [out][phase][tap][in] with kernel
// index = phase + tap * stride (PyTorch [in][out][2 stride]).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "codec.h"

namespace {

constexpr int64_t kQuantMin = 16384;
constexpr int kGroup = 32;

enum Kind { K_VEC = 0, K_2D = 1, K_CONV = 2, K_CONVT = 3 };

struct Tensor {
    int kind;
    int64_t d0, d1, d2;   // PyTorch shape (unused dims 1)
    int64_t size;
};

// The blob's tensors in order, with their kinds and PyTorch shapes.
std::vector<Tensor> blob_tensors(const codec_config* c)
{
    std::vector<Tensor> t;
    auto vec = [&](int64_t n) { t.push_back({K_VEC, n, 1, 1, n}); };
    auto two = [&](int64_t r, int64_t l) { t.push_back({K_2D, r, l, 1, r * l}); };
    auto conv = [&](int64_t co, int64_t ci, int64_t k) { t.push_back({K_CONV, co, ci, k, co * ci * k}); };
    auto convt = [&](int64_t ci, int64_t co, int64_t k) { t.push_back({K_CONVT, ci, co, k, ci * co * k}); };
    if (c->latent_dim) {                     // mu, sigma, projection, depthwise taps [d][1][2 s], bias
        vec(c->latent_dim);
        vec(c->latent_dim);
        two(c->d, c->latent_dim);
        conv(c->d, 1, 2 * c->tf_up);
        vec(c->d);
    } else {
        for (int q = 0; q < c->Q; q++) two(c->V, c->E);
        conv(c->d, c->E, c->pre_k);
        vec(c->d);
    }
    for (int l = 0; l < c->layers; l++) {
        vec(c->d);
        for (int i = 0; i < 4; i++) two(c->d, c->d);
        vec(c->d);
        two(c->ffn, c->d);
        two(c->d, c->ffn);
    }
    vec(c->d);
    int64_t cin = c->d;
    for (int u = 0; u < c->n_up; u++) {
        convt(cin, c->up_ch[u], c->up_k);
        vec(c->up_ch[u]);
        cin = c->up_ch[u];
    }
    for (int s = 0; s < c->n_stages; s++) {
        const int64_t co = c->ch[s];
        vec(cin);
        convt(cin, co, 2 * c->strides[s]);
        vec(co);
        for (int j = 0; j < c->n_rb; j++)
            for (int i = 0; i < c->n_dil; i++) {
                vec(co);
                conv(co, co, c->rb_k[j]);
                vec(co);
            }
        cin = co;
    }
    vec(cin);
    conv(1, cin, c->final_k);
    vec(1);
    return t;
}

// Rows and row length of a quantised tensor's converted layout.
void rows_of(const Tensor& t, int64_t* R, int64_t* L)
{
    switch (t.kind) {
    case K_2D: *R = t.d0; *L = t.d1; break;
    case K_CONV: *R = t.d0; *L = t.d1 * t.d2; break;            // [out][tap][in]
    case K_CONVT: *R = t.d1; *L = t.d0 * t.d2; break;           // [out][phase][tap][in]
    default: *R = 1; *L = t.size; break;
    }
}

int64_t pad4(int64_t n) { return (n + 3) & ~int64_t(3); }

int64_t tensor_bytes(const Tensor& t)
{
    if (t.size < kQuantMin) return pad4(2 * t.size);
    int64_t R, L;
    rows_of(t, &R, &L);
    return pad4(R * L) + pad4(2 * R * ((L + kGroup - 1) / kGroup));
}

__global__ void dequant_kernel(const int8_t* __restrict__ q, const __half* __restrict__ scale, int kind,
                               int64_t d0, int64_t d1, int64_t d2, int64_t R, int64_t L, float* __restrict__ out)
{
    const int64_t G = (L + kGroup - 1) / kGroup;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < R * L; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / L, c = i - r * L;
        const float v = (float)q[i] * __half2float(scale[r * G + c / kGroup]);
        int64_t dst;
        if (kind == K_CONV) {                 // c = tap * in + ci  ->  [out][in][tap]
            const int64_t tap = c / d1, ci = c - tap * d1;
            dst = (r * d1 + ci) * d2 + tap;
        } else if (kind == K_CONVT) {         // c = (p * 2 + j) * in + ci, k = p + j s  ->  [in][out][2 s]
            const int64_t s = d2 / 2;
            const int64_t pj = c / d0, ci = c - pj * d0;
            const int64_t p = pj / 2, j = pj - 2 * p;
            dst = (ci * d1 + r) * d2 + p + j * s;
        } else {
            dst = i;
        }
        out[dst] = v;
    }
}

__global__ void f16_kernel(const __half* __restrict__ h, int64_t n, float* __restrict__ out)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __half2float(h[i]);
}

}  // namespace

extern "C" {

int64_t codec_q8_bytes(const codec_config* cfg)
{
    if (!cfg || codec_weight_floats(cfg) < 0) return -1;
    int64_t n = 0;
    for (const Tensor& t : blob_tensors(cfg)) n += tensor_bytes(t);
    return n;
}

codec_status codec_create_q8(const codec_config* cfg, const void* q8, int64_t n_bytes, codec_t** out)
{
    if (!out) return CODEC_ERR_NULL;
    *out = nullptr;
    if (!cfg || !q8) return CODEC_ERR_NULL;
    const int64_t nf = codec_weight_floats(cfg);
    if (nf < 0) return CODEC_ERR_CONFIG;
    if (n_bytes != codec_q8_bytes(cfg)) return CODEC_ERR_WEIGHTS;
    const std::vector<Tensor> ts = blob_tensors(cfg);
    void* dq = nullptr;
    float* dblob = nullptr;
    if (cudaMalloc(&dq, (size_t)n_bytes) != cudaSuccess) return CODEC_ERR_OOM;
    if (cudaMalloc(&dblob, (size_t)nf * sizeof(float)) != cudaSuccess) {
        cudaFree(dq);
        return CODEC_ERR_OOM;
    }
    codec_status st = CODEC_OK;
    if (cudaMemcpy(dq, q8, (size_t)n_bytes, cudaMemcpyHostToDevice) != cudaSuccess) st = CODEC_ERR_CUDA;
    const unsigned char* base = static_cast<const unsigned char*>(dq);
    int64_t off = 0, foff = 0;
    for (const Tensor& t : ts) {
        if (st != CODEC_OK) break;
        const int blocks = (int)std::min<int64_t>((t.size + 255) / 256, 4096);
        if (t.size < kQuantMin) {
            f16_kernel<<<blocks, 256>>>(reinterpret_cast<const __half*>(base + off), t.size, dblob + foff);
        } else {
            int64_t R, L;
            rows_of(t, &R, &L);
            const __half* sc = reinterpret_cast<const __half*>(base + off + pad4(R * L));
            dequant_kernel<<<blocks, 256>>>(reinterpret_cast<const int8_t*>(base + off), sc, t.kind, t.d0, t.d1,
                                            t.d2, R, L, dblob + foff);
        }
        if (cudaGetLastError() != cudaSuccess) st = CODEC_ERR_CUDA;
        off += tensor_bytes(t);
        foff += t.size;
    }
    std::vector<float> host;
    if (st == CODEC_OK) {
        host.resize((size_t)nf);
        if (cudaMemcpy(host.data(), dblob, (size_t)nf * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
            st = CODEC_ERR_CUDA;
    }
    cudaFree(dq);
    cudaFree(dblob);
    if (st != CODEC_OK) return st;
    return codec_create(cfg, host.data(), nf, out);
}

}  // extern "C"
