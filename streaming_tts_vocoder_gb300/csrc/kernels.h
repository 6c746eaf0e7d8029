// Host-side launchers of the decoder kernels.  Every launcher enqueues on the
// given stream and returns the launch status; none synchronises.
#pragma once

#include "common.cuh"

namespace codec {

// A history tensor: the last H rows of a prefixed buffer carried per slot.
struct HistDesc {
    float* buf;        // packed activation buffer (prefixed layout)
    float* state;      // [slots][H][C]
    int C, H;
    Layout l;
};

// max_frames: the call's longest chunk (frames of its longest batch entry).
cudaError_t launch_rvq_gather(const float* cb, int Q, int V, int E, const int* codes, int T_max,
                              PlanView plan, float* e, Layout el, unsigned* err_words,
                              int max_frames, cudaStream_t s);

// Latent input: e[row] = x * sigma + mu for the call's frames (x [B][T_max][L]);
// rows of e are ldo floats apart (0: L).
cudaError_t launch_latent_fill(const float* x, int L, int T_max, PlanView plan, const float* mu,
                               const float* sigma, float* e, Layout el, int total_rows, cudaStream_t s, int ldo = 0);

cudaError_t launch_gemm_simt(const GemmArgs& a, PlanView plan, int n_row_tiles, cudaStream_t s);

// Rows of x and y run at xl.r rows per frame.  planes (optional): write the
// rows as a tensor-core GEMM's operand planes
// (interleaved hi/lo when planes_il, else the hi plane) instead of y.
cudaError_t launch_rms_norm(const float* x, Layout xl, const float* g, float eps, float* y, Layout yl,
                            int d, PlanView plan, int total_rows, cudaStream_t s, void* planes = nullptr,
                            int planes_il = 1);

// qcum: [B + 1] cumulative blocks of kSwaQueries queries per batch entry.  planes
// (optional): the output as operand planes instead of o, as for RMSNorm.
// Shared memory one attention block needs (the kernel allows up to 227 KB).
size_t swa_smem_bytes(int dh, int window);
// The tensor-core variant for long windows (head width 64, window >= 128);
// launch_swa takes it where eligible.
size_t swa_mma_smem_bytes(int window);
bool swa_mma_eligible(int dh, int window);
cudaError_t configure_swa_mma();
cudaError_t launch_swa_mma(const float* q, float* o, const float* kring, const float* vring, int d, int heads,
                           int window, int ring_R, int pos_r, PlanView plan, const int* qcum, int n_qblocks,
                           cudaStream_t s, void* planes, int planes_il);
constexpr int kSwaWindowMax = 256;
constexpr size_t kSwaSmemMax = 227 * 1024;

// tensor_cores: take the tensor-core variant where it is eligible (the fp32
// precision mode keeps every product on the CUDA cores).
cudaError_t launch_swa(const float* q, float* o, const float* kring, const float* vring, int d,
                       int heads, int window, int ring_R, int pos_r, PlanView plan, const int* qcum, int n_qblocks,
                       cudaStream_t s, void* planes = nullptr, int planes_il = 1, bool tensor_cores = false);

// Shared memory of one final-conv block (the kernel allows up to kFinalSmemMax).
size_t final_conv_smem_bytes(int C, int k);
constexpr size_t kFinalSmemMax = 160 * 1024;

cudaError_t launch_final_conv(const float* x, Layout xl, int C, const float* w, const float* bias,
                              const float* alpha, const float* inv_alpha, int k, float* audio,
                              float* pre_tanh, long long audio_ld, int spf, PlanView plan, const int* tcum,
                              int n_row_tiles, cudaStream_t s);

// y = ((y + y1) + y2) * scale over the chunk rows of a prefixed level (y2 may
// be null), the multi-receptive-field average of separately written resblocks.
cudaError_t launch_mrf_sum(float* y, const float* y1, const float* y2, Layout l, int C, float scale, PlanView plan,
                           long long total_rows, cudaStream_t s);

// Sets the kernels' shared-memory carve-outs; called once per codec.
cudaError_t configure_simt_kernels();

cudaError_t launch_hist_fill(const HistDesc* d, int nd, PlanView plan, cudaStream_t s);
cudaError_t launch_hist_commit(const HistDesc* d, int nd, PlanView plan, const int* n_frames,
                               long long* frames, cudaStream_t s);
cudaError_t launch_state_reset(const HistDesc* d, int nd, const int* slots, int n_slots,
                               long long* frames, unsigned* err_words, cudaStream_t s);

}  // namespace codec
