// Allocation-free form of codec_state_conv1d.
//
// Some callers of a decoder library cannot allocate device memory at the
// point where they need a layer computed: a real-time audio thread, where
// cudaMalloc may block for an unbounded time and synchronise the whole
// device; a host application whose GPU memory belongs to its own pool
// allocator and that forbids allocations behind its back; an embedding that
// is handed only input and output buffers.  codec_conv1d_noalloc serves them:
// it runs the same tensor-core conv as codec_state_conv1d, but every scratch
// array it needs lives in one fixed-size device array defined in this file,
// which the CUDA runtime sets up when it loads the library's module on a
// device and which every GPU that loads the library holds until the process
// exits.
#include <cuda_runtime.h>

#include <mutex>

#include "codec.h"
#include "tc_gemm.h"

namespace {

using namespace codec;

// Capacity: each of the four operand planes (A hi, A lo, B hi, B lo) holds up
// to this many fp16 values, so (H + T) * Cin and Cout * Cin * k are each
// limited to 4,194,304.  Total: 32 MiB plus a few KiB of plan words.
constexpr size_t kPlaneElems = size_t(4) << 20;
constexpr size_t kWordsBytes = (kOpWords * sizeof(int) + 255) / 256 * 256;
constexpr size_t kPlaneBytes = kPlaneElems * 2;
constexpr size_t kFlagOffset = kWordsBytes + 4 * kPlaneBytes;
constexpr size_t kScratchBytes = kFlagOffset + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host-side view per device: the array's device address, fetched once per
// device with that device current (in host code the symbol's name is only a
// host stand-in, not a device address).
struct DeviceScratch {
    unsigned char* base = nullptr;
    int sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceScratch g_dev[kMaxDevices];
std::mutex g_mu;

// The array's device address on the current device (looked up, with the
// GEMM's kernel attributes set, on the first call on that device).
codec_status device_scratch(DeviceScratch* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CODEC_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev[dev].base) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CODEC_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CODEC_ERR_CUDA;
        // the GEMM's shared-memory size and register split, as codec_create sets them
        if (tc_configure() != cudaSuccess) return CODEC_ERR_CUDA;
        g_dev[dev].base = static_cast<unsigned char*>(p);
        g_dev[dev].sms = sms;
    }
    *out = g_dev[dev];
    return CODEC_OK;
}

TcOpScratch op_scratch(const DeviceScratch& ds)
{
    TcOpScratch sc;
    sc.words = reinterpret_cast<int*>(ds.base);
    sc.a_hi = ds.base + kWordsBytes;
    sc.a_lo = ds.base + kWordsBytes + kPlaneBytes;
    sc.b_hi = ds.base + kWordsBytes + 2 * kPlaneBytes;
    sc.b_lo = ds.base + kWordsBytes + 3 * kPlaneBytes;
    sc.a_elems = kPlaneElems;
    sc.b_elems = kPlaneElems;
    sc.err = reinterpret_cast<int*>(ds.base + kFlagOffset);
    return sc;
}

}  // namespace

extern "C" codec_status codec_conv1d_noalloc(const float* x, int32_t T, int32_t Cin, const float* w,
                                             const float* bias, const float* alpha, int32_t Cout, int32_t k,
                                             int32_t dilation, float* y, void* stream)
{
    if (!x || !w || !y) return CODEC_ERR_NULL;
    DeviceScratch ds;
    const codec_status dst = device_scratch(&ds);
    if (dst != CODEC_OK) return dst;
    const TcOpScratch sc = op_scratch(ds);
    // argument errors first, then sizes beyond the array: nothing is enqueued
    switch (check_tc_conv1d(sc, T, Cin, alpha != nullptr, Cout, k, dilation)) {
    case OP_OK: break;
    case OP_BAD_ARG: return CODEC_ERR_ARG;
    default: return CODEC_ERR_CAPACITY;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    // the timeout flag describes this call only
    if (cudaMemsetAsync(sc.err, 0, sizeof(int), cs) != cudaSuccess) return CODEC_ERR_CUDA;
    const int r = run_tc_conv1d(sc, x, T, Cin, w, bias, alpha, Cout, k, dilation, y, ds.sms, cs);
    switch (r) {
    case OP_OK: return CODEC_OK;
    case OP_BAD_ARG: return CODEC_ERR_ARG;
    case OP_TOO_BIG: return CODEC_ERR_CAPACITY;
    default: return CODEC_ERR_CUDA;
    }
}

extern "C" codec_status codec_conv1d_noalloc_status(int32_t* timed_out, void* stream)
{
    if (!timed_out) return CODEC_ERR_NULL;
    *timed_out = 0;
    DeviceScratch ds;
    const codec_status dst = device_scratch(&ds);
    if (dst != CODEC_OK) return dst;
    const TcOpScratch sc = op_scratch(ds);
    int flag = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CODEC_ERR_CUDA;
    if (cudaMemcpy(&flag, sc.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CODEC_ERR_CUDA;
    *timed_out = flag ? 1 : 0;
    return CODEC_OK;
}
